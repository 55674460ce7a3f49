// pkv_host.h -- host-side helpers of libpkv (device checks, SM count,
// tensor-map encoding through the driver entry point).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {
namespace host {

// PKV_OK if the current device is an sm_103 GPU, else a PKV_ERR_* code.
int check_device();

// Number of SMs of the current device (cached per device).
int sm_count();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled through cudaGetDriverEntryPointByVersion, so the
// library needs no link-time dependency on libcuda.  Returns 0 on success.
int encode_tiled_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                    uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

}  // namespace host
}  // namespace pkv
