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

// cuTensorMapEncodeTiled (bf16 elements) through
// cudaGetDriverEntryPointByVersion, so the library needs no link-time
// dependency on libcuda.  dims/box have `rank` entries, innermost first;
// strides (bytes) has rank - 1.  Returns 0 on success.
int encode_tiled(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                 const uint32_t* box, CUtensorMapSwizzle swizzle);

}  // namespace host
}  // namespace pkv
