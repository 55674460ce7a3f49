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
inline bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// cuTensorMapEncodeTiled (bf16 elements, or bytes when `bytes`) through
// cudaGetDriverEntryPointByVersion, so the library needs no link-time
// dependency on libcuda.  dims/box have `rank` entries, innermost first;
// strides (bytes) has rank - 1.  Returns 0 on success.
int encode_tiled(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                 const uint32_t* box, CUtensorMapSwizzle swizzle, bool bytes = false);

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel of the stream is finishing, and must call pdl_wait()
// before it touches memory that kernel writes (or that later kernels of the
// previous step may still read).  Returns a cudaError_t.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace host
}  // namespace pkv
