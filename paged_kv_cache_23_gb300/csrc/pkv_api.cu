// pkv_api.cu -- version, error strings and host helpers of libpkv.
#include <cudaTypedefs.h>

#include <mutex>

#include "pkv.h"
#include "pkv_common.cuh"
#include "pkv_host.h"

namespace pkv {
namespace host {

namespace {
constexpr int kMaxDevices = 64;
int g_sm[kMaxDevices];
int g_ok[kMaxDevices];  // 0 unknown, 1 sm_103, 2 other
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

void probe(int dev) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    g_sm[dev] = sms > 0 ? sms : 1;
    g_ok[dev] = (major == 10 && minor == 3) ? 1 : 2;
}
}  // namespace

int check_device() {
    const int dev = current_device();
    if (dev < 0) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_ok[dev] == 0) probe(dev);
    return g_ok[dev] == 1 ? PKV_OK : PKV_ERR_DEVICE;
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_ok[dev] == 0) probe(dev);
    return g_sm[dev];
}

int encode_tiled(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                 const uint32_t* box, CUtensorMapSwizzle swizzle, bool bytes) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_encode == nullptr) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return -1;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    if (rank < 1 || rank > 5) return -1;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) gs[i] = strides[i];
    }
    const CUresult r = g_encode(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                (cuuint32_t)rank, const_cast<void*>(base), gd,
                                gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : -1;
}

}  // namespace host
}  // namespace pkv

extern "C" int pkv_version(void) { return 100; }

extern "C" const char* pkv_error_string(int rc) {
    switch (rc) {
        case PKV_OK: return "ok";
        case PKV_ERR_NULL: return "a required pointer is NULL";
        case PKV_ERR_SIZE: return "a size or count argument is out of range";
        case PKV_ERR_UNSUPPORTED: return "head_dim, block_size or head grouping not supported";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_ALIGN: return "a pointer is not 16-byte aligned";
        case PKV_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
        case PKV_ERR_DEVICE: return "the current device is not an sm_103 (GB300) GPU";
        case PKV_ERR_SCRATCH_LIMIT: return "needs more scratch than the no-alloc entry point's fixed buffer";
        default: return "unknown error code";
    }
}

extern "C" const char* pkv_status_string(int bit) {
    switch (bit) {
        case PKV_STATUS_BAD_BLOCK: return "block id outside the pool";
        case PKV_STATUS_BAD_SEQLEN: return "seq_len out of range";
        case PKV_STATUS_BAD_QLEN: return "q_len or append_len out of range";
        case PKV_STATUS_BAD_SLOT: return "slot outside the pool";
        case PKV_STATUS_TIMEOUT: return "a bounded device wait ran out";
        case PKV_STATUS_BAD_PAIR: return "copy pair outside the pool";
        case PKV_STATUS_BAD_TOKEN: return "draft token outside the vocabulary";
        case PKV_STATUS_BAD_DIST: return "sampling distribution without positive weight";
        case PKV_STATUS_TABLE_FULL: return "prefix-cache table full";
        case PKV_STATUS_NOT_FOUND: return "prefix-cache key not found";
        case PKV_STATUS_BAD_PLAN: return "no attention plan for this shape in the workspace";
        default: return "unknown status bit";
    }
}

// ---------------------------------------------------------------------------
// Self-test of the bounded device wait: one warp waits, with mbar_wait (the
// wait every attention kernel uses), on an mbarrier phase that nothing
// completes.  The wait must give up after limit_ns of %globaltimer, report
// PKV_STATUS_TIMEOUT and let the kernel return, leaving the context usable.
// ---------------------------------------------------------------------------
namespace pkv {
namespace {
__global__ void wait_selftest_kernel(unsigned long long limit_ns, int32_t* status) {
    __shared__ uint64_t bar;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival completes phase 0; none ever comes
        abort = 0;
        fence_mbar_init();
    }
    __syncwarp();
    bool ok = true;
    if (threadIdx.x == 0) ok = mbar_wait(&bar, 0, &abort, limit_ns);
    if (threadIdx.x == 0 && !ok) report(status, PKV_STATUS_TIMEOUT);
}
}  // namespace
}  // namespace pkv

extern "C" int pkv_wait_selftest(long long limit_ns, int32_t* status, void* stream) {
    if (limit_ns < 1 || limit_ns > 10000000000LL) return PKV_ERR_SIZE;
    if (!status) return PKV_ERR_NULL;
    const int rc = pkv::host::check_device();
    if (rc) return rc;
    pkv::wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((unsigned long long)limit_ns, status);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
