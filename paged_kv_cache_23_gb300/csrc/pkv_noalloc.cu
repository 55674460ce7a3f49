// pkv_noalloc.cu -- paged attention for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc or any allocator on the path: code that
// runs inside another runtime's memory pool or allocator hook (where a nested
// allocation would re-enter it or break its accounting), real-time serving
// loops that must not block on the driver's allocator, and plugins that are
// handed only their input and output buffers.  For them this file keeps the
// attention scratch in one fixed device array that is part of the library
// image, so a call needs nothing but its inputs and outputs.
//
// The array (kScratchBytes, 32 MiB) exists on every GPU that loads this code
// and stays there until the process exits.  Its device address is looked up
// once per device and CUDA context, by the first call made with that device
// current; make that first call before any stream capture starts.  The cached
// address is keyed on the context's unique id as well as the device ordinal,
// so after a cudaDeviceReset (or any other teardown and re-creation of the
// primary context) the next call looks the address up again instead of
// passing a stale pointer to the kernels -- and that call is then a first
// call again (before any stream capture).  All calls share the array, and
// it keeps whatever the last call left in it: the planning kernel re-initialises
// everything it needs (item queue, per-row partition counts) on every call, but two calls
// that overlap on the GPU (different streams, or different host threads on the
// same device without ordering) race on it and give wrong results.
#include <cudaTypedefs.h>

#include <mutex>

#include "pkv.h"

namespace pkv {
namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
void* g_addr[kMaxDev] = {nullptr};
unsigned long long g_ctx_id[kMaxDev] = {0};  // the context each cached address belongs to
std::mutex g_mu;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;

// Unique id of the calling thread's current CUDA context, or 0 when there is
// none (or it has been destroyed).  Context ids are never reused, unlike
// context handles.  The driver entry points are looked up through the runtime,
// so the library needs no link to libcuda.
unsigned long long current_context_id() {
    if (g_ctx_current == nullptr || g_ctx_get_id == nullptr) {
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault, &q1) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || f1 == nullptr ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
            q2 != cudaDriverEntryPointSuccess || f2 == nullptr)
            return 0;
        g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f1);
        g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f2);
    }
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (g_ctx_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
    return g_ctx_get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of g_scratch on the current device (nullptr on failure).
// Set-up, once per device and context: with the device current,
// cudaGetSymbolAddress (which also makes the runtime create the device's
// primary context if there is none yet) gives the array's device address;
// later calls reuse it while the same context is current, and look it up again
// after the context was destroyed and re-created (cudaDeviceReset).
void* scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    const unsigned long long id = current_context_id();
    if (g_addr[dev] == nullptr || id == 0 || g_ctx_id[dev] != id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) return nullptr;
        const unsigned long long id2 = current_context_id();
        if (id2 == 0) return nullptr;
        g_addr[dev] = p;
        g_ctx_id[dev] = id2;
    }
    return g_addr[dev];
}

}  // namespace
}  // namespace pkv

extern "C" size_t pkv_noalloc_scratch_bytes(void) { return pkv::kScratchBytes; }

extern "C" int pkv_paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                                  const int32_t* block_tables, int max_blocks,
                                                  const int32_t* seq_lens, const int32_t* q_lens, int num_seqs,
                                                  int total_q, int max_q_len, int max_seq_len, int num_q_heads,
                                                  int num_kv_heads,
                                                  int head_dim, int block_size, int num_blocks, float scale,
                                                  int partition_tokens, int flags, int32_t* status, void* stream) {
    const size_t need = pkv_attention_workspace_bytes(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim,
                                                      max_seq_len, partition_tokens);
    if (need == 0) return PKV_ERR_SIZE;
    if (need > pkv::kScratchBytes) return PKV_ERR_SCRATCH_LIMIT;
    void* ws = pkv::scratch_address();
    if (ws == nullptr) return PKV_ERR_CUDA;
    return pkv_paged_attention_decode(out, q, k_cache, v_cache, block_tables, max_blocks, seq_lens, q_lens, num_seqs,
                                      total_q, max_q_len, max_seq_len, num_q_heads, num_kv_heads, head_dim, block_size,
                                      num_blocks, scale, partition_tokens, flags, ws, pkv::kScratchBytes, status,
                                      stream);
}
