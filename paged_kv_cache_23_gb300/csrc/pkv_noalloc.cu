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
// once per device, by the first call made with that device current; make that
// first call before any stream capture starts.  All calls share the array, and
// it keeps whatever the last call left in it: the planning kernel re-initialises
// everything it needs (item queue, per-row partition counts) on every call, but two calls
// that overlap on the GPU (different streams, or different host threads on the
// same device without ordering) race on it and give wrong results.
#include <mutex>

#include "pkv.h"

namespace pkv {
namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
void* g_addr[kMaxDev] = {nullptr};
std::mutex g_mu;

// Device address of g_scratch on the current device (nullptr on failure).
void* scratch_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) return nullptr;
        g_addr[dev] = p;
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
