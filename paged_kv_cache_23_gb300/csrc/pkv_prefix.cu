// pkv_prefix.cu -- prefix-cache block lookup on the GPU.
//
// "Inference at Scale: KV Cache, Prefill, and Decode", section 05 (Prefix
// caching): every full block is identified by a hash of itself plus the hash
// of its parent block, i.e. of the whole prefix up to it; a new request looks
// the hashes up and, on a match, bumps the block's ref count and skips that
// part of prefill.  "Chapter 31 Serving Efficiency" 31.3: only a shared
// beginning counts (the first miss ends the match) and the key covers the
// computation version (the salt).
//
// Hash: this library's own 128-bit chained definition (two 64-bit lanes),
// stated in pkv.h: a block's key is a mix of a_j = a_{j-1} X + d_j mod
// 2^61 - 1 (the parent's value times X plus the block's own digest), whose
// affine steps compose associatively, so a CTA computes a sequence's chain as
// a parallel prefix scan rather than block after block.  Table: open addressing in device memory, 32-byte entries
// {key lane 0, key lane 1, block id, ref count}; key (0, 0) = empty,
// (1, 0) = removed; linear probing from lane 0 mod capacity.  Keys are claimed
// with a 128-bit compare-and-swap, so concurrent inserts of one key in a batch
// agree on one entry; a second kernel hands the duplicates that entry's block.
#include "pkv_common.cuh"
#include "pkv_host.h"

namespace pkv {

struct alignas(16) PrefixEntry {
    unsigned long long k0, k1;
    int block, refs;
};
static_assert(sizeof(PrefixEntry) == 32, "32-byte entries");

constexpr int kHashThreads = 256;
constexpr int kHashPer = 4;                             // consecutive blocks per thread
constexpr int kHashChunk = kHashThreads * kHashPer;     // blocks per pass of a CTA
constexpr uint64_t kP61 = (1ull << 61) - 1;
constexpr int kLookupBatch = 4;                         // probes a thread keeps in flight

__device__ __forceinline__ uint64_t hmix(uint64_t x) {
    const uint64_t M = 0xD6E8FEB86659FD93ull;
    x ^= x >> 32;
    x *= M;
    x ^= x >> 29;
    x *= M;
    x ^= x >> 32;
    return x;
}

// (a * b) mod 2^61 - 1 for a, b < 2^61 - 1 (2^61 = 1 mod P).
__device__ __forceinline__ uint64_t mulmod61(uint64_t a, uint64_t b) {
    const uint64_t lo = a * b, hi = __umul64hi(a, b);
    uint64_t r = (lo & kP61) + ((hi << 3) | (lo >> 61));
    r = (r & kP61) + (r >> 61);
    return r >= kP61 ? r - kP61 : r;
}

__device__ __forceinline__ uint64_t addmod61(uint64_t a, uint64_t b) {
    const uint64_t r = a + b;
    return r >= kP61 ? r - kP61 : r;
}

// The chain a_j = a_{j-1} X + d_j is a product of affine maps v -> v A + V;
// composing "first (A1, V1), then (A2, V2)" gives (A1 A2, V1 A2 + V2), an
// associative operation, so the chain is a prefix scan.
struct Aff {
    uint64_t A, V;
};

__device__ __forceinline__ Aff compose(Aff f, Aff g) { return Aff{mulmod61(f.A, g.A), addmod61(mulmod61(f.V, g.A), g.V)}; }

__device__ __forceinline__ Aff shfl_up_aff(Aff x, int o) {
    return Aff{__shfl_up_sync(kFull, x.A, o), __shfl_up_sync(kFull, x.V, o)};
}

__constant__ uint64_t kHashSeed[2] = {0x243F6A8885A308D3ull, 0x13198A2E03707344ull};
__constant__ uint64_t kHashX[2] = {0x0C3A5F1D2B4E6978ull, 0x15D3B7E9A1C4F286ull};

// One CTA per sequence, kHashChunk blocks per pass: every block's digest in
// parallel, each thread composes its 4 blocks' maps, a block-wide exclusive
// scan of the composed maps gives every thread the map of all blocks before
// its own, applied to the chain value carried from the previous pass.
__global__ void __launch_bounds__(kHashThreads) prefix_hash_kernel(uint64_t* __restrict__ hashes,
                                                                   const int32_t* __restrict__ tokens,
                                                                   int max_tokens, const int32_t* __restrict__ lens,
                                                                   int num_seqs, int block_size, int max_blocks,
                                                                   uint64_t salt) {
    __shared__ Aff warp_tot[2][kHashThreads / 32];
    __shared__ uint64_t carry[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_launch();
    for (int b = blockIdx.x; b < num_seqs; b += gridDim.x) {
        int nfull = lens[b] / block_size;
        if (nfull > max_blocks) nfull = max_blocks;
        if (nfull < 0) nfull = 0;
        if (tid < 2) carry[tid] = kHashSeed[tid] % kP61;
        __syncthreads();
        const int32_t* tk = tokens + (long long)b * max_tokens;
        for (int j0 = 0; j0 < nfull; j0 += kHashChunk) {
            const int jt = j0 + kHashPer * tid;  // this thread's first block
            // digests: the 4 blocks x 2 lanes are 8 independent mix chains,
            // interleaved token by token (one load per token feeds both lanes)
            uint64_t d[2][kHashPer];
            {
                uint64_t c[kHashPer][2];
                const int32_t* blk[kHashPer];
#pragma unroll
                for (int u = 0; u < kHashPer; ++u) {
                    c[u][0] = kHashSeed[0] ^ salt;
                    c[u][1] = kHashSeed[1] ^ salt;
                    blk[u] = tk + (long long)min(jt + u, nfull - 1) * block_size;  // in range; unused past nfull
                }
                for (int i = 0; i < block_size; ++i) {
                    uint32_t t[kHashPer];
#pragma unroll
                    for (int u = 0; u < kHashPer; ++u) t[u] = (uint32_t)__ldg(blk[u] + i);
#pragma unroll
                    for (int u = 0; u < kHashPer; ++u) {
                        const uint64_t add = (uint64_t)t[u] + ((uint64_t)i << 32);
                        c[u][0] = hmix(c[u][0] + add);
                        c[u][1] = hmix(c[u][1] + add);
                    }
                }
#pragma unroll
                for (int u = 0; u < kHashPer; ++u)
#pragma unroll
                    for (int L = 0; L < 2; ++L) d[L][u] = hmix(c[u][L] + 0x9E3779B97F4A7C15ull) % kP61;
            }
            Aff mine[2];
#pragma unroll
            for (int L = 0; L < 2; ++L) {
                mine[L] = Aff{1, 0};
#pragma unroll
                for (int u = 0; u < kHashPer; ++u)
                    if (jt + u < nfull) mine[L] = compose(mine[L], Aff{kHashX[L], d[L][u]});
            }
            // exclusive scan of the threads' maps, in thread order
            Aff pre[2];
#pragma unroll
            for (int L = 0; L < 2; ++L) {
                Aff x = mine[L];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const Aff y = shfl_up_aff(x, o);
                    if (lane >= o) x = compose(y, x);
                }
                if (lane == 31) warp_tot[L][warp] = x;
                const Aff up = shfl_up_aff(x, 1);
                pre[L] = lane ? up : Aff{1, 0};
            }
            __syncthreads();
#pragma unroll
            for (int L = 0; L < 2; ++L) {
                Aff w = Aff{1, 0};
                for (int k = 0; k < warp; ++k) w = compose(w, warp_tot[L][k]);
                pre[L] = compose(w, pre[L]);
            }
            // chain values of this thread's blocks
            uint64_t a[2] = {carry[0], carry[1]};
            __syncthreads();  // every thread has read the carry
#pragma unroll
            for (int L = 0; L < 2; ++L) a[L] = addmod61(mulmod61(a[L], pre[L].A), pre[L].V);
#pragma unroll
            for (int u = 0; u < kHashPer; ++u) {
                const int j = jt + u;
                if (j >= nfull) break;
                uint64_t key[2];
#pragma unroll
                for (int L = 0; L < 2; ++L) {
                    a[L] = addmod61(mulmod61(a[L], kHashX[L]), d[L][u]);
                    key[L] = hmix(a[L]);
                }
                if (key[1] == 0 && key[0] < 2) key[1] = 1;
                uint64_t* out = hashes + ((long long)b * max_blocks + j) * 2;
                out[0] = key[0];
                out[1] = key[1];
                if (j == min(nfull, j0 + kHashChunk) - 1) {
                    carry[0] = a[0];
                    carry[1] = a[1];
                }
            }
            __syncthreads();  // the next pass reads the new carry
        }
        __syncthreads();
    }
}

// Probe for `key`; returns the slot index or -1 (an empty slot or a whole lap).
__device__ __forceinline__ long long probe(const PrefixEntry* __restrict__ table, long long mask, uint64_t k0,
                                           uint64_t k1) {
    long long i = (long long)(k0 & (uint64_t)mask);
    for (long long step = 0; step <= mask; ++step) {
        const ulonglong2 key = *reinterpret_cast<const ulonglong2*>(&table[i]);
        if (key.x == k0 && key.y == k1) return i;
        if (key.x == 0 && key.y == 0) return -1;
        i = (i + 1) & mask;
    }
    return -1;
}

// One CTA per sequence: every full block probed in parallel; the first miss
// ends the match; hits before it take a reference and fill the block table.
__global__ void __launch_bounds__(kHashThreads) prefix_lookup_kernel(PrefixEntry* __restrict__ table, long long mask,
                                                                     const uint64_t* __restrict__ hashes,
                                                                     const int32_t* __restrict__ lens, int num_seqs,
                                                                     int block_size, int max_blocks,
                                                                     int32_t* __restrict__ block_tables,
                                                                     int32_t* __restrict__ cached) {
    __shared__ int first_miss;
    pdl_wait();
    pdl_launch();
    for (int b = blockIdx.x; b < num_seqs; b += gridDim.x) {
        int nfull = lens[b] / block_size;
        if (nfull > max_blocks) nfull = max_blocks;
        if (nfull < 0) nfull = 0;
        if (threadIdx.x == 0) first_miss = nfull;
        __syncthreads();
        // kLookupBatch blocks per thread at a time: their keys and home slots
        // are loaded together, so most probes cost one round trip
        for (int j0 = 0; j0 < nfull; j0 += kHashThreads * kLookupBatch) {
            ulonglong2 key[kLookupBatch], home[kLookupBatch];
#pragma unroll
            for (int u = 0; u < kLookupBatch; ++u) {
                const int j = j0 + u * kHashThreads + threadIdx.x;
                key[u] = j < nfull ? *reinterpret_cast<const ulonglong2*>(hashes + ((long long)b * max_blocks + j) * 2)
                                   : make_ulonglong2(0, 0);
            }
#pragma unroll
            for (int u = 0; u < kLookupBatch; ++u)
                home[u] = *reinterpret_cast<const ulonglong2*>(&table[key[u].x & (uint64_t)mask]);
#pragma unroll
            for (int u = 0; u < kLookupBatch; ++u) {
                const int j = j0 + u * kHashThreads + threadIdx.x;
                if (j >= nfull) continue;
                const bool hit = (home[u].x == key[u].x && home[u].y == key[u].y) ||
                                 (!(home[u].x == 0 && home[u].y == 0) && probe(table, mask, key[u].x, key[u].y) >= 0);
                if (!hit) atomicMin(&first_miss, j);
            }
        }
        __syncthreads();
        const int n = first_miss;
        for (int j = threadIdx.x; j < n; j += kHashThreads) {
            const uint64_t* k = hashes + ((long long)b * max_blocks + j) * 2;
            const long long s = probe(table, mask, k[0], k[1]);  // found in the first pass
            atomicAdd(&table[s].refs, 1);
            block_tables[(long long)b * max_blocks + j] = table[s].block;
        }
        if (threadIdx.x == 0) cached[b] = n;
        __syncthreads();
    }
}

__device__ __forceinline__ void cas128(void* addr, uint64_t c0, uint64_t c1, uint64_t v0, uint64_t v1, uint64_t& o0,
                                       uint64_t& o1) {
    asm volatile(
        "{\n\t.reg .b128 cmp, val, old;\n\t"
        "mov.b128 cmp, {%2, %3};\n\t"
        "mov.b128 val, {%4, %5};\n\t"
        "atom.global.cas.b128 old, [%6], cmp, val;\n\t"
        "mov.b128 {%0, %1}, old;\n\t}"
        : "=l"(o0), "=l"(o1)
        : "l"(c0), "l"(c1), "l"(v0), "l"(v1), "l"(addr)
        : "memory");
}

// Insert, phase 1: thread per (sequence, block).  An empty slot is claimed with
// a 128-bit CAS (the claimer stores its block id); finding the key already
// there makes the block a duplicate, recorded as -(slot + 3) for phase 2.
// Both take a reference.  resolved = the block now registered for the key.
__global__ void prefix_insert_kernel(PrefixEntry* __restrict__ table, long long mask,
                                     const uint64_t* __restrict__ hashes, const int32_t* __restrict__ block_tables,
                                     const int32_t* __restrict__ first, const int32_t* __restrict__ count,
                                     int num_seqs, int max_blocks, int32_t* __restrict__ resolved, int32_t* status) {
    pdl_wait();
    pdl_launch();
    const long long total = (long long)num_seqs * max_blocks;
    int bits = 0;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int b = (int)(e / max_blocks), j = (int)(e - (long long)b * max_blocks);
        const int f = first[b], c = count[b];
        if (j < f || j >= f + c) continue;
        const uint64_t k0 = hashes[e * 2], k1 = hashes[e * 2 + 1];
        const int blk = block_tables[e];
        long long i = (long long)(k0 & (uint64_t)mask);
        int out = -1;
        for (long long step = 0; step <= mask; ++step) {
            uint64_t o0, o1;
            cas128(&table[i], 0, 0, k0, k1, o0, o1);
            if (o0 == 0 && o1 == 0) {
                table[i].block = blk;
                atomicAdd(&table[i].refs, 1);
                out = blk;
                break;
            }
            if (o0 == k0 && o1 == k1) {
                atomicAdd(&table[i].refs, 1);
                out = (int)(-(i + 3));
                break;
            }
            i = (i + 1) & mask;
        }
        if (out == -1) bits |= PKV_STATUS_TABLE_FULL;
        resolved[e] = out;
    }
    if (bits) report(status, bits);
}

// Insert, phase 2: duplicates read the block their key's entry holds.
__global__ void prefix_resolve_kernel(const PrefixEntry* __restrict__ table, int num_entries,
                                      int32_t* __restrict__ resolved) {
    pdl_wait();
    pdl_launch();
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < num_entries;
         e += (long long)gridDim.x * blockDim.x) {
        const int r = resolved[e];
        if (r <= -3) resolved[e] = table[-(long long)r - 3].block;
    }
}

// Release: thread per (sequence, block j < count[b]) drops one reference.
__global__ void prefix_release_kernel(PrefixEntry* __restrict__ table, long long mask,
                                      const uint64_t* __restrict__ hashes, const int32_t* __restrict__ count,
                                      int num_seqs, int max_blocks, int32_t* status) {
    pdl_wait();
    pdl_launch();
    const long long total = (long long)num_seqs * max_blocks;
    int bits = 0;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int b = (int)(e / max_blocks), j = (int)(e - (long long)b * max_blocks);
        if (j >= count[b]) continue;
        const long long s = probe(table, mask, hashes[e * 2], hashes[e * 2 + 1]);
        if (s < 0) {
            bits |= PKV_STATUS_NOT_FOUND;
            continue;
        }
        atomicSub(&table[s].refs, 1);
    }
    if (bits) report(status, bits);
}

}  // namespace pkv

using namespace pkv;

namespace {
bool pow2(long long x) { return x > 0 && (x & (x - 1)) == 0; }
int grid_for(long long work, int threads) {
    long long g = (work + threads - 1) / threads;
    const long long cap = (long long)host::sm_count() * 8;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}
}  // namespace

extern "C" size_t pkv_prefix_table_bytes(int capacity) {
    return capacity > 0 ? (size_t)capacity * sizeof(PrefixEntry) : 0;
}

extern "C" int pkv_prefix_table_init(void* table, int capacity, void* stream) {
    if (!pow2(capacity)) return PKV_ERR_SIZE;
    if (!table) return PKV_ERR_NULL;
    if (!host::aligned16(table)) return PKV_ERR_ALIGN;
    const int rc = host::check_device();
    if (rc) return rc;
    return cudaMemsetAsync(table, 0, (size_t)capacity * sizeof(PrefixEntry), (cudaStream_t)stream) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

extern "C" int pkv_prefix_hash(uint64_t* hashes, const int32_t* tokens, int max_tokens, const int32_t* lens,
                               int num_seqs, int block_size, int max_blocks, uint64_t salt, void* stream) {
    if (num_seqs < 0 || max_tokens < 0 || block_size < 1 || max_blocks < 0) return PKV_ERR_SIZE;
    if ((long long)max_blocks * block_size > max_tokens) return PKV_ERR_SIZE;
    if (num_seqs == 0 || max_blocks == 0) return PKV_OK;
    if (!hashes || !tokens || !lens) return PKV_ERR_NULL;
    const int rc = host::check_device();
    if (rc) return rc;
    const int grid = num_seqs < host::sm_count() * 8 ? num_seqs : host::sm_count() * 8;
    return host::launch_pdl(prefix_hash_kernel, dim3(grid), dim3(kHashThreads), 0, (cudaStream_t)stream, hashes,
                            tokens, max_tokens, lens, num_seqs, block_size, max_blocks, salt) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

extern "C" int pkv_prefix_lookup(void* table, int capacity, const uint64_t* hashes, const int32_t* lens,
                                 int num_seqs, int block_size, int max_blocks, int32_t* block_tables,
                                 int32_t* cached_blocks, void* stream) {
    if (!pow2(capacity) || num_seqs < 0 || block_size < 1 || max_blocks < 0) return PKV_ERR_SIZE;
    if (num_seqs == 0) return PKV_OK;
    if (!table || !hashes || !lens || !block_tables || !cached_blocks) return PKV_ERR_NULL;
    const int rc = host::check_device();
    if (rc) return rc;
    const int grid = num_seqs < host::sm_count() * 8 ? num_seqs : host::sm_count() * 8;
    return host::launch_pdl(prefix_lookup_kernel, dim3(grid), dim3(kHashThreads), 0, (cudaStream_t)stream,
                            static_cast<PrefixEntry*>(table), (long long)capacity - 1, hashes, lens, num_seqs,
                            block_size, max_blocks, block_tables, cached_blocks) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

extern "C" int pkv_prefix_insert(void* table, int capacity, const uint64_t* hashes, const int32_t* block_tables,
                                 const int32_t* first, const int32_t* count, int num_seqs, int max_blocks,
                                 int32_t* resolved, int32_t* status, void* stream) {
    if (!pow2(capacity) || num_seqs < 0 || max_blocks < 0) return PKV_ERR_SIZE;
    const long long total = (long long)num_seqs * max_blocks;
    if (total == 0) return PKV_OK;
    if (total > 0x7fffffffLL) return PKV_ERR_SIZE;
    if (!table || !hashes || !block_tables || !first || !count || !resolved) return PKV_ERR_NULL;
    if (!host::aligned16(table)) return PKV_ERR_ALIGN;
    const int rc = host::check_device();
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    const int grid = grid_for(total, 256);
    if (host::launch_pdl(prefix_insert_kernel, dim3(grid), dim3(256), 0, st, static_cast<PrefixEntry*>(table),
                         (long long)capacity - 1, hashes, block_tables, first, count, num_seqs, max_blocks, resolved,
                         status) != cudaSuccess)
        return PKV_ERR_CUDA;
    return host::launch_pdl(prefix_resolve_kernel, dim3(grid), dim3(256), 0, st,
                            static_cast<const PrefixEntry*>(table), (int)total, resolved) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

extern "C" int pkv_prefix_release(void* table, int capacity, const uint64_t* hashes, const int32_t* count,
                                  int num_seqs, int max_blocks, int32_t* status, void* stream) {
    if (!pow2(capacity) || num_seqs < 0 || max_blocks < 0) return PKV_ERR_SIZE;
    const long long total = (long long)num_seqs * max_blocks;
    if (total == 0) return PKV_OK;
    if (!table || !hashes || !count) return PKV_ERR_NULL;
    const int rc = host::check_device();
    if (rc) return rc;
    return host::launch_pdl(prefix_release_kernel, dim3(grid_for(total, 256)), dim3(256), 0, (cudaStream_t)stream,
                            static_cast<PrefixEntry*>(table), (long long)capacity - 1, hashes, count, num_seqs,
                            max_blocks, status) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}
