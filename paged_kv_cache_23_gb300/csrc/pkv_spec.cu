// pkv_spec.cu -- greedy speculative acceptance.
//
// "Spending the Idle" 12.4 and "Inference at Scale: KV Cache, Prefill, and
// Decode" section 08: under greedy decoding a drafted token is accepted when it
// equals the target's argmax at that position; acceptance stops at the first
// mismatch and the round always emits one target token (the correction, or
// the bonus token after k accepted drafts).
//
// The row argmax over a 128K vocabulary is an HBM scan.  Each row is split
// across a thread-block cluster of 8 CTAs; partial (value, index) winners are
// combined through distributed shared memory in the cluster's rank-0 CTA.  A
// second tiny kernel turns the k+1 argmaxes of a sequence into the accepted
// length and the next token.
#include <cooperative_groups.h>

#include "pkv_common.cuh"
#include "pkv_host.h"

namespace cg = cooperative_groups;

namespace pkv {

constexpr int kArgmaxCluster = 8;
constexpr int kArgmaxThreads = 256;
constexpr int kNoIndex = 0x7fffffff;

// Total order of the argmax: NaN above every number, then larger value, then
// smaller index (so the first occurrence of the maximum wins).
__device__ __forceinline__ bool beats(float a, int ia, float b, int ib) {
    const bool an = a != a, bn = b != b;
    if (an != bn) return an;
    if (!an && a != b) return a > b;
    return ia < ib;
}

__device__ __forceinline__ void take(float& bv, int& bi, float v, int i) {
    if (beats(v, i, bv, bi)) {
        bv = v;
        bi = i;
    }
}

__global__ void __cluster_dims__(kArgmaxCluster, 1, 1) __launch_bounds__(kArgmaxThreads)
    row_argmax_kernel(const float* __restrict__ logits, long long vocab, int rows, int vec4,
                      int32_t* __restrict__ argmax_out) {
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    __shared__ float wv[kArgmaxThreads / 32];
    __shared__ int wi[kArgmaxThreads / 32];
    __shared__ float cv[kArgmaxCluster];
    __shared__ int ci[kArgmaxCluster];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    long long per = (vocab + kArgmaxCluster - 1) / kArgmaxCluster;
    per = (per + 3) & ~3LL;
    const long long lo = rank * per;
    const long long hi = lo + per < vocab ? lo + per : vocab;
    for (int row = blockIdx.y; row < rows; row += gridDim.y) {
        const float* x = logits + (long long)row * vocab;
        float bv = -INFINITY;
        int bi = kNoIndex;
        if (vec4) {
            // lo and vocab are multiples of 4 and the row start is 16-byte aligned
            const float4* x4 = reinterpret_cast<const float4*>(x + lo);
            const long long n4 = hi > lo ? (hi - lo) >> 2 : 0;
            long long j = tid;
            for (; j + 3 * kArgmaxThreads < n4; j += 4 * kArgmaxThreads) {
                float4 v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) v[u] = __ldg(x4 + j + u * kArgmaxThreads);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int base = (int)(lo + 4 * (j + u * kArgmaxThreads));
                    take(bv, bi, v[u].x, base);
                    take(bv, bi, v[u].y, base + 1);
                    take(bv, bi, v[u].z, base + 2);
                    take(bv, bi, v[u].w, base + 3);
                }
            }
            for (; j < n4; j += kArgmaxThreads) {
                const float4 v = __ldg(x4 + j);
                const int base = (int)(lo + 4 * j);
                take(bv, bi, v.x, base);
                take(bv, bi, v.y, base + 1);
                take(bv, bi, v.z, base + 2);
                take(bv, bi, v.w, base + 3);
            }
        } else {
            for (long long j = lo + tid; j < hi; j += kArgmaxThreads) take(bv, bi, __ldg(x + j), (int)j);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(kFull, bv, o);
            const int oi = __shfl_xor_sync(kFull, bi, o);
            take(bv, bi, ov, oi);
        }
        if (lane == 0) {
            wv[warp] = bv;
            wi[warp] = bi;
        }
        __syncthreads();
        if (tid == 0) {
            for (int w = 1; w < kArgmaxThreads / 32; ++w) take(bv, bi, wv[w], wi[w]);
            float* rv = cluster.map_shared_rank(cv, 0);
            int* ri = cluster.map_shared_rank(ci, 0);
            rv[rank] = bv;
            ri[rank] = bi;
        }
        cluster.sync();
        if (rank == 0 && tid == 0) {
            float v = cv[0];
            int i = ci[0];
            for (int r = 1; r < kArgmaxCluster; ++r) take(v, i, cv[r], ci[r]);
            argmax_out[row] = i;
        }
        cluster.sync();  // cv/ci and wv/wi are reused by the next row
    }
}

__global__ void accept_kernel(const int32_t* __restrict__ argmax, const int32_t* __restrict__ draft, int num_seqs,
                              int k, int32_t* __restrict__ accepted, int32_t* __restrict__ next_token) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= num_seqs) return;
    const int32_t* am = argmax + (long long)b * (k + 1);
    const int32_t* dr = draft + (long long)b * k;
    int a = 0;
    while (a < k && dr[a] == am[a]) ++a;
    accepted[b] = a;
    next_token[b] = am[a];
}

}  // namespace pkv

using namespace pkv;

extern "C" int pkv_spec_accept_greedy(const float* logits, const int32_t* draft, int num_seqs, int k, int vocab,
                                      int32_t* argmax_out, int32_t* accepted, int32_t* next_token, void* stream) {
    if (num_seqs < 0 || k < 1 || k > 64 || vocab < 1) return PKV_ERR_SIZE;
    if (num_seqs == 0) return PKV_OK;
    if (!logits || !draft || !argmax_out || !accepted || !next_token) return PKV_ERR_NULL;
    const int rc = host::check_device();
    if (rc) return rc;
    const long long rows = (long long)num_seqs * (k + 1);
    if (rows > 0x7fffffffLL) return PKV_ERR_SIZE;
    const int vec4 = (vocab % 4 == 0) && host::aligned16(logits);
    dim3 grid(kArgmaxCluster, (unsigned)(rows < 65535 ? rows : 65535));
    row_argmax_kernel<<<grid, kArgmaxThreads, 0, (cudaStream_t)stream>>>(logits, vocab, (int)rows, vec4, argmax_out);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    accept_kernel<<<(num_seqs + 127) / 128, 128, 0, (cudaStream_t)stream>>>(argmax_out, draft, num_seqs, k, accepted,
                                                                           next_token);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
