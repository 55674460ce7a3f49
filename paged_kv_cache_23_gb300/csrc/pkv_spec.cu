// pkv_spec.cu -- speculative acceptance: greedy, and stochastic (modified
// rejection sampling, further down).
//
// "Spending the Idle" 12.4 and "Inference at Scale: KV Cache, Prefill, and
// Decode" section 08: under greedy decoding a drafted token is accepted when it
// equals the target's argmax at that position; acceptance stops at the first
// mismatch and the round always emits one target token (the correction, or
// the bonus token after k accepted drafts).
//
// The row argmax over a 128K vocabulary is an HBM scan.  Each row is split
// across a thread-block cluster of two CTAs (persistent clusters, several rows
// each); partial (value, index) winners are combined through distributed
// shared memory in the cluster's rank-0 CTA.  A second tiny kernel turns the
// k+1 argmaxes of a sequence into the accepted length and the next token.
#include <cooperative_groups.h>

#include "pkv_common.cuh"
#include "pkv_host.h"

namespace cg = cooperative_groups;

namespace pkv {

constexpr int kArgmaxCluster = 2;
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

// max(a, b, c), NaN if any input is NaN (one instruction on sm_100 and later).
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
    float d;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// VW consecutive floats of one load: 256-bit (VW 8), 128-bit (4) or scalar.
template <int VW>
__device__ __forceinline__ void load_vec(const float* p, float* v) {
    if constexpr (VW == 8) {
        asm volatile("ld.global.nc.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
                     : "l"(p));
    } else if constexpr (VW == 4) {
        const float4 q = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = q.x;
        v[1] = q.y;
        v[2] = q.z;
        v[3] = q.w;
    } else {
        v[0] = __ldg(p);
    }
}

// Argmax of each logits row.  A cluster of kArgmaxCluster CTAs owns a row at a
// time, each CTA one contiguous slice of it (a multiple of VW values); the
// CTA's best goes to rank 0 by distributed shared memory.  Clusters are
// persistent (cluster y takes rows y, y + gridDim.y, ...).  Each thread streams
// its part of the slice in chunks of kArgmaxPer values (kArgmaxPer / VW
// loads), two chunk buffers alternating so the next chunk's loads are in
// flight while the current one is scanned.
// At line rate an SM must scan ~5 values per cycle, about one instruction a
// value at most, so the stream does no index work: a NaN-propagating 3-input
// max tree per chunk and, when that maximum beats the thread's best (larger,
// or NaN over a number), a note of the chunk.  At the end of the row the
// thread reloads that one chunk (just streamed, normally still in L2) and
// finds the first index of its best there.  A thread's chunks come in
// increasing index order, so the first chunk holding its maximum holds its
// first occurrence; threads, warps and CTAs merge with the full order (beats).
constexpr int kArgmaxPer = 32;  // values per thread and chunk
template <int VW>
__global__ void __cluster_dims__(kArgmaxCluster, 1, 1) __launch_bounds__(kArgmaxThreads, 3)
    row_argmax_kernel(const float* __restrict__ logits, long long vocab, int rows, int32_t* __restrict__ argmax_out) {
    constexpr int U = kArgmaxPer / VW;  // loads per chunk
    constexpr int T = kArgmaxThreads;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    __shared__ float wv[kArgmaxThreads / 32];
    __shared__ int wi[kArgmaxThreads / 32];
    __shared__ float cv[2][kArgmaxCluster];  // by row parity: one cluster barrier per row
    __shared__ int ci[2][kArgmaxCluster];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    long long per = (vocab + kArgmaxCluster - 1) / kArgmaxCluster;
    per = (per + VW - 1) / VW * VW;
    const long long lo = rank * per;
    const long long hi = lo + per < vocab ? lo + per : vocab;
    const long long nv = hi > lo ? (hi - lo) / VW : 0;                        // loads in this CTA's slice
    const int cpr = (int)((nv + (long long)U * T - 1) / ((long long)U * T));  // chunks per row
    const int nrows = blockIdx.y < rows ? (rows - 1 - (int)blockIdx.y) / (int)gridDim.y + 1 : 0;
    pdl_wait();  // the logits may be the previous kernel's output
    // load u of chunk c of a row: slice load c * U * T + u * T + tid (-inf past the slice)
    auto load_chunk = [&](const float* x, int c, float (&v)[kArgmaxPer]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long j = (long long)c * U * T + (long long)u * T + tid;
            if (j < nv) {
                load_vec<VW>(x + j * VW, v + u * VW);
            } else {
#pragma unroll
                for (int e = 0; e < VW; ++e) v[u * VW + e] = -INFINITY;
            }
        }
    };
    auto chunk_max = [&](const float (&v)[kArgmaxPer]) {
        float m = max3_nan(v[0], v[1], v[2]);
#pragma unroll
        for (int e = 3; e + 1 < kArgmaxPer; e += 2) m = max3_nan(m, v[e], v[e + 1]);
        if constexpr ((kArgmaxPer - 3) % 2) m = max3_nan(m, v[kArgmaxPer - 1], v[kArgmaxPer - 1]);
        return m;
    };
    float a[kArgmaxPer], b[kArgmaxPer];
    for (int rr = 0; rr < nrows; ++rr) {
        const int row = (int)blockIdx.y + rr * (int)gridDim.y;
        const float* x = logits + (long long)row * vocab + lo;
        float bv = -INFINITY;  // the thread's maximum so far (NaN beats all) ...
        int bc = -1;           // ... and the first chunk holding it
        auto note = [&](float m, int c) {
            if (c * U * T + tid < nv && bv == bv && (m != m || m > bv || bc < 0)) {
                bv = m;
                bc = c;
            }
        };
        if (cpr > 0) load_chunk(x, 0, a);
        int c = 0;
        for (; c + 1 < cpr; c += 2) {
            load_chunk(x, c + 1, b);
            note(chunk_max(a), c);
            if (c + 2 < cpr) load_chunk(x, c + 2, a);
            note(chunk_max(b), c + 1);
        }
        if (c < cpr) note(chunk_max(a), c);
        // the first index of the thread's best, from its chunk reloaded
        int bi = kNoIndex;
        if (bc >= 0) {
            load_chunk(x, bc, a);
            const bool mnan = bv != bv;
#pragma unroll
            for (int e = kArgmaxPer - 1; e >= 0; --e) {
                const long long j = (long long)bc * U * T + (long long)(e / VW) * T + tid;
                if (j < nv && (mnan ? a[e] != a[e] : a[e] == bv)) bi = (int)(lo + j * VW + e % VW);
            }
        }
        // CTA reduction, then one cluster barrier: rank 0 merges this row's slots
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
            cluster.map_shared_rank(&cv[rr & 1][0], 0)[rank] = bv;
            cluster.map_shared_rank(&ci[rr & 1][0], 0)[rank] = bi;
        }
        // every CTA's slot for this row is written; rank 0 merges it before it
        // reaches the next row's barrier, so a slot of the same parity is
        // rewritten only after it was read
        cluster.sync();
        if (rank == 0 && tid == 0) {
            float v = cv[rr & 1][0];
            int i = ci[rr & 1][0];
            for (int r = 1; r < kArgmaxCluster; ++r) take(v, i, cv[rr & 1][r], ci[rr & 1][r]);
            argmax_out[row] = i;
        }
    }
    pdl_launch();
}

__global__ void accept_kernel(const int32_t* __restrict__ argmax, const int32_t* __restrict__ draft, int num_seqs,
                              int k, int32_t* __restrict__ accepted, int32_t* __restrict__ next_token) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    pdl_wait();  // the argmax kernel's rows are complete and visible
    pdl_launch();
    if (b >= num_seqs) return;
    const int32_t* am = argmax + (long long)b * (k + 1);
    const int32_t* dr = draft + (long long)b * k;
    int a = 0;
    while (a < k && dr[a] == am[a]) ++a;
    accepted[b] = a;
    next_token[b] = am[a];
}

// ---------------------------------------------------------------------------
// Stochastic acceptance: modified rejection sampling ("Chapter 31 Serving
// Efficiency" 31.5, Example 31.3; "Spending the Idle" 12.4; "Inference at
// Scale" section 08).  Draft x_j is accepted iff r_j * q_j(x_j) < p_j(x_j)
// (fp32); at the first rejection j* the next token is drawn from
// max(0, p_j* - q_j*), or from p_k when all k drafts pass.  The draw is an
// inverse CDF over weights quantised to 2^-32 (integer sums: the same token
// whatever the summation order): T = floor(s * total), token = the first t
// whose inclusive prefix sum exceeds T.
//
// One 8-CTA cluster per sequence: every CTA finds j* (k loads), sums the
// weights of its eighth of the row in token order, keeping one partial sum
// per 128-token segment; the slice totals are exchanged through distributed
// shared memory; the CTA whose slice holds T finds the segment from its
// partial sums and one warp rescans those 128 tokens.  HBM traffic: the p and
// q rows of j* (2 x 4V bytes; 4V when all drafts pass), read once.
// ---------------------------------------------------------------------------
constexpr int kSampleCluster = 8;
constexpr int kSampleThreads = 512;
constexpr int kSampleWarps = kSampleThreads / 32;
constexpr int kSampleChunk = 4 * kSampleThreads;  // tokens per chunk: 4 consecutive per thread
constexpr int kSampleMaxSegs = 1024;               // (chunk, warp) partial sums kept per CTA

__device__ __forceinline__ uint64_t quant32(float x) {
    if (!(x > 0.0f)) return 0;  // <= 0 or NaN
    if (x >= 1.0f) return 1ull << 32;
    return __float2ull_rz(x * 4294967296.0f);  // exact scaling by 2^32, then truncation
}

// floor(s * total) for s in [0, 1), exactly (128-bit product of s's integer
// significand and total).
__device__ __forceinline__ uint64_t scaled_floor(float s, uint64_t total) {
    if (!(s > 0.0f)) return 0;
    if (s >= 1.0f) return total ? total - 1 : 0;
    const uint32_t bits = __float_as_uint(s);
    const int e = (int)((bits >> 23) & 255);
    const uint64_t m = e ? ((bits & 0x7fffffu) | 0x800000u) : (bits & 0x7fffffu);
    const int sh = e ? 150 - e : 149;  // s = m * 2^-sh
    const uint64_t lo = m * total, hi = __umul64hi(m, total);
    if (sh >= 128) return 0;
    if (sh >= 64) return hi >> (sh - 64);
    return (hi << (64 - sh)) | (lo >> sh);
}

// Weights of tokens e0..e0+3 (0 past hi): quantised p - q (residual) or p.
__device__ __forceinline__ void weights4(const float* pr, const float* qr, long long e0, long long hi, bool vec,
                                         int residual, uint64_t w[4]) {
    if (vec && e0 + 3 < hi) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(pr + e0));
        if (residual) {
            const float4 c = __ldg(reinterpret_cast<const float4*>(qr + e0));
            w[0] = quant32(__fsub_rn(a.x, c.x));
            w[1] = quant32(__fsub_rn(a.y, c.y));
            w[2] = quant32(__fsub_rn(a.z, c.z));
            w[3] = quant32(__fsub_rn(a.w, c.w));
        } else {
            w[0] = quant32(a.x);
            w[1] = quant32(a.y);
            w[2] = quant32(a.z);
            w[3] = quant32(a.w);
        }
        return;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const long long t = e0 + u;
        w[u] = 0;
        if (t < hi) {
            const float pv = __ldg(pr + t);
            w[u] = residual ? quant32(__fsub_rn(pv, __ldg(qr + t))) : quant32(pv);
        }
    }
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__global__ void __cluster_dims__(kSampleCluster, 1, 1) __launch_bounds__(kSampleThreads, 2)
    spec_sample_kernel(const float* __restrict__ p, const float* __restrict__ q, const int32_t* __restrict__ draft,
                       const float* __restrict__ r, const float* __restrict__ s, int num_seqs, int k, int vocab,
                       int vec4, int32_t* __restrict__ accepted, int32_t* __restrict__ next_token,
                       int32_t* status) {
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    // partial sums per (chunk, warp) in token order: segment i covers tokens
    // lo + (i / W) * chunk + (i % W) * 128 ... + 127
    __shared__ uint64_t seg[kSampleMaxSegs];
    __shared__ uint64_t wsum[kSampleWarps];
    __shared__ uint64_t slice_total;
    __shared__ uint64_t s_tot[3];  // total, before this slice, this slice
    __shared__ int s_rej, s_bad, s_seg;
    __shared__ uint64_t s_run;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long V = vocab;
    long long per = (V + kSampleCluster - 1) / kSampleCluster;
    per = (per + 3) & ~3LL;
    const long long lo = rank * per < V ? rank * per : V;
    const long long hi = lo + per < V ? lo + per : V;
    const int nchunks = (int)((hi - lo + kSampleChunk - 1) / kSampleChunk);  // <= kSampleMaxSegs / kSampleWarps
    pdl_wait();
    pdl_launch();
    for (int b = blockIdx.y; b < num_seqs; b += gridDim.y) {
        // accepted length: the first draft that fails r * q(x) < p(x)
        if (warp == 0) {
            int rej = k, bad = 0;
            for (int c0 = 0; c0 < k; c0 += 32) {
                const int j = c0 + lane;
                bool ok = true, isbad = false;
                if (j < k) {
                    const int32_t x = draft[(long long)b * k + j];
                    if (x < 0 || x >= vocab) {
                        ok = false;
                        isbad = true;
                    } else {
                        const float px = __ldg(p + ((long long)b * (k + 1) + j) * V + x);
                        const float qx = __ldg(q + ((long long)b * k + j) * V + x);
                        ok = __fmul_rn(__ldg(r + (long long)b * k + j), qx) < px;
                    }
                }
                const unsigned m = __ballot_sync(kFull, !ok);
                if (m) {
                    const int first = __ffs(m) - 1;
                    rej = c0 + first;
                    bad = __shfl_sync(kFull, (int)isbad, first);
                    break;
                }
            }
            if (lane == 0) {
                s_rej = rej;
                s_bad = bad;
            }
        }
        __syncthreads();
        const int j = s_rej;
        const float* pr = p + ((long long)b * (k + 1) + j) * V;
        const float* qr = j < k ? q + ((long long)b * k + j) * V : p;
        const bool vec = vec4 != 0;
        int residual = j < k ? 1 : 0;
        uint64_t total = 0, before = 0, mine = 0;
        for (;;) {
            // one pass over this CTA's slice in token order; each warp keeps the
            // sum of its 128 tokens of every chunk
            uint64_t acc = 0;
#pragma unroll 8
            for (int c = 0; c < nchunks; ++c) {
                uint64_t w[4];
                weights4(pr, qr, lo + (long long)c * kSampleChunk + 4 * tid, hi, vec, residual, w);
                const uint64_t sw = warp_sum_u64(w[0] + w[1] + w[2] + w[3]);
                if (lane == 0) seg[c * kSampleWarps + warp] = sw;
                acc += sw;
            }
            if (lane == 0) wsum[warp] = acc;
            __syncthreads();
            if (warp == 0) {
                uint64_t t = lane < kSampleWarps ? wsum[lane] : 0;
                t = warp_sum_u64(t);
                if (lane == 0) slice_total = t;
            }
            cluster.sync();
            // lanes 0-7 of warp 0 read the slice totals of the cluster once
            if (warp == 0) {
                const uint64_t t = lane < kSampleCluster ? *cluster.map_shared_rank(&slice_total, lane) : 0;
                const uint64_t tot = warp_sum_u64(t);
                const uint64_t bef = warp_sum_u64(lane < rank ? t : 0);
                if (lane == 0) {
                    s_tot[0] = tot;
                    s_tot[1] = bef;
                }
                if (lane == rank) s_tot[2] = t;
            }
            cluster.sync();  // slice_total is rewritten by a second pass; s_tot is complete
            total = s_tot[0];
            before = s_tot[1];
            mine = s_tot[2];
            if (total == 0 && residual) {
                residual = 0;  // no positive residual: draw from p itself
                continue;
            }
            break;
        }
        if (rank == 0 && tid == 0) {
            accepted[b] = j;
            int bits = s_bad && j < k ? PKV_STATUS_BAD_TOKEN : 0;
            if (total == 0) {
                next_token[b] = -1;
                bits |= PKV_STATUS_BAD_DIST;
            }
            if (bits) report(status, bits);
        }
        const uint64_t T = scaled_floor(__ldg(s + b), total);
        if (total > 0 && mine > 0 && T >= before && T - before < mine) {
            // the 128-token segment that holds T (warp 0 scans the segment sums,
            // m consecutive segments per lane), then the token inside it
            if (warp == 0) {
                const int nseg = nchunks * kSampleWarps;
                const int m = (nseg + 31) / 32;
                const int i0 = lane * m, i1 = min(nseg, i0 + m);
                uint64_t mine_s = 0;
                for (int i = i0; i < i1; ++i) mine_s += seg[i];
                uint64_t incl = mine_s;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint64_t y = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += y;
                }
                uint64_t run = before + incl - mine_s;
                if (run <= T && run + mine_s > T) {
                    int i = i0;
                    for (; i < i1 - 1; ++i) {
                        if (run + seg[i] > T) break;
                        run += seg[i];
                    }
                    s_seg = i;
                    s_run = run;
                }
            }
            __syncthreads();
            if (warp == 0) {
                const int i = s_seg;
                const long long e0 = lo + (long long)(i / kSampleWarps) * kSampleChunk + (i % kSampleWarps) * 128 + 4 * lane;
                uint64_t w[4];
                weights4(pr, qr, e0, hi, vec, residual, w);
                const uint64_t mine4 = w[0] + w[1] + w[2] + w[3];
                uint64_t incl = mine4;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint64_t y = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += y;
                }
                const uint64_t run = s_run;
                const uint64_t excl = incl - mine4;
                if (run + excl <= T && run + incl > T) {
                    uint64_t cum = run + excl;
                    int u = 0;
                    for (; u < 3; ++u) {
                        cum += w[u];
                        if (cum > T) break;
                    }
                    next_token[b] = (int32_t)(e0 + u);
                }
            }
        }
        cluster.sync();  // shared state is reused for the next sequence
    }
}

}  // namespace pkv

using namespace pkv;

extern "C" int pkv_spec_accept_sample(const float* p, const float* q, const int32_t* draft, const float* r,
                                      const float* s, int num_seqs, int k, int vocab, int32_t* accepted,
                                      int32_t* next_token, int32_t* status, void* stream) {
    if (num_seqs < 0 || k < 1 || k > 1024 || vocab < 1) return PKV_ERR_SIZE;
    if (num_seqs == 0) return PKV_OK;
    if (!p || !q || !draft || !r || !s || !accepted || !next_token) return PKV_ERR_NULL;
    const int rc = host::check_device();
    if (rc) return rc;
    if ((long long)num_seqs * (k + 1) * vocab > (1LL << 40)) return PKV_ERR_SIZE;
    // each CTA of a cluster keeps one partial sum per (chunk, warp) of its slice
    const long long slice = ((long long)vocab + kSampleCluster - 1) / kSampleCluster + 3;
    if ((slice + kSampleChunk - 1) / kSampleChunk * kSampleWarps > kSampleMaxSegs) return PKV_ERR_SIZE;
    const int vec4 = (vocab % 4 == 0) && host::aligned16(p) && host::aligned16(q);
    dim3 grid(kSampleCluster, (unsigned)(num_seqs < 65535 ? num_seqs : 65535));
    const cudaError_t e = host::launch_pdl(spec_sample_kernel, grid, dim3(kSampleThreads), 0, (cudaStream_t)stream,
                                           p, q, draft, r, s, num_seqs, k, vocab, vec4, accepted, next_token, status);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_spec_accept_greedy(const float* logits, const int32_t* draft, int num_seqs, int k, int vocab,
                                      int32_t* argmax_out, int32_t* accepted, int32_t* next_token, void* stream) {
    if (num_seqs < 0 || k < 1 || k > 64 || vocab < 1) return PKV_ERR_SIZE;
    if (num_seqs == 0) return PKV_OK;
    if (!logits || !draft || !argmax_out || !accepted || !next_token) return PKV_ERR_NULL;
    const int rc = host::check_device();
    if (rc) return rc;
    const long long rows = (long long)num_seqs * (k + 1);
    if (rows > 0x7fffffffLL) return PKV_ERR_SIZE;
    // persistent clusters, as many as are resident at once (at most one per
    // row); 256-bit loads where every slice start is 32-byte aligned, else
    // 128-bit or scalar loads
    const int vw = (vocab % 8 == 0 && host::aligned_to(logits, 32)) ? 8
                   : (vocab % 4 == 0 && host::aligned16(logits)) ? 4 : 1;
    const int vi = vw == 8 ? 2 : vw == 4 ? 1 : 0;
    static int fit_dev[64][3] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return PKV_ERR_CUDA;
    if (fit_dev[dev][vi] == 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kArgmaxCluster, 1);
        cfg.blockDim = dim3(kArgmaxThreads);
        int nc = 0;
        const cudaError_t oe = vw == 8   ? cudaOccupancyMaxActiveClusters(&nc, row_argmax_kernel<8>, &cfg)
                               : vw == 4 ? cudaOccupancyMaxActiveClusters(&nc, row_argmax_kernel<4>, &cfg)
                                         : cudaOccupancyMaxActiveClusters(&nc, row_argmax_kernel<1>, &cfg);
        if (oe != cudaSuccess || nc < 1) nc = 1;
        fit_dev[dev][vi] = nc;
    }
    long long ny = rows < fit_dev[dev][vi] ? rows : fit_dev[dev][vi];
    if (ny < 1) ny = 1;
    if (ny > 65535) ny = 65535;
    const dim3 grid(kArgmaxCluster, (unsigned)ny), block(kArgmaxThreads);
    const cudaStream_t st = (cudaStream_t)stream;
    const cudaError_t le =
        vw == 8   ? host::launch_pdl(row_argmax_kernel<8>, grid, block, 0, st, logits, vocab, (int)rows, argmax_out)
        : vw == 4 ? host::launch_pdl(row_argmax_kernel<4>, grid, block, 0, st, logits, vocab, (int)rows, argmax_out)
                  : host::launch_pdl(row_argmax_kernel<1>, grid, block, 0, st, logits, vocab, (int)rows, argmax_out);
    if (le != cudaSuccess) return PKV_ERR_CUDA;
    return host::launch_pdl(accept_kernel, dim3((num_seqs + 127) / 128), dim3(128), 0, (cudaStream_t)stream,
                            (const int32_t*)argmax_out, draft, num_seqs, k, accepted, next_token) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}
