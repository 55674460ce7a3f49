// pkv_attention.cuh -- paged attention for decode, speculative verification and
// chunked prefill, in one persistent launch.
//
// What it computes ("Inference at Scale: KV Cache, Prefill, and Decode"):
//   section 05  K/V are read through a per-sequence block table;
//   section 07  online softmax (running max m, running sum l, the output
//               rescaled by exp(m_old - m_new)), the FlashAttention block loop,
//               and Flash-Decoding: split K/V into partitions, keep each
//               partition's log-sum-exp statistics, merge with the same
//               rescaling ("Chapter 31 Serving Efficiency", Example 31.2:
//               combine tile statistics, never tile averages);
//   section 08  verification of k drafted tokens is a short causal prefill.
//
// How it runs on GB300 (sm_103a):
//   * A small planning kernel turns (seq_lens, q_lens) into a list of work
//     items (sequence, kv head, partition[, query tile]) -- multi-query items
//     first -- and zeroes the merge tickets.
//   * The attention kernel is persistent (grid = SMs x resident CTAs).  Each CTA
//     has one producer warp and four consumer warps.  The producer takes items
//     from a global atomic queue, reads block-table entries 32 at a time, and
//     streams every 16-token (block, kv head) tile of K and V into an 8-stage
//     shared-memory ring with 2-D TMA loads (128-byte swizzle) completing on
//     mbarriers.  It never waits for compute except through the ring.
//   * Single-query rows (decode, q_len = 1) run on CUDA cores: the g query
//     heads of a GQA group share each K/V tile; 8 lanes own one token's dot
//     product, packed fp32x2 FMAs, a split-butterfly reduction leaves one head
//     per lane pair, warp-shuffle max/sum for the online softmax.  The four
//     consumer warps take alternate tiles and are combined at the end.
//   * Multi-query rows (speculative k > 1, prefill chunks) run on tensor cores
//     (mma.sync m16n8k16 bf16 -> fp32): rows = (query, head) pairs, 16 per
//     warp; S = Q K^T and O += P V with ldmatrix from the swizzled tiles; the
//     causal limit of each row is applied to the scores.
//   * A partition's partial (O, m, l) goes to the workspace; the CTA that
//     finishes the last partition of a group (an atomic ticket, no waiting)
//     merges them in partition order, so results are deterministic.
#pragma once

#include "pkv_common.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr int kTileT = 16;                  // tokens per pipeline stage
constexpr int kCWarps = 4;                  // consumer warps
constexpr int kThreads = (kCWarps + 1) * 32;
constexpr int kStages = 8;
constexpr int kSlots = 4;                   // item descriptors in flight
constexpr int kMqRows = 64;                 // (query, head) rows per multi-query item
constexpr int kMaxParts = 1024;             // partitions per sequence
constexpr int kPlanThreads = 1024;

enum { KIND_END = -1, KIND_DEC = 0, KIND_MQ = 1 };

struct Desc {
    int b, kvh, part, nparts;
    int t_begin, t_end, t_vis, q_row0;
    int nq, kind, pad0, pad1;
};
static_assert(sizeof(Desc) == 48, "descriptor is three int4");

struct AttnParams {
    __nv_bfloat16* out;
    const __nv_bfloat16* q;
    const int32_t* block_tables;
    const int4* items;
    int* hdr;        // [0] item count, [1] queue head
    int* tickets;    // [total_q * n_kv]
    float* part_o;   // [(row * n_q + h) * np_max + part][D]
    float2* part_ml; // [(row * n_q + h) * np_max + part] = (m in log2 units, l)
    int32_t* status;
    int max_blocks, n_q, n_kv, G, bs, num_blocks, np_max, flags;
    float scale_log2;  // scale * log2(e): scores live in base-2 units
};

struct PlanParams {
    const int32_t* seq_lens;
    const int32_t* q_lens;
    int4* items;
    int* hdr;
    int* seq_q0;
    int* seq_flag;
    int* seq_mq_off;
    int* seq_dec_off;
    int* tickets;
    __nv_bfloat16* out;
    int32_t* status;
    int num_seqs, total_q, n_q, n_kv, G, D, P, max_blocks, bs, max_seq_len, decode_ok;
};

template <int D>
struct Smem {
    uint8_t kv[kStages][2][D / 64][kTileT * 128];  // [stage][K,V][128-byte box][16 rows x 128 B], swizzled
    float comb_o[kCWarps][16 * D];                 // per-warp partial O; reused as the [64][D] result
    float comb_m[kCWarps][16];
    float comb_l[kCWarps][16];
    float fin_m[kMqRows];
    float fin_l[kMqRows];
    float pbuf[kCWarps][kTileT * 8];               // decode: p[token][head]
    float corr[kCWarps][8];
    Desc desc[kSlots];
    int poison[kSlots];
    int okw[kCWarps];
    int bcast;
    int abort;
    uint64_t full[kStages], empty[kStages], ifull[kSlots], iempty[kSlots];
};

__device__ __forceinline__ void consumer_bar() { named_bar(1, kCWarps * 32); }

// ---------------------------------------------------------------------------
// Producer warp: item queue, block-table reads, TMA tile stream.
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void producer(Smem<D>& sm, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                         const AttnParams& p, int lane) {
    volatile int* abort = &sm.abort;
    if (lane == 0) {
        prefetch_tmap(tmk);
        prefetch_tmap(tmv);
    }
    const int num_items = p.hdr[0];
    int next = 0;
    if (lane == 0) next = atomicAdd(&p.hdr[1], 1);
    next = __shfl_sync(kFull, next, 0);
    const int box_rows = p.bs < kTileT ? p.bs : kTileT;
    uint32_t g = 0;
    for (int islot = 0;; ++islot) {
        const int si = islot % kSlots;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&sm.iempty[si], ((islot / kSlots) & 1) ^ 1, abort);
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) break;  // abort: publish nothing more
        const int cur = next;
        const bool end = cur >= num_items || *abort;
        Desc d;
        if (!end) {
            const int4 a = p.items[3LL * cur], b = p.items[3LL * cur + 1], c = p.items[3LL * cur + 2];
            d = Desc{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w, c.x, c.y, c.z, c.w};
            if (lane == 0) next = atomicAdd(&p.hdr[1], 1);
            next = __shfl_sync(kFull, next, 0);
        } else {
            d = Desc{0, 0, 0, 1, 0, 0, 0, 0, 0, KIND_END, 0, 0};
        }
        if (lane == 0) {
            sm.desc[si] = d;
            sm.poison[si] = 0;
            mbar_arrive(&sm.ifull[si]);
        }
        if (end) break;
        const int tb = d.t_begin / kTileT, te = (d.t_end + kTileT - 1) / kTileT;
        const int32_t* bt = p.block_tables + (long long)d.b * p.max_blocks;
        const int e_lim = (d.t_end + p.bs - 1) / p.bs;
        int tab_base = -(1 << 30), tab = 0;
        for (int i = tb; i < te; ++i, ++g) {
            const int t0 = i * kTileT;
            const int tvalid = min(kTileT, d.t_end - t0);
            const int e0 = t0 / p.bs;
            const int ne = p.bs >= kTileT ? 1 : (tvalid + p.bs - 1) / p.bs;
            if (e0 < tab_base || e0 + ne > tab_base + 32) {
                tab_base = e0;
                const int e = e0 + lane;
                tab = e < e_lim ? __ldg(bt + e) : 0;
            }
            int my = __shfl_sync(kFull, tab, (e0 - tab_base + lane) & 31);
            const bool in = lane < ne;
            const bool okb = !in || (my >= 0 && my < p.num_blocks);
            if (!okb) my = 0;
            const unsigned badmask = __ballot_sync(kFull, !okb);
            const int s = (int)(g % kStages);
            if (lane == 0) {
                if (badmask) {
                    sm.poison[si] = 1;
                    report(p.status, PKV_STATUS_BAD_BLOCK);
                }
                mbar_wait(&sm.empty[s], ((g / kStages) & 1) ^ 1, abort);
                mbar_arrive_expect_tx(&sm.full[s], 2u * (D / 64) * ne * box_rows * 128u);
            }
            for (int k = 0; k < ne; ++k) {
                const int blk = __shfl_sync(kFull, my, k);
                if (lane == 0) {
                    const int y = (blk * p.n_kv + d.kvh) * p.bs + (p.bs > kTileT ? (t0 % p.bs) : 0);
#pragma unroll
                    for (int x = 0; x < D / 64; ++x) {
                        tma_load_2d(&sm.kv[s][0][x][k * box_rows * 128], tmk, x * 64, y, &sm.full[s]);
                        tma_load_2d(&sm.kv[s][1][x][k * box_rows * 128], tmv, x * 64, y, &sm.full[s]);
                    }
                }
            }
            __syncwarp();
        }
    }
    // drain: wait (bounded) until every issued tile has landed
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) {
            if (g <= (uint32_t)s) continue;
            const uint32_t last = g - 1 - ((g - 1 - s) % kStages);
            mbar_wait(&sm.full[s], (last / kStages) & 1, abort);
        }
    }
}

// ---------------------------------------------------------------------------
// Split-butterfly reduction over the 8 lanes of a group: G partial sums in,
// one full sum out (head li / (8 / G)).
// ---------------------------------------------------------------------------
template <int N>
__device__ __forceinline__ void split_step(float* v, int li, int m) {
    if constexpr (N > 1) {
        const bool up = (li & m) != 0;
#pragma unroll
        for (int j = 0; j < N / 2; ++j) {
            const float send = up ? v[j] : v[j + N / 2];
            const float keep = up ? v[j + N / 2] : v[j];
            v[j] = keep + __shfl_xor_sync(kFull, send, m);
        }
    } else {
        v[0] += __shfl_xor_sync(kFull, v[0], m);
    }
}

template <int G>
__device__ __forceinline__ float reduce8(float* v, int li) {
    split_step<G>(v, li, 4);
    split_step<(G > 1 ? G / 2 : 1)>(v, li, 2);
    split_step<(G > 2 ? G / 4 : 1)>(v, li, 1);
    return v[0];
}

// ---------------------------------------------------------------------------
// Item epilogue: direct bf16 write, or partial + ticket + merge.
// F_o = comb_o viewed as [64][D] (unnormalised), fin_m / fin_l per row.
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void finish_item(Smem<D>& sm, const AttnParams& p, const Desc& d, int R, bool poisoned,
                                            int tid) {
    constexpr int C8 = D / 8;
    const float* Fo = &sm.comb_o[0][0];
    const int G = p.G;
    const float qnan = __int_as_float(0x7fc00000);
    if (d.nparts == 1) {
        for (int e = tid; e < R * C8; e += kCWarps * 32) {
            const int r = e / C8, c = (e - r * C8) * 8;
            const int qi = r / G, hh = r - qi * G;
            const long long orow = (long long)(d.q_row0 + qi) * p.n_q + (long long)d.kvh * G + hh;
            const float inv = 1.0f / sm.fin_l[r];
            const float* src = Fo + r * D + c;
            uint4 v;
            v.x = float2_to_bf16x2(src[0] * inv, src[1] * inv);
            v.y = float2_to_bf16x2(src[2] * inv, src[3] * inv);
            v.z = float2_to_bf16x2(src[4] * inv, src[5] * inv);
            v.w = float2_to_bf16x2(src[6] * inv, src[7] * inv);
            if (poisoned) v = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
            *reinterpret_cast<uint4*>(p.out + orow * D + c) = v;
        }
        return;
    }
    // partial of this partition
    for (int e = tid; e < R * C8; e += kCWarps * 32) {
        const int r = e / C8, c = (e - r * C8) * 8;
        const int qi = r / G, hh = r - qi * G;
        const long long orow = (long long)(d.q_row0 + qi) * p.n_q + (long long)d.kvh * G + hh;
        const float* src = Fo + r * D + c;
        float4 a = make_float4(src[0], src[1], src[2], src[3]);
        float4 b = make_float4(src[4], src[5], src[6], src[7]);
        if (poisoned) a = b = make_float4(qnan, qnan, qnan, qnan);
        float4* dst = reinterpret_cast<float4*>(p.part_o + ((orow * p.np_max + d.part) * D + c));
        __stcg(dst, a);
        __stcg(dst + 1, b);
        if (c == 0) __stcg(p.part_ml + orow * p.np_max + d.part, make_float2(sm.fin_m[r], sm.fin_l[r]));
    }
    __threadfence();
    consumer_bar();
    if (tid == 0) sm.bcast = atomicAdd(&p.tickets[(long long)d.q_row0 * p.n_kv + d.kvh], 1);
    consumer_bar();
    if (sm.bcast != d.nparts - 1) return;
    __threadfence();
    // last partition of this group: merge every partition in order
    const int np = d.nparts;
    float2* W = reinterpret_cast<float2*>(&sm.comb_o[0][0]);
    if (R * np <= 32 * D) {
        for (int e = tid; e < R * np; e += kCWarps * 32) {
            const int r = e / np, pp = e - r * np;
            const int qi = r / G, hh = r - qi * G;
            const long long orow = (long long)(d.q_row0 + qi) * p.n_q + (long long)d.kvh * G + hh;
            W[e] = __ldcg(p.part_ml + orow * p.np_max + pp);
        }
        consumer_bar();
        for (int r = tid; r < R; r += kCWarps * 32) {
            float M = -INFINITY;
            for (int pp = 0; pp < np; ++pp) M = fmaxf(M, W[r * np + pp].x);
            const float mu = M == -INFINITY ? 0.f : M;
            float L = 0.f;
            for (int pp = 0; pp < np; ++pp) L += W[r * np + pp].y * exp2f(W[r * np + pp].x - mu);
            const float invL = 1.0f / L;
            for (int pp = 0; pp < np; ++pp) W[r * np + pp].x = exp2f(W[r * np + pp].x - mu) * invL;
        }
        consumer_bar();
        for (int e = tid; e < R * C8; e += kCWarps * 32) {
            const int r = e / C8, c = (e - r * C8) * 8;
            const int qi = r / G, hh = r - qi * G;
            const long long orow = (long long)(d.q_row0 + qi) * p.n_q + (long long)d.kvh * G + hh;
            float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            const float4* src = reinterpret_cast<const float4*>(p.part_o + (orow * p.np_max) * D + c);
#pragma unroll 4
            for (int pp = 0; pp < np; ++pp) {
                const float w = W[r * np + pp].x;
                const float4 a = __ldcg(src + (long long)pp * (D / 4));
                const float4 b = __ldcg(src + (long long)pp * (D / 4) + 1);
                acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
                acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
            }
            uint4 v;
            v.x = float2_to_bf16x2(acc[0], acc[1]);
            v.y = float2_to_bf16x2(acc[2], acc[3]);
            v.z = float2_to_bf16x2(acc[4], acc[5]);
            v.w = float2_to_bf16x2(acc[6], acc[7]);
            *reinterpret_cast<uint4*>(p.out + orow * D + c) = v;
        }
    } else {
        // many partitions: statistics straight from global memory
        for (int e = tid; e < R * C8; e += kCWarps * 32) {
            const int r = e / C8, c = (e - r * C8) * 8;
            const int qi = r / G, hh = r - qi * G;
            const long long orow = (long long)(d.q_row0 + qi) * p.n_q + (long long)d.kvh * G + hh;
            const float2* ml = p.part_ml + orow * p.np_max;
            float M = -INFINITY;
            for (int pp = 0; pp < np; ++pp) M = fmaxf(M, __ldcg(ml + pp).x);
            const float mu = M == -INFINITY ? 0.f : M;
            float L = 0.f, acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            const float4* src = reinterpret_cast<const float4*>(p.part_o + (orow * p.np_max) * D + c);
            for (int pp = 0; pp < np; ++pp) {
                const float2 s = __ldcg(ml + pp);
                const float w = exp2f(s.x - mu);
                L += s.y * w;
                const float4 a = __ldcg(src + (long long)pp * (D / 4));
                const float4 b = __ldcg(src + (long long)pp * (D / 4) + 1);
                acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
                acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
            }
            const float invL = 1.0f / L;
            uint4 v;
            v.x = float2_to_bf16x2(acc[0] * invL, acc[1] * invL);
            v.y = float2_to_bf16x2(acc[2] * invL, acc[3] * invL);
            v.z = float2_to_bf16x2(acc[4] * invL, acc[5] * invL);
            v.w = float2_to_bf16x2(acc[6] * invL, acc[7] * invL);
            *reinterpret_cast<uint4*>(p.out + orow * D + c) = v;
        }
    }
}

// ---------------------------------------------------------------------------
// Decode item on CUDA cores (q_len = 1, G query heads share the K/V tiles).
// ---------------------------------------------------------------------------
template <int D, int G>
__device__ __forceinline__ void decode_item(Smem<D>& sm, const AttnParams& p, const Desc& d, int warp, int lane,
                                            uint32_t gbase, int ntiles, volatile int* abort) {
    constexpr int NB = D / 64;   // 128-byte boxes per row
    constexpr int HL = 8 / G;    // lanes per head in an 8-lane group
    constexpr int DV = D / 32;   // PV dims per lane
    const int grp = lane >> 3, li = lane & 7;
    const int myh = li / HL;
    float2 q2[G][4 * NB];
    {
        const __nv_bfloat16* qb = p.q + ((long long)d.q_row0 * p.n_q + (long long)d.kvh * G) * D;
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int x = 0; x < NB; ++x) {
                const uint4 v = *reinterpret_cast<const uint4*>(qb + h * D + x * 64 + li * 8);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = bf16x2_to_float2(w[j]);
                    q2[h][4 * x + j] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
                }
            }
        }
    }
    float m_run = -INFINITY, l_run = 0.f;
    float2 acc[G][DV / 2];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int j = 0; j < DV / 2; ++j) acc[h][j] = make_float2(0.f, 0.f);
    const int vbox = DV == 4 ? (lane >> 4) : 0;
    const int vch = DV == 4 ? ((lane & 15) >> 1) : (lane >> 2);
    const int voff = DV == 4 ? ((lane & 1) << 3) : ((lane & 3) << 2);
    const int tb = d.t_begin / kTileT;
    for (int i = warp; i < ntiles; i += kCWarps) {
        const uint32_t gi = gbase + i;
        const int s = (int)(gi % kStages);
        mbar_wait(&sm.full[s], (gi / kStages) & 1, abort);
        const uint8_t* kb = &sm.kv[s][0][0][0];
        const uint8_t* vb = &sm.kv[s][1][0][0];
        const int t0 = (tb + i) * kTileT;
        const int nvalid = min(kTileT, d.t_end - t0);
        float sc[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = grp + 4 * r;
            float2 a[G];
#pragma unroll
            for (int h = 0; h < G; ++h) a[h] = make_float2(0.f, 0.f);
#pragma unroll
            for (int x = 0; x < NB; ++x) {
                const uint4 kv = *reinterpret_cast<const uint4*>(kb + x * (kTileT * 128) + row * 128 +
                                                                 ((li ^ (row & 7)) << 4));
                const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 kf = bf16x2_to_float2(w[j]);
#pragma unroll
                    for (int h = 0; h < G; ++h) a[h] = __ffma2_rn(q2[h][4 * x + j], kf, a[h]);
                }
            }
            float v[G];
#pragma unroll
            for (int h = 0; h < G; ++h) v[h] = a[h].x + a[h].y;
            const float sum = reduce8<G>(v, li);
            sc[r] = row < nvalid ? sum : -INFINITY;
        }
        float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, 16));
        const float m_new = fmaxf(m_run, mt);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        float ps[4], psum = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            ps[r] = exp2f(sc[r] - m_use);
            psum += ps[r];
        }
        psum += __shfl_xor_sync(kFull, psum, 8);
        psum += __shfl_xor_sync(kFull, psum, 16);
        const float cr = exp2f(m_run - m_use);
        l_run = l_run * cr + psum;
        m_run = m_new;
        if ((li % HL) == 0) {
#pragma unroll
            for (int r = 0; r < 4; ++r) sm.pbuf[warp][(grp + 4 * r) * G + myh] = ps[r];
            if (grp == 0) sm.corr[warp][myh] = cr;
        }
        __syncwarp();
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float c = sm.corr[warp][h];
#pragma unroll
            for (int j = 0; j < DV / 2; ++j) acc[h][j] = __fmul2_rn(acc[h][j], make_float2(c, c));
        }
        const uint8_t* vrow = vb + vbox * (kTileT * 128) + voff;
        for (int t = 0; t < nvalid; ++t) {
            float pv[G];
#pragma unroll
            for (int h = 0; h < G; ++h) pv[h] = sm.pbuf[warp][t * G + h];
            const uint8_t* src = vrow + t * 128 + ((vch ^ (t & 7)) << 4);
            if constexpr (DV == 4) {
                const uint2 w = *reinterpret_cast<const uint2*>(src);
                const float2 f0 = bf16x2_to_float2(w.x), f1 = bf16x2_to_float2(w.y);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float2 pp = make_float2(pv[h], pv[h]);
                    acc[h][0] = __ffma2_rn(pp, f0, acc[h][0]);
                    acc[h][1] = __ffma2_rn(pp, f1, acc[h][1]);
                }
            } else {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
                const float2 f0 = bf16x2_to_float2(w);
#pragma unroll
                for (int h = 0; h < G; ++h) acc[h][0] = __ffma2_rn(make_float2(pv[h], pv[h]), f0, acc[h][0]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s], kCWarps);
    }
    // per-warp state -> shared memory, then combine the four warps
    if (grp == 0 && (li % HL) == 0) {
        sm.comb_m[warp][myh] = m_run;
        sm.comb_l[warp][myh] = l_run;
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int j = 0; j < DV / 2; ++j) {
            sm.comb_o[warp][h * D + DV * lane + 2 * j] = acc[h][j].x;
            sm.comb_o[warp][h * D + DV * lane + 2 * j + 1] = acc[h][j].y;
        }
    consumer_bar();
    const int tid = warp * 32 + lane;
    for (int e = tid; e < G * D; e += kCWarps * 32) {
        const int h = e / D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kCWarps; ++w) M = fmaxf(M, sm.comb_m[w][h]);
        const float mu = M == -INFINITY ? 0.f : M;
        float o = 0.f, L = 0.f;
#pragma unroll
        for (int w = 0; w < kCWarps; ++w) {
            const float f = exp2f(sm.comb_m[w][h] - mu);
            o += sm.comb_o[w][e] * f;
            L += sm.comb_l[w][h] * f;
        }
        sm.comb_o[0][e] = o;  // each element is read and written by this thread only
        if (e - h * D == 0) {
            sm.fin_m[h] = M;
            sm.fin_l[h] = L;
        }
    }
    consumer_bar();
}

// ---------------------------------------------------------------------------
// Multi-query item on tensor cores (mma.sync m16n8k16, bf16 in, fp32 acc).
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void mq_item(Smem<D>& sm, const AttnParams& p, const Desc& d, int warp, int lane,
                                        uint32_t gbase, int ntiles, volatile int* abort) {
    const int G = p.G;
    const int R = d.nq * G;
    const int RG = R <= 16 ? 1 : (R <= 32 ? 2 : 4);
    const int TG = kCWarps / RG;
    const int rg = warp % RG, tg = warp / RG;
    const int qd = lane & 3, qr = lane >> 2;
    const int rA = rg * 16 + qr, rB = rA + 8;
    auto row_lim = [&](int r) {
        int qi = r / G;
        if (qi >= d.nq) qi = d.nq - 1;
        return d.t_vis - d.nq + qi;  // last visible position of this row
    };
    const int limA = row_lim(rA), limB = row_lim(rB);
    // Q as A fragments (exact bf16; the softmax scale is applied to the scores)
    uint32_t qf[D / 16][4];
    {
        auto qptr = [&](int r) -> const uint32_t* {
            const int qi = r / G, hh = r - qi * G;
            if (qi >= d.nq) return nullptr;
            return reinterpret_cast<const uint32_t*>(
                p.q + ((long long)(d.q_row0 + qi) * p.n_q + (long long)d.kvh * G + hh) * D);
        };
        const uint32_t* pa = qptr(rA);
        const uint32_t* pb = qptr(rB);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const int w0 = (16 * ks + 2 * qd) >> 1, w1 = w0 + 4;
            qf[ks][0] = pa ? pa[w0] : 0u;
            qf[ks][1] = pb ? pb[w0] : 0u;
            qf[ks][2] = pa ? pa[w1] : 0u;
            qf[ks][3] = pb ? pb[w1] : 0u;
        }
    }
    float o[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    const int tb = d.t_begin / kTileT;
    // ldmatrix row addresses (per lane) inside a tile
    const int mi = lane >> 3, mrow = lane & 7;
    const int k_tok = ((mi >> 1) << 3) + mrow;  // K: matrices (tok 0-7, d lo), (tok 0-7, d hi), (tok 8-15, ...)
    const int k_hi = mi & 1;
    const int v_tok = ((mi & 1) << 3) + mrow;   // V: (tok 0-7, d lo), (tok 8-15, d lo), (tok 0-7, d hi), ...
    const int v_hi = mi >> 1;
    for (int i = tg; i < ntiles; i += TG) {
        const uint32_t gi = gbase + i;
        const int s = (int)(gi % kStages);
        mbar_wait(&sm.full[s], (gi / kStages) & 1, abort);
        const uint32_t kb = smem_u32(&sm.kv[s][0][0][0]);
        const uint32_t vb = smem_u32(&sm.kv[s][1][0][0]);
        const int t0 = (tb + i) * kTileT;
        const int nvalid = min(kTileT, d.t_end - t0);
        float sf[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const int chunk = 2 * ks + k_hi;
            const uint32_t addr = kb + (chunk >> 3) * (kTileT * 128) + k_tok * 128 + (((chunk & 7) ^ (k_tok & 7)) << 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(addr, b0, b1, b2, b3);
            mma_bf16_16816(sf[0], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
            mma_bf16_16816(sf[1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
        }
        // scale, causal / tail mask
        float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int tl = 8 * nt + 2 * qd + (j & 1);
                const int lim = j < 2 ? limA : limB;
                const bool vis = tl < nvalid && t0 + tl <= lim;
                const float v = vis ? sf[nt][j] * p.scale_log2 : -INFINITY;
                sf[nt][j] = v;
                if (j < 2) mxA = fmaxf(mxA, v); else mxB = fmaxf(mxB, v);
            }
        mxA = fmaxf(mxA, __shfl_xor_sync(kFull, mxA, 1));
        mxA = fmaxf(mxA, __shfl_xor_sync(kFull, mxA, 2));
        mxB = fmaxf(mxB, __shfl_xor_sync(kFull, mxB, 1));
        mxB = fmaxf(mxB, __shfl_xor_sync(kFull, mxB, 2));
        const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
        const float uA = nA == -INFINITY ? 0.f : nA, uB = nB == -INFINITY ? 0.f : nB;
        const float cA = exp2f(mA - uA), cB = exp2f(mB - uB);
        float sA = 0.f, sB = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            sf[nt][0] = exp2f(sf[nt][0] - uA);
            sf[nt][1] = exp2f(sf[nt][1] - uA);
            sf[nt][2] = exp2f(sf[nt][2] - uB);
            sf[nt][3] = exp2f(sf[nt][3] - uB);
            sA += sf[nt][0] + sf[nt][1];
            sB += sf[nt][2] + sf[nt][3];
        }
        sA += __shfl_xor_sync(kFull, sA, 1);
        sA += __shfl_xor_sync(kFull, sA, 2);
        sB += __shfl_xor_sync(kFull, sB, 1);
        sB += __shfl_xor_sync(kFull, sB, 2);
        lA = lA * cA + sA;
        lB = lB * cB + sB;
        mA = nA;
        mB = nB;
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
            o[nt][0] *= cA;
            o[nt][1] *= cA;
            o[nt][2] *= cB;
            o[nt][3] *= cB;
        }
        const uint32_t pa0 = float2_to_bf16x2(sf[0][0], sf[0][1]);
        const uint32_t pa1 = float2_to_bf16x2(sf[0][2], sf[0][3]);
        const uint32_t pa2 = float2_to_bf16x2(sf[1][0], sf[1][1]);
        const uint32_t pa3 = float2_to_bf16x2(sf[1][2], sf[1][3]);
        // V rows past the valid tokens may hold anything (even NaN): zero them
        const uint32_t keep0 = (2 * qd < nvalid ? 0x0000ffffu : 0u) | (2 * qd + 1 < nvalid ? 0xffff0000u : 0u);
        const uint32_t keep1 =
            (8 + 2 * qd < nvalid ? 0x0000ffffu : 0u) | (8 + 2 * qd + 1 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
            const int chunk = 2 * dp + v_hi;
            const uint32_t addr = vb + (chunk >> 3) * (kTileT * 128) + v_tok * 128 + (((chunk & 7) ^ (v_tok & 7)) << 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(addr, b0, b1, b2, b3);
            b0 &= keep0;
            b1 &= keep1;
            b2 &= keep0;
            b3 &= keep1;
            mma_bf16_16816(o[2 * dp], pa0, pa1, pa2, pa3, b0, b1);
            mma_bf16_16816(o[2 * dp + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s], (uint32_t)TG);
    }
    // per-warp state -> shared memory
    float* ow = &sm.comb_o[warp][0];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
        const int c = 8 * nt + 2 * qd;
        ow[qr * D + c] = o[nt][0];
        ow[qr * D + c + 1] = o[nt][1];
        ow[(qr + 8) * D + c] = o[nt][2];
        ow[(qr + 8) * D + c + 1] = o[nt][3];
    }
    if (qd == 0) {
        sm.comb_m[warp][qr] = mA;
        sm.comb_l[warp][qr] = lA;
        sm.comb_m[warp][qr + 8] = mB;
        sm.comb_l[warp][qr + 8] = lB;
    }
    consumer_bar();
    const int tid = warp * 32 + lane;
    if (TG > 1) {
        // rows of group rg live in warp rg (tg = 0); fold in warps rg + RG * tg
        for (int e = tid; e < RG * 16 * D; e += kCWarps * 32) {
            const int g = e / (16 * D), loc = e - g * 16 * D, r = loc / D;
            float M = -INFINITY;
            for (int t = 0; t < TG; ++t) M = fmaxf(M, sm.comb_m[g + RG * t][r]);
            const float mu = M == -INFINITY ? 0.f : M;
            float acc = 0.f, L = 0.f;
            for (int t = 0; t < TG; ++t) {
                const float f = exp2f(sm.comb_m[g + RG * t][r] - mu);
                acc += sm.comb_o[g + RG * t][loc] * f;
                L += sm.comb_l[g + RG * t][r] * f;
            }
            sm.comb_o[g][loc] = acc;
            if (loc - r * D == 0) {
                sm.fin_m[g * 16 + r] = M;
                sm.fin_l[g * 16 + r] = L;
            }
        }
    } else {
        for (int r = tid; r < kMqRows; r += kCWarps * 32) {
            sm.fin_m[r] = sm.comb_m[r >> 4][r & 15];
            sm.fin_l[r] = sm.comb_l[r >> 4][r & 15];
        }
    }
    consumer_bar();
}

// ---------------------------------------------------------------------------
// Consumer warps
// ---------------------------------------------------------------------------
template <int D, int GD>
__device__ __forceinline__ void consumer(Smem<D>& sm, const AttnParams& p, int warp, int lane) {
    volatile int* abort = &sm.abort;
    const int tid = warp * 32 + lane;
    uint32_t g = 0;
    for (int islot = 0;; ++islot) {
        const int si = islot % kSlots;
        const bool ok = mbar_wait(&sm.ifull[si], (islot / kSlots) & 1, abort);
        if (lane == 0) sm.okw[warp] = ok ? 1 : 0;
        consumer_bar();
        const Desc d = sm.desc[si];
        bool go = d.kind != KIND_END;
#pragma unroll
        for (int w = 0; w < kCWarps; ++w) go = go && sm.okw[w] != 0;
        consumer_bar();  // okw is rewritten next item
        if (!go) break;
        const int ntiles = (d.t_end + kTileT - 1) / kTileT - d.t_begin / kTileT;
        int R;
        if constexpr (GD > 0) {
            if (d.kind == KIND_DEC) {
                decode_item<D, GD>(sm, p, d, warp, lane, g, ntiles, abort);
                R = GD;
            } else {
                mq_item<D>(sm, p, d, warp, lane, g, ntiles, abort);
                R = d.nq * p.G;
            }
        } else {
            mq_item<D>(sm, p, d, warp, lane, g, ntiles, abort);
            R = d.nq * p.G;
        }
        const bool poisoned = sm.poison[si] != 0;
        finish_item<D>(sm, p, d, R, poisoned, tid);
        consumer_bar();  // comb buffers are free again
        if (lane == 0) mbar_arrive(&sm.iempty[si]);
        g += (uint32_t)ntiles;
    }
}

template <int D, int GD>
__global__ void __launch_bounds__(kThreads, 2)
    paged_attention_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                           const __grid_constant__ AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    Smem<D>& sm = *reinterpret_cast<Smem<D>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kCWarps);
        }
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&sm.ifull[i], 1);
            mbar_init(&sm.iempty[i], kCWarps);
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == kCWarps) {
        producer<D>(sm, &tmk, &tmv, p, lane);
    } else {
        consumer<D, GD>(sm, p, warp, lane);
    }
    if (threadIdx.x == 0 && sm.abort) report(p.status, PKV_STATUS_TIMEOUT);
}

template <int D, int GD>
int launch_attention(const CUtensorMap& tmk, const CUtensorMap& tmv, const AttnParams& p, long long max_items,
                            cudaStream_t st) {
    static int configured[64] = {0};
    static int occ[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = sizeof(Smem<D>) + 1024;
    if (dev < 0 || dev >= 64) return PKV_ERR_CUDA;
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(paged_attention_kernel<D, GD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return PKV_ERR_CUDA;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, paged_attention_kernel<D, GD>, kThreads, smem) !=
                cudaSuccess ||
            n < 1)
            return PKV_ERR_CUDA;
        occ[dev] = n;
        configured[dev] = 1;
    }
    long long grid = (long long)host::sm_count() * occ[dev];
    if (grid > max_items) grid = max_items;
    if (grid < 1) grid = 1;
    paged_attention_kernel<D, GD><<<(unsigned)grid, kThreads, smem, st>>>(tmk, tmv, p);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <int D>
int dispatch_g(int GD, const CUtensorMap& tmk, const CUtensorMap& tmv, const AttnParams& p, long long mi,
                      cudaStream_t st) {
    switch (GD) {
        case 1: return launch_attention<D, 1>(tmk, tmv, p, mi, st);
        case 2: return launch_attention<D, 2>(tmk, tmv, p, mi, st);
        case 4: return launch_attention<D, 4>(tmk, tmv, p, mi, st);
        case 8: return launch_attention<D, 8>(tmk, tmv, p, mi, st);
        default: return launch_attention<D, 0>(tmk, tmv, p, mi, st);
    }
}


int dispatch_attention_d64(int GD, const CUtensorMap& tmk, const CUtensorMap& tmv, const AttnParams& p, long long mi, cudaStream_t st);
int dispatch_attention_d128(int GD, const CUtensorMap& tmk, const CUtensorMap& tmv, const AttnParams& p, long long mi, cudaStream_t st);

}  // namespace pkv
