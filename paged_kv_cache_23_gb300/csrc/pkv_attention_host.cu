// pkv_attention_host.cu -- planning kernel, workspace layout and the C entry
// points of the paged attention (kernels in pkv_attention.cuh).
#include <string.h>

#include "pkv_attention.cuh"

namespace pkv {

struct PlanParams {
    const int32_t* seq_lens;
    const int32_t* q_lens;
    int4* items;     // {b, part, qt, hg}
    int4* seqs;      // {seq_len, q_len, first query row, kind | hps << 4 | wph << 8 | qt_len << 12}
    int* hdr;
    int* seq_q0;     // first query row
    int* seq_flag;   // PKV_STATUS_* bits of the sequence (0 = valid)
    int* seq_mq;     // exclusive prefix of multi-query item counts
    int* seq_p;      // partition length of each sequence (read by the attention kernel)
    int* row_np;     // [total_q] partitions of each query row (-1: row of an invalid sequence)
    int32_t* status;
    int num_seqs, total_q, n_q, n_kv, G, D, P, max_blocks, bs, max_seq_len, max_q_len, decode_ok;
    int fp8;         // e4m3 pool: every row on the transposed tensor-core item
    int tc;          // tcgen05 tiles allowed (head_dim 128, bf16, block_size >= 16, P % 128 == 0)
    int adapt_P;     // 1: P is a floor; the planning kernel sizes each sequence's partitions
    int sms;         // SM count (persistent CTAs of the attention kernel)
    int plan_key;    // key of the shape this plan is made for (header int 4)
};

__host__ __device__ inline int gcd_pow2(int n, int m) {  // largest power of two <= m dividing n (m a power of 2)
    int h = m;
    while (h > 1 && n % h) h >>= 1;
    return h;
}

// Shape of the work of one sequence: kind, kv heads per stage, warps per kv
// head, queries per tile.
struct SeqShape {
    int kind, hps, wph, qt;
};

// decode_fma: run q_len = 1 rows on the CUDA-core path (else tensor cores).
// fp8: e4m3 pool -- tiles of up to 16 (query, q head) columns per kv head.
// bf16 q_len * g <= kDecCols (24): one tile of q_len queries on the
// transposed tensor-core item (decode_tc_item) -- decode rows and short
// verifications (k = 5 drafts at g = 4: 20 columns), one warp per kv head,
// every kv head of a block in one stage; longer multi-query rows on mma.sync
// row tiles (mq_item).
// tc: a sequence with more than kTcMinCols (= kDecCols) (query, q head) rows
// per kv head runs as tcgen05 tiles of 128 rows (128 / G queries), one kv
// head each.
__device__ __forceinline__ SeqShape seq_shape(int ql, int G, int n_kv, int decode_fma, int fp8, int tc) {
    SeqShape s;
    if (tc && ql * G > kTcMinCols && kTcRows % G == 0) {
        s.kind = KIND_TC;
        s.hps = 1;
        s.wph = kCWarps;
        s.qt = kTcRows / G;
        return s;
    }
    if (fp8) {
        s.kind = KIND_DEC;
        s.hps = gcd_pow2(n_kv, kMaxHPS);
        s.wph = 1;
        s.qt = G <= 16 ? 16 / G : 1;
        return s;
    }
    if (ql <= 1 && G <= 8 && decode_fma) {
        s.kind = KIND_DECF;
        s.hps = gcd_pow2(n_kv, kMaxHPS);
        s.wph = 1;
        s.qt = 1;
        return s;
    }
    if (ql * G <= kDecCols) {
        // decode rows and short verifications: one query tile of up to 24
        // (query, q head) columns per kv head, one warp per kv head, so every
        // kv head of a block shares a stage
        s.kind = KIND_DEC;
        s.hps = gcd_pow2(n_kv, kMaxHPS);
        s.wph = 1;
        s.qt = ql > 1 ? ql : 1;
        return s;
    }
    s.kind = KIND_MQ;
    const int rows = ql * G;
    int w = 1;
    while (w < kCWarps && 16 * w < rows) w <<= 1;
    while (w < kCWarps && 16 * w < G) w <<= 1;
    s.wph = w;
    s.hps = gcd_pow2(n_kv, kCWarps / w);
    s.qt = (16 * w) / G;
    return s;
}

__device__ __forceinline__ int mq_parts_of(int L, int ql, int QT, int P) {
    int n = 0;
    for (int qt = 0; qt * QT < ql; ++qt) {
        const int last = min(ql, (qt + 1) * QT);
        n += ceil_div(L - ql + last, P);
    }
    return n;
}

// Largest i in [0, n) with a[i] <= x, for a non-decreasing a with a[0] <= x.
__device__ __forceinline__ int last_le(const int* a, int n, int x) {
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

constexpr int kPlanSmemSeqs = 1024;  // batches up to this size keep their records in shared memory

// Block-wide exclusive scans of K ints per thread at once (blockDim.x ==
// 1024): one pair of barriers for all K.  `tmp` holds 32 * K ints; v is
// replaced by its exclusive prefixes and tot receives the block sums.
template <int K>
__device__ __forceinline__ void block_scan_k(int (&v)[K], int (&tot)[K], int* tmp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        x[k] = v[k];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, x[k], o);
            if (lane >= o) x[k] += y;
        }
        if (lane == 31) tmp[warp * K + k] = x[k];
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            int w = tmp[lane * K + k];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, w, o);
                if (lane >= o) w += y;
            }
            tmp[lane * K + k] = w;  // inclusive prefix over warps
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < K; ++k) {
        tot[k] = tmp[31 * K + k];
        v[k] = (warp > 0 ? tmp[(warp - 1) * K + k] : 0) + x[k] - v[k];
    }
    __syncthreads();
}
constexpr int kAutoPMax = 8192;       // automatic partition length: upper bound of the target
constexpr int kAutoItemsPerSM = 2;    // automatic partition length: target items per SM

// Partition length of one sequence.  Explicit: P.  Automatic: the sequence's
// L positions are cut into n = round(L / C) partitions of (nearly) equal
// length, C being the batch's target item length, rounded up to whole stages
// (16 tokens, 128 for tcgen05 tiles) and no shorter than the floor P (so no
// row ever has more partitions than the workspace holds).  Uniform partitions
// of one length leave each sequence a short tail and the batch a ragged last
// wave of the dynamic queue; equal cuts make every item of the batch about C
// long.
// adapt: 0 explicit; 1 nearest count, n = round(L / C) (items about C long,
// up to 1.5 C); 2 ceiling count, n = ceil(L / C) (items at most C long).
__device__ __forceinline__ int seq_partition(int L, int C, int P, int align, int adapt) {
    if (!adapt) return P;
    const int n = adapt == 2 ? max(1, ceil_div(L, C)) : max(1, (L + C / 2) / C);
    const int pb = ceil_div(ceil_div(L, n), align) * align;
    return max(pb, P);
}

// Granularity of automatic partition lengths: whole stages -- 128 tokens for
// tcgen05 tiles, 32 (two 16-token stages) for FP8 pools, whose items consume
// stages in pairs, else 16.
__device__ __forceinline__ int part_align(int kind, int fp8) {
    return kind == KIND_TC ? kTcT : fp8 ? 2 * kTileT : kTileT;
}

// Items of one sequence for partition length pb: np partitions of each of its
// query tiles, times its head groups.
__device__ __forceinline__ int seq_items(int L, int ql, const SeqShape& sh, int pb, int ngroups) {
    int cnt = 0;
    for (int qt = 0; qt * sh.qt < ql; ++qt) cnt += ceil_div(L - ql + qt * sh.qt + min(sh.qt, ql - qt * sh.qt), pb);
    return cnt * ngroups;
}

// Longest-first class of an item of `len` positions, items no longer than Pn
// (inv = kTailBuckets / Pn): 0 for the longest.  In fp32: the class only
// orders the queue, and a 64-bit integer division per item was a third of
// the planning kernel's time.
__device__ __forceinline__ int len_bucket(int len, int Pn, float inv) {
    const int b = __float2int_rz((float)(Pn - len) * inv);
    return min(kTailBuckets - 1, max(0, b));
}

// Work list for a batch: multi-query items first (mma.sync rows and tcgen05
// tiles: compute-heavy, started early), in sequence order; then every
// decode-style item (decode rows and transposed short verifications) ordered
// longest first by a counting sort over kTailBuckets length classes, so the
// dynamic queue ends on the shortest items.  The list depends only on the
// lengths, so one plan serves every layer of a decode step.
//   pass A  one thread per sequence: validity, query rows, partition length,
//           multi-query item counts and their prefix sums, length-class
//           histogram of the other items;
//   pass B  multi-query items written over the item index space (one thread
//           per item, which finds its sequence by binary search in the prefix
//           sums, so consecutive threads write consecutive 16-byte items);
//           decode-style items by one thread per sequence into ranges it
//           reserves in its items' length classes; per-row partition counts.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ PlanParams pp) {
    __shared__ int tmp[32 * 2];
    __shared__ int hist[kTailBuckets];
    __shared__ int s_q0[kPlanSmemSeqs], s_mq[kPlanSmemSeqs], s_p[kPlanSmemSeqs], s_flag[kPlanSmemSeqs];
    __shared__ int4 s_seq[kPlanSmemSeqs];
    __shared__ int s_len[kPlanSmemSeqs], s_ql[kPlanSmemSeqs], s_cnt[32];
    const int tid = threadIdx.x;
    const int n = pp.num_seqs;
    const bool small = n <= kPlanSmemSeqs;
    int* a_q0 = small ? s_q0 : pp.seq_q0;
    int* a_mq = small ? s_mq : pp.seq_mq;
    int* a_p = small ? s_p : pp.seq_p;
    int* a_flag = small ? s_flag : pp.seq_flag;
    const int4* a_seq = small ? s_seq : pp.seqs;  // per-sequence records of pass A (global copy always written)
    if (tid < kTailBuckets) hist[tid] = 0;
    // Programmatic launch: the attention kernel may be scheduled at once (it
    // waits for this grid to complete before it reads the plan), but this
    // kernel reads nothing before the previous kernel of the stream has
    // completed and its writes are visible -- seq_lens and q_lens may be the
    // output of that very kernel (a caller advancing its lengths on the GPU),
    // and the work list may still be read by a previous call's kernels.
    pdl_launch();
    pdl_wait();
    // this thread's first sequence, read once for the target length and pass A
    const int L0 = tid < n ? pp.seq_lens[tid] : 0, ql0 = tid < n ? pp.q_lens[tid] : 0;
    const int P = pp.P;  // explicit length, or the floor of the automatic ones
    int C = P;           // target item length
    int rule = 0;        // seq_partition's adapt mode
    if (pp.adapt_P) {
        // about kAutoItemsPerSM items per SM over the batch's work (positions
        // x head groups x query tiles), each no shorter than the floor
        long long tok = 0, tok_rows = 0;
        for (int b = tid; b < n; b += kPlanThreads) {
            const int L = b == tid ? L0 : pp.seq_lens[b], ql = b == tid ? ql0 : pp.q_lens[b];
            if (small) {
                s_len[b] = L;
                s_ql[b] = ql;
            }
            if (L <= 0 || ql <= 0 || ql > L || L > pp.max_seq_len || ql > pp.max_q_len) continue;
            const SeqShape sh = seq_shape(ql, pp.G, pp.n_kv, pp.decode_ok, pp.fp8, pp.tc);
            const long long t = (long long)L * (pp.n_kv / sh.hps) * ceil_div(ql, sh.qt);
            tok += t;
            if (ql > 1 && !multi_query_kind(sh.kind)) tok_rows += t;
        }
        // block sums in units of 16 tokens (fit an int for any accepted batch)
        const int cap = (1 << 30) / kPlanThreads;
        int v2[2] = {(int)min(tok >> 4, (long long)cap), (int)min(tok_rows >> 4, (long long)cap)}, t2[2];
        block_scan_k<2>(v2, t2, tmp);
        const int per = kAutoItemsPerSM * pp.sms;
        const int c16 = (t2[0] + per - 1) / per;  // in units of 16 tokens
        C = max(P, min(kAutoPMax / kTileT, c16) * kTileT);
        rule = 1;
        if (small && 2LL * t2[1] > t2[0]) {
            // Mostly multi-row decode-style items (speculative verification):
            // each writes q_len times the partial results of a decode item, so
            // the batch runs best as one wave -- the shortest item length whose
            // items (ceiling counts, every item at most C long) fit on the
            // SMs.  Warp j tries C_lo (16 + j) / 16, C_lo the length of
            // perfectly even items; the smallest that fits wins.
            const int warp = tid >> 5, lane = tid & 31;
            const int c_lo = max(P / kTileT, (t2[0] + pp.sms - 1) / pp.sms);
            const int cj = min(kAutoPMax / kTileT, (c_lo * (16 + warp) + 15) / 16) * kTileT;
            int cnt = 0;
            for (int b = lane; b < n; b += 32) {
                const int L = s_len[b], ql = s_ql[b];
                if (L <= 0 || ql <= 0 || ql > L || L > pp.max_seq_len || ql > pp.max_q_len) continue;
                const SeqShape sh = seq_shape(ql, pp.G, pp.n_kv, pp.decode_ok, pp.fp8, pp.tc);
                const int pb = seq_partition(L, cj, P, part_align(sh.kind, pp.fp8), 2);
                cnt += seq_items(L, ql, sh, pb, pp.n_kv / sh.hps);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
            if (lane == 0) s_cnt[warp] = cnt;
            __syncthreads();
            int best = -1;
            for (int j = 0; j < 32 && best < 0; ++j)
                if (s_cnt[j] <= pp.sms) best = j;
            if (best >= 0) {
                C = min(kAutoPMax / kTileT, (c_lo * (16 + best) + 15) / 16) * kTileT;
                rule = 2;
            }
        }
    }
    // item lengths are at most Pn: explicit P, or 1.5 C + one 128-token round-up
    const int Pn = pp.adapt_P ? 2 * C : P;
    const float inv_pn = (float)kTailBuckets / (float)Pn;
    if (tid == 0) pp.hdr[HDR_P] = C;
    __syncthreads();
    int bits = 0, any_tc = 0;
    // pass A
    long long carry = 0;
    int c_mq = 0;
    for (int base = 0; base < n; base += kPlanThreads) {
        const int b = base + tid;
        int qlc = 0, flag = 0, L = 0, ql = 0;
        if (b < n) {
            L = b == tid ? L0 : pp.seq_lens[b];
            ql = b == tid ? ql0 : pp.q_lens[b];
            if (L < 0 || (long long)L > (long long)pp.max_blocks * pp.bs || L > pp.max_seq_len)
                flag |= PKV_STATUS_BAD_SEQLEN;
            if (ql < 0 || ql > L || ql > pp.max_q_len) flag |= PKV_STATUS_BAD_QLEN;
            // clamp so the scan cannot overflow (total_q <= 2^20 is checked on the host)
            qlc = ql > 0 ? min(ql, pp.total_q + 1) : 0;
        }
        int tot;
        const int ex = block_exclusive_scan_1024(qlc, tmp, &tot);
        int nmq = 0, q0 = 0;
        if (b < n) {
            const long long q0l = carry + ex;
            if (q0l + qlc > pp.total_q) flag |= PKV_STATUS_BAD_QLEN;  // rows would overflow q/out
            q0 = (int)(q0l < pp.total_q ? q0l : pp.total_q);
            bits |= flag;
            const SeqShape sh = seq_shape(ql, pp.G, pp.n_kv, pp.decode_ok, pp.fp8, pp.tc);
            const int ngroups = pp.n_kv / sh.hps;
            const int pb = seq_partition(L, C, P, part_align(sh.kind, pp.fp8), rule);
            if (flag == 0 && ql > 0) {
                if (sh.kind == KIND_TC) any_tc = 1;
                if (multi_query_kind(sh.kind)) {
                    nmq = mq_parts_of(L, ql, sh.qt, pb) * ngroups;
                } else {
                    // query tile qt sees t_vis positions: np - 1 items of pb and a tail
                    for (int qt = 0; qt * sh.qt < ql; ++qt) {
                        const int nq = min(sh.qt, ql - qt * sh.qt);
                        const int tv = L - ql + qt * sh.qt + nq;
                        const int np = ceil_div(tv, pb);
                        if (np > 1) atomicAdd(&hist[len_bucket(pb, Pn, inv_pn)], (np - 1) * ngroups);
                        atomicAdd(&hist[len_bucket(tv - (np - 1) * pb, Pn, inv_pn)], ngroups);
                    }
                }
            }
            const int4 rec = make_int4(L, ql, q0, sh.kind | (sh.hps << 4) | (sh.wph << 8) | (sh.qt << 12));
            pp.seqs[b] = rec;
            pp.seq_p[b] = pb;
            if (small) {
                s_seq[b] = rec;
                s_p[b] = pb;
            }
            a_flag[b] = flag;
        }
        carry += tot;
        int v1[1] = {nmq}, t1[1];
        block_scan_k<1>(v1, t1, tmp);
        if (b < n) {
            a_q0[b] = q0;
            a_mq[b] = c_mq + v1[0];
        }
        c_mq += t1[0];
    }
    // length classes -> first slot of each class (exclusive scan), after the
    // multi-query items
    any_tc = __syncthreads_or(any_tc);
    int c_dec;
    {
        const int v = tid < kTailBuckets ? hist[tid] : 0;
        const int ex = block_exclusive_scan_1024(v, tmp, &c_dec);
        if (tid < kTailBuckets) hist[tid] = c_mq + ex;
    }
    if (tid == 0) {
        pp.hdr[HDR_ITEMS] = c_mq + c_dec;
        pp.hdr[HDR_HEAD] = 0;
        pp.hdr[HDR_TC] = any_tc;  // the attention kernel allocates tensor memory only then
        pp.hdr[HDR_KEY] = pp.plan_key;
    }
    __syncthreads();
    // pass B1: one thread per sequence -- decode-style items, reserved per
    // length class (the order inside a class does not matter: every item's
    // partial lands at its own (row, partition) index)
    for (int b = tid; b < n; b += kPlanThreads) {
        const int4 sq = a_seq[b];
        const int L = sq.x, ql = sq.y;
        if (a_flag[b] || ql <= 0) continue;  // invalid rows are written NaN by each call's combine kernel
        if (multi_query_kind(sq.w & 15)) continue;
        const int ngroups = pp.n_kv / ((sq.w >> 4) & 15);
        const int QT = (sq.w >> 12) & 4095;
        const int pb = a_p[b];
        for (int qt = 0; qt * QT < ql; ++qt) {
            const int nq = min(QT, ql - qt * QT);
            const int tv = L - ql + qt * QT + nq;
            const int np = ceil_div(tv, pb);
            if (np > 1) {
                int at = atomicAdd(&hist[len_bucket(pb, Pn, inv_pn)], (np - 1) * ngroups);
                for (int part = 0; part < np - 1; ++part)
                    for (int hg = 0; hg < ngroups; ++hg) pp.items[at++] = make_int4(b, part, qt, hg);
            }
            const int at = atomicAdd(&hist[len_bucket(tv - (np - 1) * pb, Pn, inv_pn)], ngroups);
            for (int hg = 0; hg < ngroups; ++hg) pp.items[at + hg] = make_int4(b, np - 1, qt, hg);
        }
    }
    // pass B2: multi-query items
    for (int it = tid; it < c_mq; it += kPlanThreads) {
        const int b = last_le(a_mq, n, it);
        int li = it - a_mq[b];
        const int4 sq = a_seq[b];
        const int L = sq.x, ql = sq.y, QT = (sq.w >> 12) & 4095;
        const int ngroups = pp.n_kv / ((sq.w >> 4) & 15);
        const int pb = a_p[b];
        for (int qt = 0; qt * QT < ql; ++qt) {
            const int nq = min(QT, ql - qt * QT);
            const int cnt = ceil_div(L - ql + qt * QT + nq, pb) * ngroups;
            if (li < cnt) {
                const int part = li / ngroups;
                pp.items[it] = make_int4(b, part, qt, li - part * ngroups);
                break;
            }
            li -= cnt;
        }
    }
    // pass B3: partitions per query row; -1 for the rows of an invalid
    // sequence (inside the q/out extent), which each call's combine kernel
    // writes NaN; 0 for rows past the last sequence's queries
    for (int r = tid; r < pp.total_q; r += kPlanThreads) {
        int np = 0;
        if (r < carry) {
            const int b = last_le(a_q0, n, r);
            const int4 sq = a_seq[b];
            const int L = sq.x, ql = sq.y, q0 = sq.z;
            if (a_flag[b] != 0) {
                const int qlc = ql > 0 ? min(ql, pp.total_q) : 0;
                if (r - q0 < qlc) np = -1;
            } else if (r - q0 < ql) {
                // query tile of row r; a decode row is a tile of one query
                const int QT = (sq.w >> 12) & 4095;
                const int qt = (r - q0) / QT;
                const int nq = min(QT, ql - qt * QT);
                np = ceil_div(L - ql + qt * QT + nq, a_p[b]);
            }
        }
        pp.row_np[r] = np;
    }
    if (bits) report(pp.status, bits);
}

struct WsLayout {
    size_t hdr, items, seqs, seqaux, rownp, ml, o, total;
    long long max_items;
    int np_max;
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static WsLayout ws_layout(int num_seqs, int total_q, int n_q, int n_kv, int D, int max_seq_len, int P) {
    WsLayout w{};
    w.np_max = max_seq_len > 0 ? (max_seq_len + P - 1) / P : 1;
    if (w.np_max < 1) w.np_max = 1;
    w.max_items = (long long)total_q * w.np_max * n_kv;
    size_t off = 0;
    w.hdr = off;
    off = align256(off + 64);
    w.items = off;
    off = align256(off + (size_t)w.max_items * sizeof(int4));
    w.seqs = off;
    off = align256(off + (size_t)num_seqs * sizeof(int4));
    w.seqaux = off;
    off = align256(off + (size_t)num_seqs * 4 * sizeof(int));
    w.rownp = off;
    off = align256(off + (size_t)total_q * sizeof(int));
    w.ml = off;
    off = align256(off + (size_t)total_q * n_q * w.np_max * sizeof(float2));
    w.o = off;
    off = align256(off + (size_t)total_q * n_q * w.np_max * D * sizeof(float));
    w.total = off;
    return w;
}

}  // namespace pkv

using namespace pkv;

extern "C" int pkv_attention_auto_partition(int num_seqs, int total_q, int num_kv_heads, int max_seq_len) {
    (void)num_seqs;
    (void)total_q;
    (void)num_kv_heads;
    int P = 512;
    while (max_seq_len > 0 && (max_seq_len + P - 1) / P > kMaxParts) P *= 2;
    return P;
}

extern "C" size_t pkv_attention_workspace_bytes(int num_seqs, int total_q, int num_q_heads, int num_kv_heads,
                                                int head_dim, int max_seq_len, int partition_tokens) {
    if (num_seqs < 0 || total_q < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1 || max_seq_len < 0)
        return 0;
    int P = partition_tokens > 0 ? partition_tokens
                                 : pkv_attention_auto_partition(num_seqs, total_q, num_kv_heads, max_seq_len);
    return ws_layout(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, max_seq_len, P).total;
}

namespace {

// Everything the host derives from one call's sizes and flags: checked once,
// shared by the plan and the run, and condensed into the key the plan leaves
// in the workspace header (a run over a workspace planned for another shape
// does nothing and reports PKV_STATUS_BAD_PLAN).
struct Shape {
    int num_seqs, total_q, max_q_len, max_seq_len, max_blocks, n_q, n_kv, D, bs, flags;
    int G, GD, P, adapt;
    bool fp8, decode_fma, tc, empty;
    WsLayout w;
    int key;
};

// FNV-1a over the fields that decide the work list and the workspace layout,
// folded to a positive nonzero int.
int shape_key(const Shape& s) {
    const long long f[] = {s.num_seqs, s.total_q, s.max_q_len, s.max_seq_len, s.max_blocks, s.n_q, s.n_kv, s.D,
                           s.bs, s.P, s.adapt, s.fp8, s.decode_fma, s.tc, s.w.np_max};
    uint32_t h = 2166136261u;
    for (long long v : f)
        for (int k = 0; k < 8; ++k) {
            h ^= (uint32_t)((unsigned long long)v >> (8 * k)) & 0xffu;
            h *= 16777619u;
        }
    return (int)((h & 0x7fffffffu) | 1u);
}

// Host checks of a call's sizes (no pointers); PKV_OK and a filled Shape, or
// an error code.  fp8: e4m3 pools.
int check_shape(Shape& s, bool fp8, int num_seqs, int total_q, int max_q_len, int max_seq_len, int max_blocks,
                int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks, int partition_tokens,
                int flags) {
    if (num_seqs < 0 || total_q < 0 || max_q_len < 0 || max_blocks < 1 || max_seq_len < 0 || num_q_heads < 1 ||
        num_kv_heads < 1 || num_blocks < 1 || block_size < 1)
        return PKV_ERR_SIZE;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads) return PKV_ERR_UNSUPPORTED;
    const int G = num_q_heads / num_kv_heads;
    if (G > 64) return PKV_ERR_UNSUPPORTED;
    if ((block_size & (block_size - 1)) || block_size > 256) return PKV_ERR_UNSUPPORTED;
    if ((long long)num_blocks * num_kv_heads * block_size >= (1LL << 31)) return PKV_ERR_SIZE;
    if (flags & ~(PKV_ATTN_DECODE_CUDA_CORES | PKV_ATTN_NO_TCGEN05)) return PKV_ERR_SIZE;
    if (fp8 && (head_dim != 128 || G > 16)) return PKV_ERR_UNSUPPORTED;
    s = Shape{};
    s.empty = num_seqs == 0 || total_q == 0;
    if (s.empty) return PKV_OK;
    if (num_seqs > (1 << 24) || total_q > (1 << 20)) return PKV_ERR_SIZE;
    int P = partition_tokens;
    if (P == 0) P = pkv_attention_auto_partition(num_seqs, total_q, num_kv_heads, max_seq_len);
    if (P < kTileT || P % kTileT) return PKV_ERR_SIZE;
    s.w = ws_layout(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, max_seq_len, P);
    if (s.w.np_max > kMaxParts) return PKV_ERR_SIZE;
    if (s.w.max_items > 0x7fffffffLL) return PKV_ERR_SIZE;
    s.num_seqs = num_seqs;
    s.total_q = total_q;
    s.max_q_len = max_q_len;
    s.max_seq_len = max_seq_len;
    s.max_blocks = max_blocks;
    s.n_q = num_q_heads;
    s.n_kv = num_kv_heads;
    s.D = head_dim;
    s.bs = block_size;
    s.flags = flags;
    s.G = G;
    s.GD = (G == 1 || G == 2 || G == 4 || G == 8) ? G : 0;
    s.P = P;
    s.adapt = partition_tokens == 0 ? 1 : 0;
    s.fp8 = fp8;
    s.decode_fma = !fp8 && s.GD > 0 && (flags & PKV_ATTN_DECODE_CUDA_CORES);
    // tcgen05 tiles: bf16 head_dim 128, boxes of >= 16 rows, partitions made of
    // whole 128-token stages (every automatic length is one), decode rows on
    // tensor cores, and a batch that may hold a multi-query row of more than
    // kTcMinCols (query, q head) pairs; otherwise the variant without tile
    // code runs
    s.tc = !fp8 && head_dim == 128 && block_size >= 16 && P % kTcT == 0 && !s.decode_fma &&
           !(flags & PKV_ATTN_NO_TCGEN05) && (long long)max_q_len * G > kTcMinCols && kTcRows % G == 0;
    s.key = shape_key(s);
    return PKV_OK;
}

int check_workspace(const Shape& s, const void* workspace, size_t workspace_bytes) {
    if (!workspace || workspace_bytes < s.w.total) return PKV_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return PKV_ERR_ALIGN;
    return PKV_OK;
}

// The planning kernel over the lengths (one CTA).
int launch_plan(const Shape& s, const int32_t* seq_lens, const int32_t* q_lens, void* workspace, int32_t* status,
                cudaStream_t st) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* aux = reinterpret_cast<int*>(ws + s.w.seqaux);
    PlanParams pp{};
    pp.seq_lens = seq_lens;
    pp.q_lens = q_lens;
    pp.items = reinterpret_cast<int4*>(ws + s.w.items);
    pp.seqs = reinterpret_cast<int4*>(ws + s.w.seqs);
    pp.hdr = reinterpret_cast<int*>(ws + s.w.hdr);
    pp.seq_q0 = aux;
    pp.seq_flag = aux + s.num_seqs;
    pp.seq_mq = aux + 2 * s.num_seqs;
    pp.seq_p = aux + 3 * s.num_seqs;
    pp.row_np = reinterpret_cast<int*>(ws + s.w.rownp);
    pp.status = status;
    pp.num_seqs = s.num_seqs;
    pp.total_q = s.total_q;
    pp.n_q = s.n_q;
    pp.n_kv = s.n_kv;
    pp.G = s.G;
    pp.D = s.D;
    pp.P = s.P;
    pp.max_blocks = s.max_blocks;
    pp.bs = s.bs;
    pp.max_seq_len = s.max_seq_len;
    pp.max_q_len = s.max_q_len;
    pp.decode_ok = s.decode_fma ? 1 : 0;
    pp.adapt_P = s.adapt;
    pp.fp8 = s.fp8 ? 1 : 0;
    pp.tc = s.tc ? 1 : 0;
    pp.sms = host::sm_count();
    pp.plan_key = s.key;
    return host::launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, pp) == cudaSuccess ? PKV_OK
                                                                                                  : PKV_ERR_CUDA;
}

// The attention kernel and the combine kernel over a planned workspace.  fq
// (FP8 pools): bit 0 = e5m2 codes, bit 1 = per-block scales.
int launch_run(const Shape& s, void* out, const void* q, const void* k_cache, const void* v_cache,
               const float* k_scale, const float* v_scale, int fq, const int32_t* block_tables, int num_blocks,
               float scale, void* workspace, int32_t* status, cudaStream_t st) {
    // 5-D views of each pool, one per box height in kv heads (a row is D values
    // of 2 bytes, or of 1 byte in e4m3).  Rows of more than 128 bytes are
    // viewed as [num_blocks][n_kv][row / 128 B][bs][128 B] (the 128-byte box
    // outside the row, a non-monotonic stride), so a box lands in shared memory
    // as [head][box][row]: consecutive tokens of one box in consecutive
    // 128-byte lines, which the 128-byte swizzle maps to distinct banks.
    const int head_dim = s.D, block_size = s.bs, num_kv_heads = s.n_kv;
    const bool fp8 = s.fp8;
    TMaps tm;
    {
        const uint64_t row = (uint64_t)head_dim * (fp8 ? 1 : 2);
        const uint64_t inner = fp8 ? 128 : 64;  // elements per 128-byte box
        const uint64_t nb = row / 128;
        const uint32_t box_rows = block_size < kTileT ? (uint32_t)block_size : (uint32_t)kTileT;
        const uint64_t blk = (uint64_t)block_size * row, head = (uint64_t)num_kv_heads * blk;
        const bool split = nb > 1;
        const uint64_t dims[5] = {inner, split ? (uint64_t)block_size : nb, split ? nb : (uint64_t)block_size,
                                  (uint64_t)num_kv_heads, (uint64_t)num_blocks};
        const uint64_t strides[4] = {split ? row : 128, split ? 128 : row, blk, head};
        for (int i = 0; i < 4; ++i) {
            uint32_t hb = 1u << i;
            if (hb > (uint32_t)num_kv_heads) hb = (uint32_t)num_kv_heads;
            const uint32_t box[5] = {(uint32_t)inner, split ? box_rows : (uint32_t)nb, split ? (uint32_t)nb : box_rows,
                                     hb, 1};
            if (host::encode_tiled(&tm.k[i], k_cache, 5, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, fp8) ||
                host::encode_tiled(&tm.v[i], v_cache, 5, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B, fp8))
                return PKV_ERR_CUDA;
        }
    }
    bool tc_pair = false;
    if (s.tc) {
        const uint64_t row = 256;
        const uint64_t blk = (uint64_t)block_size * row, head = (uint64_t)num_kv_heads * blk;
        // K (and V unless paired): [num_blocks][n_kv][bs][2 slabs][64], one slab
        // of min(bs, 128) rows per box
        {
            const uint64_t dims[5] = {64, 2, (uint64_t)block_size, (uint64_t)num_kv_heads, (uint64_t)num_blocks};
            const uint64_t strides[4] = {128, row, blk, head};
            const uint32_t box[5] = {64, 1, (uint32_t)(block_size < kTcT ? block_size : kTcT), 1, 1};
            if (host::encode_tiled(&tm.k_tc, k_cache, 5, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
                host::encode_tiled(&tm.v_tc, v_cache, 5, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
                return PKV_ERR_CUDA;
        }
        // V with block_size 16: the view [num_blocks][n_kv][2 slabs][bs][64]
        // (the slab outside the row), one box = both slabs of a block
        if (block_size == 16) {
            const uint64_t dims[5] = {64, 16, 2, (uint64_t)num_kv_heads, (uint64_t)num_blocks};
            const uint64_t strides[4] = {row, 128, blk, head};
            const uint32_t box[5] = {64, 16, 2, 1, 1};
            CUtensorMap v2;
            if (host::encode_tiled(&v2, v_cache, 5, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) == 0) {
                tm.v_tc = v2;
                tc_pair = true;
            }
        }
    } else {
        memset(&tm.k_tc, 0, sizeof(tm.k_tc));
        memset(&tm.v_tc, 0, sizeof(tm.v_tc));
    }

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    AttnParams ap{};
    ap.out = static_cast<__nv_bfloat16*>(out);
    ap.q = static_cast<const __nv_bfloat16*>(q);
    ap.block_tables = block_tables;
    ap.items = reinterpret_cast<const int4*>(ws + s.w.items);
    ap.seqs = reinterpret_cast<const int4*>(ws + s.w.seqs);
    ap.seq_p = reinterpret_cast<const int*>(ws + s.w.seqaux) + 3 * s.num_seqs;
    ap.hdr = reinterpret_cast<int*>(ws + s.w.hdr);
    ap.part_o = reinterpret_cast<float*>(ws + s.w.o);
    ap.part_ml = reinterpret_cast<float2*>(ws + s.w.ml);
    ap.status = status;
    ap.max_blocks = s.max_blocks;
    ap.n_q = s.n_q;
    ap.n_kv = s.n_kv;
    ap.G = s.G;
    ap.bs = block_size;
    ap.num_blocks = num_blocks;
    ap.np_max = s.w.np_max;
    ap.row_bytes = head_dim * 2;
    ap.scale_log2 = scale * 1.4426950408889634f;
    ap.k_scale = k_scale;
    ap.v_scale = v_scale;
    ap.scale_pb = (fq & 2) ? 1 : 0;
    {
        // FP8 items take gcd_pow2(n_kv, 8) kv heads a stage: their scale rows
        // are that many floats at (block * n_kv + group * hps) floats
        const int hps = gcd_pow2(s.n_kv, kMaxHPS);
        ap.scale_bulk = ap.scale_pb && (hps * 4) % 16 == 0 && (s.n_kv * 4) % 16 == 0 &&
                                host::aligned16(k_scale) && host::aligned16(v_scale)
                            ? 1
                            : 0;
    }
    ap.tc = s.tc ? 1 : 0;
    ap.tc_pair = tc_pair ? 1 : 0;
    ap.plan_key = s.key;
    // transposed items wider than one n-tile (8 columns) are possible when q_len * g > 8
    const bool wide = (long long)s.max_q_len * s.G > 8;
    const int rc = fp8 ? dispatch_attention_fp8_d128(fq, tm, ap, s.w.max_items, st)
                   : head_dim == 128
                       ? dispatch_attention_d128(s.decode_fma ? s.GD : 0, s.tc, wide, tm, ap, s.w.max_items, st)
                       : dispatch_attention_d64(s.decode_fma ? s.GD : 0, wide, tm, ap, s.w.max_items, st);
    if (rc != PKV_OK) return rc;
    // The combine runs even when no row can span partitions: it writes the NaN
    // rows of invalid sequences, resets the item queue for the next call over
    // the same plan, and triggers the next kernel of the stream only after the
    // attention grid has finished.
    CombineParams cp{};
    cp.out = ap.out;
    cp.part_o = ap.part_o;
    cp.part_ml = ap.part_ml;
    cp.row_np = reinterpret_cast<const int*>(ws + s.w.rownp);
    cp.hdr = ap.hdr;
    cp.status = status;
    cp.total_q = s.total_q;
    cp.n_q = s.n_q;
    cp.np_max = s.w.np_max;
    cp.plan_key = s.key;
    return head_dim == 128 ? combine_d128(cp, st) : combine_d64(cp, st);
}

int run_pointers_ok(const void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables) {
    if (!out || !q || !k_cache || !v_cache || !block_tables) return PKV_ERR_NULL;
    if (!host::aligned16(out) || !host::aligned16(q) || !host::aligned16(k_cache) || !host::aligned16(v_cache))
        return PKV_ERR_ALIGN;
    return PKV_OK;
}

// FP8 format and scale granularity -> the kernel variant's fq bits, or -1.
int fp8_mode(int kv_format, int scale_mode) {
    if (kv_format != PKV_FP8_E4M3 && kv_format != PKV_FP8_E5M2) return -1;
    if (scale_mode != PKV_FP8_SCALE_PER_HEAD && scale_mode != PKV_FP8_SCALE_PER_BLOCK) return -1;
    return (kv_format == PKV_FP8_E5M2 ? 1 : 0) | (scale_mode == PKV_FP8_SCALE_PER_BLOCK ? 2 : 0);
}

// Plan + run in one call (bf16 pools with k_scale == nullptr, or FP8 pools
// with dequantisation scales; fq as in launch_run).
int attention_call(void* out, const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                   const float* v_scale, bool fp8, int fq, const int32_t* block_tables, int max_blocks,
                   const int32_t* seq_lens, const int32_t* q_lens, int num_seqs, int total_q, int max_q_len,
                   int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                   float scale, int partition_tokens, int flags, void* workspace, size_t workspace_bytes,
                   int32_t* status, void* stream) {
    Shape s;
    int rc = check_shape(s, fp8, num_seqs, total_q, max_q_len, max_seq_len, max_blocks, num_q_heads, num_kv_heads,
                         head_dim, block_size, num_blocks, partition_tokens, flags);
    if (rc || s.empty) return rc;
    if (fp8 && (!k_scale || !v_scale)) return PKV_ERR_NULL;
    if ((rc = run_pointers_ok(out, q, k_cache, v_cache, block_tables))) return rc;
    if (!seq_lens || !q_lens) return PKV_ERR_NULL;
    if ((rc = check_workspace(s, workspace, workspace_bytes))) return rc;
    if ((rc = host::check_device())) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((rc = launch_plan(s, seq_lens, q_lens, workspace, status, st))) return rc;
    return launch_run(s, out, q, k_cache, v_cache, k_scale, v_scale, fq, block_tables, num_blocks, scale, workspace,
                      status, st);
}

}  // namespace

extern "C" int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                                          const int32_t* q_lens, int num_seqs, int total_q, int max_q_len,
                                          int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                                          int block_size, int num_blocks, float scale, int partition_tokens,
                                          int flags, void* workspace, size_t workspace_bytes, int32_t* status,
                                          void* stream) {
    return attention_call(out, q, k_cache, v_cache, nullptr, nullptr, false, 0, block_tables, max_blocks, seq_lens,
                          q_lens, num_seqs, total_q, max_q_len, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                          block_size, num_blocks, scale, partition_tokens, flags, workspace, workspace_bytes, status,
                          stream);
}

extern "C" int pkv_paged_attention_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                              const float* k_scale, const float* v_scale,
                                              const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                                              const int32_t* q_lens, int num_seqs, int total_q, int max_q_len,
                                              int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                                              int block_size, int num_blocks, float scale, int partition_tokens,
                                              void* workspace, size_t workspace_bytes, int32_t* status,
                                              void* stream) {
    return attention_call(out, q, k_cache, v_cache, k_scale, v_scale, true, 0, block_tables, max_blocks, seq_lens,
                          q_lens, num_seqs, total_q, max_q_len, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                          block_size, num_blocks, scale, partition_tokens, 0, workspace, workspace_bytes, status,
                          stream);
}

extern "C" int pkv_paged_attention_decode_fp8_ex(void* out, const void* q, const void* k_cache, const void* v_cache,
                                                 const float* k_scale, const float* v_scale, int kv_format,
                                                 int scale_mode, const int32_t* block_tables, int max_blocks,
                                                 const int32_t* seq_lens, const int32_t* q_lens, int num_seqs,
                                                 int total_q, int max_q_len, int max_seq_len, int num_q_heads,
                                                 int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                                 float scale, int partition_tokens, void* workspace,
                                                 size_t workspace_bytes, int32_t* status, void* stream) {
    const int fq = fp8_mode(kv_format, scale_mode);
    if (fq < 0) return PKV_ERR_UNSUPPORTED;
    return attention_call(out, q, k_cache, v_cache, k_scale, v_scale, true, fq, block_tables, max_blocks, seq_lens,
                          q_lens, num_seqs, total_q, max_q_len, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                          block_size, num_blocks, scale, partition_tokens, 0, workspace, workspace_bytes, status,
                          stream);
}

extern "C" int pkv_attention_plan(const int32_t* seq_lens, const int32_t* q_lens, int num_seqs, int total_q,
                                  int max_q_len, int max_seq_len, int max_blocks, int num_q_heads, int num_kv_heads,
                                  int head_dim, int block_size, int partition_tokens, int flags, void* workspace,
                                  size_t workspace_bytes, int32_t* status, void* stream) {
    const bool fp8 = (flags & PKV_ATTN_PLAN_FP8) != 0;
    flags &= ~PKV_ATTN_PLAN_FP8;
    if (fp8 && flags) return PKV_ERR_SIZE;  // the e4m3 attention takes no other flag
    Shape s;
    // the pool size does not enter the plan: any positive count passes the check
    int rc = check_shape(s, fp8, num_seqs, total_q, max_q_len, max_seq_len, max_blocks, num_q_heads, num_kv_heads,
                         head_dim, block_size, 1, partition_tokens, flags);
    if (rc || s.empty) return rc;
    if (!seq_lens || !q_lens) return PKV_ERR_NULL;
    if ((rc = check_workspace(s, workspace, workspace_bytes))) return rc;
    if ((rc = host::check_device())) return rc;
    return launch_plan(s, seq_lens, q_lens, workspace, status, static_cast<cudaStream_t>(stream));
}

extern "C" int pkv_paged_attention_run(void* out, const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_tables, int max_blocks, int num_seqs, int total_q,
                                       int max_q_len, int max_seq_len, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, int num_blocks, float scale,
                                       int partition_tokens, int flags, void* workspace, size_t workspace_bytes,
                                       int32_t* status, void* stream) {
    Shape s;
    int rc = check_shape(s, false, num_seqs, total_q, max_q_len, max_seq_len, max_blocks, num_q_heads, num_kv_heads,
                         head_dim, block_size, num_blocks, partition_tokens, flags);
    if (rc || s.empty) return rc;
    if ((rc = run_pointers_ok(out, q, k_cache, v_cache, block_tables))) return rc;
    if ((rc = check_workspace(s, workspace, workspace_bytes))) return rc;
    if ((rc = host::check_device())) return rc;
    return launch_run(s, out, q, k_cache, v_cache, nullptr, nullptr, 0, block_tables, num_blocks, scale, workspace,
                      status, static_cast<cudaStream_t>(stream));
}

extern "C" int pkv_paged_attention_run_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                           const float* k_scale, const float* v_scale, int kv_format, int scale_mode,
                                           const int32_t* block_tables, int max_blocks, int num_seqs, int total_q,
                                           int max_q_len, int max_seq_len, int num_q_heads, int num_kv_heads,
                                           int head_dim, int block_size, int num_blocks, float scale,
                                           int partition_tokens, void* workspace, size_t workspace_bytes,
                                           int32_t* status, void* stream) {
    const int fq = fp8_mode(kv_format, scale_mode);
    if (fq < 0) return PKV_ERR_UNSUPPORTED;
    Shape s;
    int rc = check_shape(s, true, num_seqs, total_q, max_q_len, max_seq_len, max_blocks, num_q_heads, num_kv_heads,
                         head_dim, block_size, num_blocks, partition_tokens, 0);
    if (rc || s.empty) return rc;
    if (!k_scale || !v_scale) return PKV_ERR_NULL;
    if ((rc = run_pointers_ok(out, q, k_cache, v_cache, block_tables))) return rc;
    if ((rc = check_workspace(s, workspace, workspace_bytes))) return rc;
    if ((rc = host::check_device())) return rc;
    return launch_run(s, out, q, k_cache, v_cache, k_scale, v_scale, fq, block_tables, num_blocks, scale, workspace,
                      status, static_cast<cudaStream_t>(stream));
}
