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
    int* seq_full;   // exclusive prefix of full decode-partition item counts
    int* row_np;     // [total_q] partitions of each query row
    __nv_bfloat16* out;
    int32_t* status;
    int num_seqs, total_q, n_q, n_kv, G, D, P, max_blocks, bs, max_seq_len, max_q_len, decode_ok;
    int fp8;         // e4m3 pool: every row on the transposed tensor-core item
    int tc;          // tcgen05 tiles allowed (head_dim 128, bf16, block_size >= 16, P % 128 == 0)
    int adapt_P;     // 1: P is a floor; the planning kernel may raise it
    int sms;         // SM count (persistent CTAs of the attention kernel)
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
// tc: a sequence with at least 128 (query, q head) rows per kv head runs as
// tcgen05 tiles of 128 rows (128 / G queries), one kv head each.
__device__ __forceinline__ SeqShape seq_shape(int ql, int G, int n_kv, int decode_fma, int fp8, int tc) {
    SeqShape s;
    if (tc && ql * G >= kTcRows && kTcRows % G == 0) {
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
    if (ql == 1 && G <= 8) {
        s.kind = decode_fma ? KIND_DECF : KIND_DEC;
        s.hps = gcd_pow2(n_kv, kMaxHPS);
        s.wph = 1;
        s.qt = 1;
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
constexpr int kAutoPMax = 8192;       // automatic partition length: upper bound
// automatic partition length: target partitions per SM (decode-heavy and
// multi-query-heavy batches)
constexpr int kAutoItemsPerSM = 2, kAutoItemsPerSMMQ = 3;

// Work list for one call: multi-query items first (the compute-heavy tiles
// start early), then every full decode partition, then the decode partition
// tails ordered longest first (counting sort over kTailBuckets length
// classes), so the dynamic queue ends on the shortest items.
//   pass A  one thread per sequence: validity, query rows, item counts and
//           their prefix sums, tail-length histogram;
//   pass B  items and per-row partition counts written over the item (row)
//           index space, one thread per item (row), which finds its sequence
//           by binary search in the prefix sums -- consecutive threads write
//           consecutive 16-byte items, so the stores coalesce.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ PlanParams pp) {
    __shared__ int tmp[32 * 2];
    __shared__ int hist[kTailBuckets];
    __shared__ int s_q0[kPlanSmemSeqs], s_mq[kPlanSmemSeqs], s_full[kPlanSmemSeqs], s_flag[kPlanSmemSeqs];
    __shared__ int4 s_seq[kPlanSmemSeqs];
    const int tid = threadIdx.x;
    const int n = pp.num_seqs;
    const bool small = n <= kPlanSmemSeqs;
    int* a_q0 = small ? s_q0 : pp.seq_q0;
    int* a_mq = small ? s_mq : pp.seq_mq;
    int* a_full = small ? s_full : pp.seq_full;
    int* a_flag = small ? s_flag : pp.seq_flag;
    const int4* a_seq = small ? s_seq : pp.seqs;  // per-sequence records of pass A (global copy always written)
    // this thread's first sequence, read once for the partition choice and pass A
    const int L0 = tid < n ? pp.seq_lens[tid] : 0, ql0 = tid < n ? pp.q_lens[tid] : 0;
    if (tid < kTailBuckets) hist[tid] = 0;
    // Programmatic launch: the previous kernel of the stream may still run
    // while passes A and B1-B3 do.  They read only seq_lens and q_lens, which
    // no kernel of this library writes, and write only work-list state the
    // previous step's attention kernel read -- and that kernel has finished:
    // this kernel starts no earlier than its predecessor's own wait, which
    // completes everything before it.  The per-row counts and NaN output rows
    // (read and written by a previous combine) wait for the predecessor, and
    // so does this kernel's completion, which the attention kernel waits on.
    pdl_launch();
    int P = pp.P;
    if (pp.adapt_P) {
        // automatic partition length: the floor P, raised along the ladder
        // P, 3P/2, 2P, 3P, 4P, ... (up to kAutoPMax) while the batch would give
        // more than kAutoItemsPerSM partitions per SM -- fewer, longer items
        // cost fewer partial results and item switches, and the finer steps
        // keep the last wave of the dynamic queue from being nearly empty (on
        // the speculative workload P = 768 beat both 512 and 1024 by 8-12 %)
        long long tok = 0, tok_mq = 0;
        for (int b = tid; b < n; b += kPlanThreads) {
            const int L = b == tid ? L0 : pp.seq_lens[b], ql = b == tid ? ql0 : pp.q_lens[b];
            if (L <= 0 || ql <= 0 || ql > L || L > pp.max_seq_len || ql > pp.max_q_len) continue;
            const SeqShape sh = seq_shape(ql, pp.G, pp.n_kv, pp.decode_ok, pp.fp8, pp.tc);
            const bool multi = multi_query_kind(sh.kind) || ql > 1;
            const long long t = (long long)L * (pp.n_kv / sh.hps) * (multi ? ceil_div(ql, sh.qt) : 1);
            tok += t;
            if (multi) tok_mq += t;
        }
        // block sums in units of 16 tokens (fit an int for any accepted batch)
        const int cap = (1 << 30) / kPlanThreads;
        int v2[2] = {(int)min(tok >> 4, (long long)cap), (int)min(tok_mq >> 4, (long long)cap)}, t2[2];
        block_scan_k<2>(v2, t2, tmp);
        const int tot16 = t2[0], mq16 = t2[1];
        const long long T = (long long)tot16 << 4;
        // multi-query items cost more compute per token: a batch made of them
        // (speculative verification) balances better with more items
        const int per_sm = 4 * (long long)mq16 > 3 * (long long)tot16 ? kAutoItemsPerSMMQ : kAutoItemsPerSM;
        while (P < kAutoPMax && T > (long long)P * per_sm * pp.sms) P = (P & (P - 1)) == 0 ? P + P / 2 : P + P / 3;
    }
    if (tid == 0) pp.hdr[2] = P;
    __syncthreads();
    int bits = 0, any_tc = 0;
    // pass A
    long long carry = 0;
    int c_mq = 0, c_full = 0;
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
        int nmq = 0, nfull = 0, q0 = 0;
        if (b < n) {
            const long long q0l = carry + ex;
            if (q0l + qlc > pp.total_q) flag |= PKV_STATUS_BAD_QLEN;  // rows would overflow q/out
            q0 = (int)(q0l < pp.total_q ? q0l : pp.total_q);
            bits |= flag;
            const SeqShape sh = seq_shape(ql, pp.G, pp.n_kv, pp.decode_ok, pp.fp8, pp.tc);
            const int ngroups = pp.n_kv / sh.hps;
            if (flag == 0) {
                if (sh.kind == KIND_TC) any_tc = 1;
                if (!multi_query_kind(sh.kind) && ql == 1) {
                    const int np = ceil_div(L, P);
                    nfull = (np - 1) * ngroups;
                    const int tl = L - (np - 1) * P;  // in [1, P]
                    atomicAdd(&hist[(int)(((long long)(P - tl) * kTailBuckets) / P)], ngroups);
                } else if (ql > 0) {
                    nmq = mq_parts_of(L, ql, sh.qt, P) * ngroups;
                }
            }
            const int4 rec = make_int4(L, ql, q0, sh.kind | (sh.hps << 4) | (sh.wph << 8) | (sh.qt << 12));
            pp.seqs[b] = rec;
            if (small) s_seq[b] = rec;
            a_flag[b] = flag;
        }
        carry += tot;
        int v2[2] = {nmq, nfull}, t2[2];
        block_scan_k<2>(v2, t2, tmp);
        if (b < n) {
            a_q0[b] = q0;
            a_mq[b] = c_mq + v2[0];
            a_full[b] = c_full + v2[1];
        }
        c_mq += t2[0];
        c_full += t2[1];
    }
    // tail buckets -> first slot of each bucket (exclusive scan)
    any_tc = __syncthreads_or(any_tc);
    int c_tail;
    {
        const int v = tid < kTailBuckets ? hist[tid] : 0;
        const int ex = block_exclusive_scan_1024(v, tmp, &c_tail);
        if (tid < kTailBuckets) hist[tid] = c_mq + c_full + ex;
    }
    if (tid == 0) {
        pp.hdr[0] = c_mq + c_full + c_tail;
        pp.hdr[1] = 0;
        pp.hdr[3] = any_tc;  // the attention kernel allocates tensor memory only then
    }
    __syncthreads();
    // pass B1: one thread per sequence -- decode tails and invalid sequences
    for (int b = tid; b < n; b += kPlanThreads) {
        const int4 sq = a_seq[b];
        const int L = sq.x, ql = sq.y;
        if (a_flag[b]) continue;  // its rows are written NaN after the wait below
        if (ql != 1 || multi_query_kind(sq.w & 15)) continue;  // multi-query tiles are counted in pass B2
        const int ngroups = pp.n_kv / ((sq.w >> 4) & 15);
        const int np = ceil_div(L, P);
        const int tl = L - (np - 1) * P;
        const int t0 = atomicAdd(&hist[(int)(((long long)(P - tl) * kTailBuckets) / P)], ngroups);
        for (int hg = 0; hg < ngroups; ++hg) pp.items[t0 + hg] = make_int4(b, np - 1, 0, hg);
    }
    // pass B2: multi-query items
    for (int it = tid; it < c_mq; it += kPlanThreads) {
        const int b = last_le(a_mq, n, it);
        int li = it - a_mq[b];
        const int4 sq = a_seq[b];
        const int L = sq.x, ql = sq.y, QT = (sq.w >> 12) & 4095;
        const int ngroups = pp.n_kv / ((sq.w >> 4) & 15);
        for (int qt = 0; qt * QT < ql; ++qt) {
            const int nq = min(QT, ql - qt * QT);
            const int cnt = ceil_div(L - ql + qt * QT + nq, P) * ngroups;
            if (li < cnt) {
                const int part = li / ngroups;
                pp.items[it] = make_int4(b, part, qt, li - part * ngroups);
                break;
            }
            li -= cnt;
        }
    }
    // pass B3: full decode partitions
    {
        const int ngroups = pp.n_kv / gcd_pow2(pp.n_kv, kMaxHPS);
        for (int it = tid; it < c_full; it += kPlanThreads) {
            const int b = last_le(a_full, n, it);
            const int li = it - a_full[b];
            const int part = li / ngroups;
            pp.items[c_mq + it] = make_int4(b, part, 0, li - part * ngroups);
        }
    }
    pdl_wait();
    // rows of an invalid sequence are NaN (inside the q/out extent)
    for (int b = tid; b < n; b += kPlanThreads) {
        if (!a_flag[b]) continue;
        const int4 sq = a_seq[b];
        const int ql = sq.y, q0 = sq.z;
        const int qlc = ql > 0 ? min(ql, pp.total_q) : 0;
        const int rows = min(qlc, pp.total_q - q0);
        const long long n16 = (long long)rows * pp.n_q * pp.D / 8;
        uint4* o = reinterpret_cast<uint4*>(pp.out + (long long)q0 * pp.n_q * pp.D);
        for (long long e = 0; e < n16; ++e) o[e] = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
    }
    // pass B4: partitions per query row (0 for rows of invalid sequences and
    // rows past the last sequence's queries: nothing to merge)
    for (int r = tid; r < pp.total_q; r += kPlanThreads) {
        int np = 0;
        if (r < carry) {
            const int b = last_le(a_q0, n, r);
            const int4 sq = a_seq[b];
            const int L = sq.x, ql = sq.y, q0 = sq.z;
            if (a_flag[b] == 0 && r - q0 < ql) {
                // query tile of row r; a decode row is a tile of one query
                const int QT = (sq.w >> 12) & 4095;
                const int qt = (r - q0) / QT;
                const int nq = min(QT, ql - qt * QT);
                np = ceil_div(L - ql + qt * QT + nq, P);
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

// Both entry points: bf16 pools (k_scale == nullptr) or e4m3 pools with
// per-kv-head dequantisation scales.
int run_attention(void* out, const void* q, const void* k_cache, const void* v_cache, const float* k_scale,
                  const float* v_scale, bool fp8, const int32_t* block_tables, int max_blocks,
                  const int32_t* seq_lens, const int32_t* q_lens, int num_seqs, int total_q, int max_q_len,
                  int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                  float scale, int partition_tokens, int flags, void* workspace, size_t workspace_bytes,
                  int32_t* status, void* stream) {
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
    if (fp8 && (!k_scale || !v_scale)) return PKV_ERR_NULL;
    if (num_seqs == 0 || total_q == 0) return PKV_OK;
    if (num_seqs > (1 << 24) || total_q > (1 << 20)) return PKV_ERR_SIZE;
    int P = partition_tokens;
    if (P == 0) P = pkv_attention_auto_partition(num_seqs, total_q, num_kv_heads, max_seq_len);
    if (P < kTileT || P % kTileT) return PKV_ERR_SIZE;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !q_lens) return PKV_ERR_NULL;
    if (!host::aligned16(out) || !host::aligned16(q) || !host::aligned16(k_cache) || !host::aligned16(v_cache))
        return PKV_ERR_ALIGN;
    const WsLayout w = ws_layout(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, max_seq_len, P);
    if (w.np_max > kMaxParts) return PKV_ERR_SIZE;
    if (!workspace || workspace_bytes < w.total) return PKV_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return PKV_ERR_ALIGN;
    if (w.max_items > 0x7fffffffLL) return PKV_ERR_SIZE;
    const int rc = host::check_device();
    if (rc) return rc;

    // 5-D views of each pool, one per box height in kv heads (a row is D values
    // of 2 bytes, or of 1 byte in e4m3).  Rows of more than 128 bytes are
    // viewed as [num_blocks][n_kv][row / 128 B][bs][128 B] (the 128-byte box
    // outside the row, a non-monotonic stride), so a box lands in shared memory
    // as [head][box][row]: consecutive tokens of one box in consecutive
    // 128-byte lines, which the 128-byte swizzle maps to distinct banks.
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

    // tcgen05 tiles: bf16 head_dim 128, boxes of >= 16 rows, partitions made of
    // whole 128-token stages, decode rows on tensor cores, and a batch that may
    // hold a 128-row tile (max_q_len * g >= 128); otherwise the variant
    // without tile code runs
    const int GD = (G == 1 || G == 2 || G == 4 || G == 8) ? G : 0;
    const bool decode_fma = !fp8 && GD > 0 && (flags & PKV_ATTN_DECODE_CUDA_CORES);
    const bool tc = !fp8 && head_dim == 128 && block_size >= 16 && P % kTcT == 0 && !decode_fma &&
                    !(flags & PKV_ATTN_NO_TCGEN05) && (long long)max_q_len * G >= kTcRows;
    bool tc_pair = false;
    if (tc) {
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
    int* aux = reinterpret_cast<int*>(ws + w.seqaux);

    PlanParams pp{};
    pp.seq_lens = seq_lens;
    pp.q_lens = q_lens;
    pp.items = reinterpret_cast<int4*>(ws + w.items);
    pp.seqs = reinterpret_cast<int4*>(ws + w.seqs);
    pp.hdr = reinterpret_cast<int*>(ws + w.hdr);
    pp.seq_q0 = aux;
    pp.seq_flag = aux + num_seqs;
    pp.seq_mq = aux + 2 * num_seqs;
    pp.seq_full = aux + 3 * num_seqs;
    pp.row_np = reinterpret_cast<int*>(ws + w.rownp);
    pp.out = static_cast<__nv_bfloat16*>(out);
    pp.status = status;
    pp.num_seqs = num_seqs;
    pp.total_q = total_q;
    pp.n_q = num_q_heads;
    pp.n_kv = num_kv_heads;
    pp.G = G;
    pp.D = head_dim;
    pp.P = P;
    pp.max_blocks = max_blocks;
    pp.bs = block_size;
    pp.max_seq_len = max_seq_len;
    pp.max_q_len = max_q_len;
    pp.decode_ok = decode_fma ? 1 : 0;
    pp.adapt_P = partition_tokens == 0 ? 1 : 0;
    pp.fp8 = fp8 ? 1 : 0;
    pp.tc = tc ? 1 : 0;
    pp.sms = host::sm_count();
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (host::launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, pp) != cudaSuccess) return PKV_ERR_CUDA;

    AttnParams ap{};
    ap.out = static_cast<__nv_bfloat16*>(out);
    ap.q = static_cast<const __nv_bfloat16*>(q);
    ap.block_tables = block_tables;
    ap.items = pp.items;
    ap.seqs = pp.seqs;
    ap.hdr = pp.hdr;
    ap.part_o = reinterpret_cast<float*>(ws + w.o);
    ap.part_ml = reinterpret_cast<float2*>(ws + w.ml);
    ap.status = status;
    ap.max_blocks = max_blocks;
    ap.n_q = num_q_heads;
    ap.n_kv = num_kv_heads;
    ap.G = G;
    ap.bs = block_size;
    ap.num_blocks = num_blocks;
    ap.np_max = w.np_max;
    ap.row_bytes = head_dim * 2;
    ap.scale_log2 = scale * 1.4426950408889634f;
    ap.k_scale = k_scale;
    ap.v_scale = v_scale;
    ap.tc = tc ? 1 : 0;
    ap.tc_pair = tc_pair ? 1 : 0;
    const int rc2 = fp8                ? dispatch_attention_fp8_d128(tm, ap, w.max_items, st)
                    : head_dim == 128 ? dispatch_attention_d128(decode_fma ? GD : 0, tc, tm, ap, w.max_items, st)
                                      : dispatch_attention_d64(decode_fma ? GD : 0, tm, ap, w.max_items, st);
    // The combine runs even when no row can span partitions (it then only
    // waits and exits): it triggers the next kernel of the stream only after
    // the attention grid has finished, which the next call's planning kernel
    // relies on before it rewrites the work list.
    if (rc2 != PKV_OK) return rc2;
    CombineParams cp{};
    cp.out = ap.out;
    cp.part_o = ap.part_o;
    cp.part_ml = ap.part_ml;
    cp.row_np = pp.row_np;
    cp.total_q = total_q;
    cp.n_q = num_q_heads;
    cp.np_max = w.np_max;
    return head_dim == 128 ? combine_d128(cp, st) : combine_d64(cp, st);
}

}  // namespace

extern "C" int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                                          const int32_t* q_lens, int num_seqs, int total_q, int max_q_len,
                                          int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                                          int block_size, int num_blocks, float scale, int partition_tokens,
                                          int flags, void* workspace, size_t workspace_bytes, int32_t* status,
                                          void* stream) {
    return run_attention(out, q, k_cache, v_cache, nullptr, nullptr, false, block_tables, max_blocks, seq_lens,
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
    return run_attention(out, q, k_cache, v_cache, k_scale, v_scale, true, block_tables, max_blocks, seq_lens,
                         q_lens, num_seqs, total_q, max_q_len, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                         block_size, num_blocks, scale, partition_tokens, 0, workspace, workspace_bytes, status,
                         stream);
}
