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
//   * A planning kernel turns (seq_lens, q_lens) into per-sequence records and
//     a list of 16-byte work items (sequence, partition, query tile, head
//     group): multi-query items first, then every decode-style item longest
//     first (a counting sort over length classes), so the dynamic queue ends
//     on short items.  It also records how many partitions each query row has.
//   * The attention kernel is persistent, one CTA per SM, three warpgroups:
//     eight consumer warps (224 registers each) and a side warpgroup (56
//     each, by setmaxnreg) holding the producer warp, the V warp and, in the
//     variant with tcgen05 tiles, the MMA and helper TMA warps.  A pipeline
//     stage is 16 tokens of K and V for a group of kv heads of one block --
//     for the 8B shape all 8 heads, 32 KB of K plus 32 KB of V -- fetched
//     with one 5-D TMA box per tensor (128-byte swizzle) into a 3-slot,
//     192 KB shared-memory ring, the producer copying K and the V warp V.  A
//     TMA-issuing warp sustains only a couple of copies per microsecond
//     whatever their size, so copies have to be tens of KB to keep HBM busy.
//   * Decode rows and short verifications run on tensor cores (mma.sync
//     m16n8k16 bf16 -> fp32), one warp per kv head, in the transposed form
//     S^T = K Q^T: the 16 tokens of a stage on M, the (query, q head) columns
//     of the kv head on N -- up to 24 (three n-tiles), so k = 5 drafts at
//     g = 4 stream exactly like decode; each column's causal limit is applied
//     to its scores.  A CUDA-core variant for q_len = 1 (8 lanes per token,
//     packed fp32x2 FMAs) is kept behind a flag.
//   * Wider multi-query rows (prefill chunks) run as tcgen05 tiles of 128
//     rows, or, with those off, on mma.sync row tiles (16 (query, head) rows
//     per warp, the warps of one kv head splitting its rows).
//   * Consumer warps run independently: each waits for its own stages and
//     releases them as it finishes, with no CTA-wide barrier per item.
//   * A partition's partial (O, m, l) goes to the workspace; a separate combine
//     kernel, launched as a programmatic dependent of the attention kernel,
//     merges the partials of each row in partition order (deterministic).
#pragma once

#include "pkv_common.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr int kTileT = 16;                  // tokens per pipeline stage
constexpr int kCWarps = 8;                  // consumer warps
constexpr int kCThreads = kCWarps * 32;
// A CTA is three warpgroups: the eight consumer warps, then the producer, the
// MMA warp and the helper TMA warp of the tcgen05 variant (idle in the other
// variant), and the V warp, which issues the V copies of 16-token stages
// beside the producer's K copies.  With 12 warps every SM
// sub-partition holds three, which caps the launch at 168 registers a thread;
// the side warpgroup then gives most of its registers to the consumers
// (setmaxnreg), so their items can hold up to 24 columns of Q^T and O^T.
constexpr int kThreads = 12 * 32;
constexpr int kLaunchRegs = 168;            // registers a thread at launch (65536 / 384, in steps of 8)
constexpr int kConsumerRegs = 224;
constexpr int kSideRegs = 56;
static_assert(kSideRegs * 128 + kConsumerRegs * 256 <= kLaunchRegs * kThreads, "register split exceeds the launch");
constexpr int kMaxHPS = 8;                  // kv heads per stage
constexpr int kDecCols = 24;                // (query, q head) columns of a transposed tensor-core tile
constexpr int kTcMinCols = kDecCols;        // multi-query rows of more columns run as tcgen05 tiles (when enabled)
constexpr int kRingSlots = 3;
constexpr int kSlots = 4;                   // item descriptors in flight
constexpr int kClaimAhead = 6;              // stages before an item's end at which the next is claimed
constexpr float kRescaleSlack = 8.0f;       // lazy-rescale threshold of the running max, base-2 units
constexpr int kMaxParts = 1024;             // partitions per sequence
constexpr int kPlanThreads = 1024;
constexpr int kTailBuckets = 256;           // tail-length classes of the longest-first ordering

// tcgen05 chunk tiles: 128 rows = (query, q head) pairs of one kv head, stages
// of 128 tokens, tensor-memory columns [S | P0 P1 | O_0 | O_1]: one fp32 S
// buffer, two bf16 P buffers (two values a column) by stage parity.
constexpr int kTcT = 128;                   // tokens per stage
constexpr int kTcRows = 128;                // tile rows (the MMA's M)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0, kTmemP = 128, kTmemO = 256;

// KIND_DEC: q_len = 1 rows on tensor cores; KIND_DECF: on CUDA cores; KIND_MQ:
// q_len > 1 on mma.sync; KIND_TC: query tiles of 128 rows on tcgen05.
enum { KIND_END = -1, KIND_DEC = 0, KIND_MQ = 1, KIND_DECF = 2, KIND_TC = 3 };

__host__ __device__ constexpr bool multi_query_kind(int kind) { return kind == KIND_MQ || kind == KIND_TC; }

struct Desc {
    int b, part, nparts, hg;        // sequence, partition, partitions of the group, head group
    int t_begin, t_end, t_vis, q_row0;
    int nq, kind, hps, wph;         // queries in the tile, kind, kv heads per stage, warps per kv head
};

// Tensor maps over a cache pool viewed as [num_blocks][n_kv][bs][D/64][64]
// (innermost last), one per box height in kv heads (1, 2, 4, 8).
struct TMaps {
    CUtensorMap k[4];
    CUtensorMap v[4];
    CUtensorMap k_tc, v_tc;  // tcgen05 stages: see produce_tc
};

struct AttnParams {
    __nv_bfloat16* out;
    const __nv_bfloat16* q;
    const int32_t* block_tables;
    const int4* items;   // {b, part, qt, hg}
    const int4* seqs;    // {seq_len, q_len, first query row, kind | hps << 4 | wph << 8 | qt_len << 12}
    const int* seq_p;    // partition length of each sequence
    int* hdr;            // [0] item count, [1] queue head, [2] partition length (target length when automatic)
    float* part_o;       // [(row * n_q + h) * np_max + part][D]
    float2* part_ml;     // [(row * n_q + h) * np_max + part] = (m in log2 units, l)
    int32_t* status;
    const float* k_scale;  // FP8 pools: dequantisation scales per kv head, or [num_blocks][n_kv] (null for bf16)
    const float* v_scale;
    int scale_pb;          // FP8 pools: 1 = a scale per (block, kv head) tile
    int scale_bulk;        // per-block scale rows are 16-byte aligned multiples of 16 bytes: fetched by bulk copies
    int max_blocks, n_q, n_kv, G, bs, num_blocks, np_max, row_bytes;
    int tc;              // tcgen05 tiles possible: tensor memory is allocated when the plan made some
    int tc_pair;         // tcgen05 stages of block_size 16: one V box holds both slabs of a block
    int plan_key;        // shape key the workspace's plan must carry (hdr[4]); else nothing runs
    float scale_log2;    // scale * log2(e): scores live in base-2 units
};

// Workspace header (ints): [0] item count, [1] queue head (reset to 0 by the
// planning kernel and again by each call's combine kernel, so one plan serves
// any number of calls), [2] partition length (explicit) or target item length
// (automatic: each sequence's own length is in the seq_p array), [3] tcgen05 tiles present,
// [4] key of the shape the plan was made for.
enum { HDR_ITEMS = 0, HDR_HEAD = 1, HDR_P = 2, HDR_TC = 3, HDR_KEY = 4 };

// Stage geometry of a pool: bf16 (2-byte values, 3 ring slots of 64 KB at the
// 8B shape) or e4m3 (1-byte values, 6 ring slots of 32 KB -- the same 192 KB
// of shared memory holds twice the stages, so twice the copies in flight).
template <int D, bool F8>
struct Geo {
    static constexpr int kElem = F8 ? 1 : 2;
    static constexpr int kRow = D * kElem;                  // bytes of one token of one head
    static constexpr int kNB = kRow / 128;                  // 128-byte boxes per row
    static constexpr int kSlots = F8 ? 6 : kRingSlots;      // ring slots
    static constexpr int kHalf = kTileT * kMaxHPS * kRow;   // K (or V) bytes of one stage
};

template <int D, bool F8 = false>
struct Smem {
    using G = Geo<D, F8>;
    static constexpr bool kTC = D == 128 && !F8;             // the pool shape with tcgen05 tiles
    uint8_t kv[G::kSlots][2][G::kHalf];                      // [slot][K,V][rows of 128 B], swizzled
    union {
        float pbuf[kCWarps][kTileT * 8];                     // decode on CUDA cores: p[token][head]
        uint8_t qbuf[kTC ? kTcRows * D * 2 : 16];            // tcgen05 tile: Q, K-major, 128-byte swizzle
    };
    // FP8 pools with per-block scales: the K and V scales of each block of a
    // stage for its kv heads, [slot][K,V][block of the stage][head of the stage]
    alignas(16) float scl[F8 ? G::kSlots : 1][2][F8 ? kTileT : 1][kMaxHPS];
    Desc desc[kSlots];
    int poison[kSlots];
    int abort;
    uint64_t full[G::kSlots], empty[G::kSlots], ifull[kSlots], iempty[kSlots];
    // tcgen05 tiles: S ready, PV done (per buffer), P written (per half),
    // half-row merge, tile entry, Q written, final drain, warps done with
    // tensor memory
    // P ready is double-buffered by stage parity: the softmax warps may finish
    // stages k and k + 1 before the MMA warp waits for stage k's phase (it
    // issues S_{k+1} first), and one barrier would then have moved on twice
    uint64_t sbar, sfree, obar[2], pready[2][2], xbar, ebar, qbar, tdone, dbar;
    uint32_t tmem;
    float red[kTC ? 2 : 1][2][kTcRows];                       // [m, l][half][row]
};
// the tcgen05 operands (ring slabs, Q) start on 1024-byte swizzle atoms
using SmemTc = Smem<128, false>;
static_assert(sizeof(SmemTc::kv) % 1024 == 0, "ring size");
static_assert(offsetof(SmemTc, qbuf) == sizeof(SmemTc::kv), "Q follows the ring");

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int log2i(int x) { return 31 - __clz(x); }

// Transpose of an 8x8 b16 matrix held one 32-bit pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Index of the 128-byte shared-memory row that holds (head h of the stage,
// token r of the tile, 128-byte box x of the token's row): the TMA boxes of one
// stage are [op][head][box][rows of the op], one op per block when
// block_size < 16.  Rows per op are a power of two, 1 << lb; hps_lb =
// hps << lb, h_lb = h << lb.  With the box outside the rows, the 8 consecutive
// tokens an ldmatrix reads for one box sit in 8 consecutive 128-byte rows, so
// the 128-byte swizzle spreads them over all banks (rows [token][box] would
// put tokens r and r + 4 on the same banks).
__device__ __forceinline__ int srow(int h_lb, int r, int x, int hps_lb, int lb, int nb) {
    return ((r >> lb) * hps_lb + h_lb) * nb + (x << lb) + (r & ((1 << lb) - 1));
}

__device__ __forceinline__ void tma_load_5d(void* smem_dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            int c4, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5, %6}], [%7];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(bar))
        : "memory");
}

// Work-item record -> descriptor (the same arithmetic the planning kernel used
// to count items).
__device__ __forceinline__ Desc make_desc(const int4 it, const int4 sq, int P) {
    Desc d;
    d.b = it.x;
    d.part = it.y;
    const int qt = it.z;
    d.hg = it.w;
    const int L = sq.x, ql = sq.y, q0 = sq.z;
    d.kind = sq.w & 15;
    d.hps = (sq.w >> 4) & 15;
    d.wph = (sq.w >> 8) & 15;
    const int QT = (sq.w >> 12) & 4095;
    // query tile qt holds queries [qt*QT, qt*QT + nq); its last query sees t_vis
    // positions (a decode row is a tile of one query: t_vis = L)
    d.nq = min(QT, ql - qt * QT);
    d.t_vis = L - ql + qt * QT + d.nq;
    d.q_row0 = q0 + qt * QT;
    d.nparts = ceil_div(d.t_vis, P);
    d.t_begin = d.part * P;
    d.t_end = min(d.t_begin + P, d.t_vis);
    return d;
}

// ---------------------------------------------------------------------------
// Ring slots of a tcgen05 tile.  A stage is 128 tokens of one kv head; K and V
// each take 32 KB of 128-byte rows (128-byte swizzle): the K-major B operand of
// S = Q K^T and the MN-major B operand of O += P V.  The slots are skewed: slot
// j holds K of stage j and V of stage j - 1 (n + 1 slots for n stages), so a
// slot is free once S_j and PV_{j-1} have run -- one stage earlier than with
// K_j and V_j together, which doubles how far ahead the ring can fetch.
// A TMA copy costs the issuing warp about the same time whatever its size, so
// the stage is fetched in as few boxes as the paged layout and the MMA
// operands allow.  K: one box per (slab, block), [slab][token] -- slab x at
// x * 16 KB, rows contiguous, 8-row groups 1 KB apart, so S is one N = 128
// MMA chain.  V: the same with block_size >= 32; with block_size 16 one 4 KB
// box per block holds both slabs of its 16 rows, [slab][row], block b of the
// stage at b * 4 KB (the MN-major operand of a 16-token k-step is one block:
// slabs 2 KB apart, its two 8-row groups 1 KB apart).  Two warps issue the
// copies of a slot in parallel, half each (12 copies apiece with block_size
// 16): the producer and the helper warp.
// Blocks that start past the item's last position are not fetched (the
// consumers zero those V rows).
// Returns false when the pipeline was aborted.
// ---------------------------------------------------------------------------
template <int D, bool F8>
__device__ __forceinline__ bool produce_tc(Smem<D, F8>& sm, const TMaps* tm, const AttnParams& p, const Desc& d,
                                           int si, int lane, uint32_t& g, int& next, bool helper) {
    if constexpr (!Smem<D, F8>::kTC) {
        return false;
    } else {
        constexpr int RS = Geo<D, F8>::kSlots;
        volatile int* abort = &sm.abort;
        const int rows = p.bs < kTcT ? p.bs : kTcT;  // rows per box
        const int nblk = kTcT / rows;                // blocks per stage (<= 8)
        const bool pair = p.tc_pair != 0;  // block_size 16: one V box = both slabs of a block
        // two warps split every slot: warp w (0 = producer, 1 = helper) copies
        // slab w of K for every block (lanes l < nblk: block l), then half of V:
        // paired boxes of blocks [w nblk / 2, (w + 1) nblk / 2), or slab w of
        // every block -- K first, since S_j needs it before PV_{j-1} needs V
        const int w = helper ? 1 : 0;
        int tv = 0, x = w, jb = lane;
        bool lane_ok = lane < nblk;
        if (lane >= nblk) {
            const int l2 = lane - nblk;
            tv = 1;
            x = pair ? 0 : w;
            jb = pair ? l2 + w * (nblk / 2) : l2;
            lane_ok = l2 < (pair ? nblk / 2 : nblk);
        }
        const bool pv = pair && tv;                  // this lane copies a paired V box
        const uint32_t slab_bytes = (uint32_t)rows * 128;
        const int tb = d.t_begin / kTcT, te = (d.t_end + kTcT - 1) / kTcT;
        const int n = te - tb;
        const int32_t* bt = p.block_tables + (long long)d.b * p.max_blocks;
        const int e_lim = (d.t_end + p.bs - 1) / p.bs;
        int tab_base = tb * kTcT / p.bs;
        int tab = tab_base + lane < e_lim ? __ldg(bt + tab_base + lane) : 0;
        int tab_next = tab_base + 32 + lane < e_lim ? __ldg(bt + tab_base + 32 + lane) : 0;
        const int j_claim = max(0, n + 1 - kClaimAhead);
        for (int j = 0; j <= n; ++j, ++g) {
            if (!helper && j == j_claim && lane == 0) next = atomicAdd(&p.hdr[HDR_HEAD], 1);
            // V (stage j - 1) trails K (stage j) by one stage: the table window
            // follows V's first entry; K's entries are at most 8 further
            const int tk = (tb + j) * kTcT, tvv = tk - kTcT;
            const int e_lo = (j > 0 ? tvv : tk) / p.bs;
            if (e_lo >= tab_base + 32) {
                tab = tab_next;
                tab_base += 32;
                const int en = tab_base + 32 + lane;
                tab_next = en < e_lim ? __ldg(bt + en) : 0;
            }
            const int t0 = tv ? tvv : tk;          // this lane's stage
            const bool has = tv ? j > 0 : j < n;   // slot j holds that stage
            const int nvb_k = j < n ? min(nblk, (d.t_end - tk + rows - 1) / rows) : 0;
            const int nvb_v = j > 0 ? min(nblk, (d.t_end - tvv + rows - 1) / rows) : 0;
            const int off = (has ? t0 / p.bs : e_lo) - tab_base + jb;  // in [0, 48)
            const int lo = __shfl_sync(kFull, tab, off & 31);
            const int hi = __shfl_sync(kFull, tab_next, off & 31);
            int my = off < 32 ? lo : hi;
            const bool in = lane_ok && has && jb < (tv ? nvb_v : nvb_k) && jb < nblk;
            const bool okb = !in || (my >= 0 && my < p.num_blocks);
            if (!okb) my = 0;
            const unsigned badmask = __ballot_sync(kFull, !okb);
            const int s = (int)(g % RS);
            bool got = true;
            if (lane == 0) {
                // every block of the stage has a producer lane (slab 0 of K; V
                // stage j - 1 reads the blocks K stage j - 1 was checked on): the
                // producer alone reports, and alone arms the slot's barrier with
                // both warps' bytes (the helper's copies may land first: the
                // phase cannot complete before this arrival)
                if (badmask && !helper) {
                    sm.poison[si] = 1;
                    report(p.status, PKV_STATUS_BAD_BLOCK);
                }
                got = mbar_wait(&sm.empty[s], ((g / RS) & 1) ^ 1, abort);
                if (got && !helper) mbar_arrive_expect_tx(&sm.full[s], 2u * (nvb_k + nvb_v) * slab_bytes);
            }
            if (!__shfl_sync(kFull, got, 0)) return false;  // never arm a barrier whose previous phase is open
            if (in) {
                const int row0 = p.bs > kTcT ? (t0 % p.bs) : 0;
                if (pv)  // view {64, bs, slab, n_kv, nb}: [slab][16 rows] of block my, 4 KB at 4 KB steps
                    tma_load_5d(&sm.kv[s][1][jb * 4096], &tm->v_tc, 0, 0, 0, d.hg, my, &sm.full[s]);
                else     // view {64, slab, bs, n_kv, nb}: one slab of `rows` rows
                    tma_load_5d(&sm.kv[s][tv][x * (kTcT * 128) + jb * slab_bytes], tv ? &tm->v_tc : &tm->k_tc, 0, x,
                                row0, d.hg, my, &sm.full[s]);
            }
            __syncwarp();
        }
        return true;
    }
}

// ---------------------------------------------------------------------------
// The 16-token stages of one item (not a tcgen05 tile): block-table entries,
// slot waits and TMA copies, one box per tensor and block holding every head
// of the group.  Two warps share each stage, each issuing the copies of one
// tensor: a warp sustains only a couple of copies per microsecond, and a
// stage of an FP8 pool is two 16 KB copies.
//   vwarp false (the producer): claims the next item a few stages ahead,
//     reports bad blocks, stores FP8 per-block scales, arms the stage's
//     barrier with both tensors' bytes and copies K;
//   vwarp true (the V warp): copies V once the slot is free (its copies may
//     land before the producer's arrival; the phase cannot complete without it).
// Lane e < ne handles the stage's block e (ne blocks per stage when
// block_size < 16); for per-block FP8 scales lanes 16 + e load V's.
// Returns false when the pipeline was aborted (a wait gave up).
// ---------------------------------------------------------------------------
template <int D, bool F8>
__device__ __forceinline__ bool stream_item(Smem<D, F8>& sm, const TMaps* tm, const AttnParams& p, const Desc& d,
                                            int si, int lane, uint32_t& g, int& next, bool vwarp) {
    constexpr int RS = Geo<D, F8>::kSlots;
    volatile int* abort = &sm.abort;
    const int bsr = p.bs < kTileT ? p.bs : kTileT;
    const CUtensorMap* map = vwarp ? &tm->v[log2i(d.hps)] : &tm->k[log2i(d.hps)];
    const uint32_t op_bytes = (uint32_t)d.hps * bsr * Geo<D, F8>::kRow;
    const int tb = d.t_begin / kTileT, te = (d.t_end + kTileT - 1) / kTileT;
    const int32_t* bt = p.block_tables + (long long)d.b * p.max_blocks;
    const int e_lim = (d.t_end + p.bs - 1) / p.bs;
    int tab_base = tb * kTileT / p.bs;
    int tab = tab_base + lane < e_lim ? __ldg(bt + tab_base + lane) : 0;
    int tab_next = tab_base + 32 + lane < e_lim ? __ldg(bt + tab_base + 32 + lane) : 0;
    // the next item is claimed a few stages before this one's last, so a
    // CTA never holds a second item for long and the queue balances finely
    const int i_claim = max(tb, te - kClaimAhead);
    const int be = lane & 15;  // this lane's block of the stage
    for (int i = tb; i < te; ++i, ++g) {
        if (!vwarp && i == i_claim && lane == 0) next = atomicAdd(&p.hdr[HDR_HEAD], 1);
        const int t0 = i * kTileT;
        const int tvalid = min(kTileT, d.t_end - t0);
        const int e0 = t0 / p.bs;
        const int ne = p.bs >= kTileT ? 1 : (tvalid + p.bs - 1) / p.bs;
        if (e0 >= tab_base + 32) {
            // entries advance by at most 16 per stage: shift in the prefetched batch
            tab = tab_next;
            tab_base += 32;
            const int en = tab_base + 32 + lane;
            tab_next = en < e_lim ? __ldg(bt + en) : 0;
        }
        const int off = e0 - tab_base + be;  // in [0, 48)
        const int lo = __shfl_sync(kFull, tab, off & 31);
        const int hi = __shfl_sync(kFull, tab_next, off & 31);
        int my = off < 32 ? lo : hi;
        const bool in = be < ne;
        const bool okb = !in || (my >= 0 && my < p.num_blocks);
        if (!okb) my = 0;
        const int s = (int)(g % RS);
        // FP8 pools with per-block scales (producer): lane 16 v + e loads the K
        // (v = 0) or V (v = 1) scales of block e for the group's kv heads now,
        // and stores them into the slot's scale rows once the slot is free --
        // before the barrier is armed, so the consumers' wait on it orders them
        float scv[kMaxHPS];
        const bool pbs = F8 && !vwarp && p.scale_pb != 0;
        // aligned scale rows travel as bulk copies on the stage's barrier
        const bool pbulk = pbs && p.scale_bulk != 0;
        const uint32_t scl_bytes = (uint32_t)d.hps * 4u;
        if (pbs && !pbulk && in) {
            // the scale rows (a few MB) are kept in L2 under evict-last: the
            // K/V stream would otherwise push them out, and a load that misses
            // to HBM here holds up every copy of the stage
            const uint64_t keep = l2_evict_last_policy();
            const float* src = ((lane >> 4) ? p.v_scale : p.k_scale) + (long long)my * p.n_kv + d.hg * d.hps;
#pragma unroll
            for (int h = 0; h < kMaxHPS; ++h) scv[h] = h < d.hps ? ld_keep_l2(src + h, keep) : 0.f;
        }
        bool got = true;
        const unsigned badmask = __ballot_sync(kFull, !okb);
        if (lane == 0) {
            if (!vwarp && badmask) {
                sm.poison[si] = 1;
                report(p.status, PKV_STATUS_BAD_BLOCK);
            }
            got = mbar_wait(&sm.empty[s], ((g / RS) & 1) ^ 1, abort);
        }
        if (!__shfl_sync(kFull, got, 0)) return false;  // never arm a barrier whose previous phase is open
        if (pbs && !pbulk) {
            if (in) {
#pragma unroll
                for (int h = 0; h < kMaxHPS; ++h)
                    if (h < d.hps) sm.scl[s][lane >> 4][be][h] = scv[h];
            }
            __syncwarp();
        }
        if (!vwarp && lane == 0)
            mbar_arrive_expect_tx(&sm.full[s], 2u * ne * op_bytes + (pbulk ? 2u * ne * scl_bytes : 0u));
        if (pbulk && in) {
            // lane 16 v + e: the K (v = 0) or V (v = 1) scale row of block e
            const float* src = ((lane >> 4) ? p.v_scale : p.k_scale) + (long long)my * p.n_kv + d.hg * d.hps;
            bulk_load(&sm.scl[s][lane >> 4][be][0], src, scl_bytes, &sm.full[s]);
        }
        if (in && lane < 16) {
            const int row0 = p.bs > kTileT ? (t0 % p.bs) : 0;
            // map dimensions {column of a 128-byte box, row, box, kv head,
            // block}; rows of a single box: {column, box, row, ...}
            uint8_t* dst = &sm.kv[s][vwarp ? 1 : 0][be * op_bytes];
            if constexpr (Geo<D, F8>::kNB > 1)
                tma_load_5d(dst, map, 0, row0, 0, d.hg * d.hps, my, &sm.full[s]);
            else
                tma_load_5d(dst, map, 0, 0, row0, d.hg * d.hps, my, &sm.full[s]);
        }
        __syncwarp();
    }
    return true;
}

// ---------------------------------------------------------------------------
// Producer warp: item queue and descriptors; the K copies of 16-token stages,
// both tensors of tcgen05 tile stages (with the helper warp).
// ---------------------------------------------------------------------------
template <int D, bool F8>
__device__ __forceinline__ void producer(Smem<D, F8>& sm, const TMaps* tm, const AttnParams& p, int lane) {
    constexpr int RS = Geo<D, F8>::kSlots;
    volatile int* abort = &sm.abort;
    if (lane < 4) {
        prefetch_tmap(&tm->k[lane]);
        prefetch_tmap(&tm->v[lane]);
    }
    // a workspace whose plan was made for another shape runs nothing (the
    // combine kernel then writes every output row NaN and reports it)
    const int num_items = p.hdr[HDR_KEY] == p.plan_key ? p.hdr[HDR_ITEMS] : 0;
    int next = 0;
    if (lane == 0) next = atomicAdd(&p.hdr[HDR_HEAD], 1);
    next = __shfl_sync(kFull, next, 0);
    uint32_t g = 0;
    for (int islot = 0;; ++islot) {
        const int si = islot % kSlots;
        const int cur = next;
        const bool end = cur >= num_items || *abort;
        Desc d;
        if (!end) {
            const int4 it = __ldg(p.items + cur);
            const int4 sq = __ldg(p.seqs + it.x);
            d = make_desc(it, sq, __ldg(p.seq_p + it.x));
        } else {
            d = Desc{0, 0, 1, 0, 0, 0, 0, 0, 0, KIND_END, 1, 1};
        }
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&sm.iempty[si], ((islot / kSlots) & 1) ^ 1, abort);
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) break;  // abort: publish nothing more
        if (lane == 0) {
            sm.desc[si] = d;
            sm.poison[si] = 0;
            mbar_arrive(&sm.ifull[si]);
        }
        if (end) break;
        if (d.kind == KIND_TC) {
            if (!produce_tc<D, F8>(sm, tm, p, d, si, lane, g, next, false)) break;
        } else {
            if (!stream_item<D, F8>(sm, tm, p, d, si, lane, g, next, false)) break;
        }
        next = __shfl_sync(kFull, next, 0);
    }
    // drain: wait until every issued stage has landed, bounded by time only --
    // an abort must not cut it short, or the CTA could exit with copies still
    // landing in its shared memory
    if (lane == 0) drain_ring<RS>(sm.full, g);
}

// The V warp's item loop: it follows the item sequence (and the ring's stage
// count) and copies V of every 16-token stage (tcgen05 tiles are the
// producer's and the helper warp's).
template <int D, bool F8>
__device__ __forceinline__ void v_warp(Smem<D, F8>& sm, const TMaps* tm, const AttnParams& p, int lane) {
    volatile int* abort = &sm.abort;
    uint32_t g = 0;
    int unused = 0;
    bool aborted = false;
    for (int islot = 0;; ++islot) {
        const int si = islot % kSlots;
        if (!mbar_wait(&sm.ifull[si], (islot / kSlots) & 1, abort)) {
            aborted = true;
            break;
        }
        const Desc d = sm.desc[si];
        if (d.kind == KIND_END) break;
        const int T = d.kind == KIND_TC ? kTcT : kTileT;
        const int ntiles = (d.t_end + T - 1) / T - d.t_begin / T;
        if (d.kind != KIND_TC) {
            uint32_t gg = g;
            if (!stream_item<D, F8>(sm, tm, p, d, si, lane, gg, unused, true)) {
                g = gg;  // stages up to the last one this warp waited for
                aborted = true;
                break;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.iempty[si]);
        g += (uint32_t)(d.kind == KIND_TC ? ntiles + 1 : ntiles);
    }
    // This warp's copies land on the producer's barriers: after the last item
    // g is the producer's own stage count, and the drain waits for the latest
    // phase of every slot; after an abort, for the stages it copied into,
    // bounded by time only.
    if (lane == 0 && (aborted || g > 0)) drain_ring<Geo<D, F8>::kSlots>(sm.full, g);
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
// Decode item on CUDA cores (q_len = 1): warp w < hps owns kv head
// hg * hps + w and its G query heads over every stage of the item.
// Lane layout: grp = lane / 8 owns tokens grp, grp+4, grp+8, grp+12 of a stage
// for the QK dot products (li = lane % 8 covers 8 dims per 128-byte box); for
// PV every lane owns D/32 output dims of all G heads.
// ---------------------------------------------------------------------------
template <int D, int G>
__device__ __forceinline__ void decode_item(Smem<D, false>& sm, const AttnParams& p, const Desc& d, int warp, int lane,
                                            uint32_t gbase, int ntiles, int si, volatile int* abort) {
    constexpr int NB = D / 64;   // 128-byte boxes per row
    constexpr int HL = 8 / G;    // lanes per head in an 8-lane group
    constexpr int DV = D / 32;   // PV dims per lane
    const bool active = warp < d.hps;
    const int lb = log2i(p.bs < kTileT ? p.bs : kTileT);
    const int hps_lb = d.hps << lb, h_lb = warp << lb;
    const int grp = lane >> 3, li = lane & 7;
    const int myh = li / HL;
    const int kvh = d.hg * d.hps + warp;
    float2 q2[G][4 * NB];
    if (active) {
        const __nv_bfloat16* qb = p.q + ((long long)d.q_row0 * p.n_q + (long long)kvh * G) * D;
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
    for (int i = 0; i < ntiles; ++i) {
        const uint32_t gi = gbase + i;
        const int s = (int)(gi % kRingSlots);
        mbar_wait(&sm.full[s], (gi / kRingSlots) & 1, abort);
        if (!active) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
            continue;
        }
        const uint8_t* kb = &sm.kv[s][0][0];
        const uint8_t* vb = &sm.kv[s][1][0];
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
                const int R = srow(h_lb, row, x, hps_lb, lb, NB);
                const uint4 kv = *reinterpret_cast<const uint4*>(kb + R * 128 + ((li ^ (R & 7)) << 4));
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
        }
        __syncwarp();
        // the correction factor is uniform over a head's lanes: fetch each head's
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float c = __shfl_sync(kFull, cr, h * HL);
#pragma unroll
            for (int j = 0; j < DV / 2; ++j) acc[h][j] = __fmul2_rn(acc[h][j], make_float2(c, c));
        }
#pragma unroll
        for (int t = 0; t < kTileT; ++t) {
            if (t < nvalid) {  // rows past the valid tokens may hold anything, even NaN
                float pv[G];
#pragma unroll
                for (int h = 0; h < G; ++h) pv[h] = sm.pbuf[warp][t * G + h];
                const int R = srow(h_lb, t, vbox, hps_lb, lb, NB);
                const uint8_t* src = vb + R * 128 + ((vch ^ (R & 7)) << 4) + voff;
                uint32_t vw[2];
                if constexpr (DV == 4) {
                    const uint2 w = *reinterpret_cast<const uint2*>(src);
                    vw[0] = w.x;
                    vw[1] = w.y;
                } else {
                    vw[0] = *reinterpret_cast<const uint32_t*>(src);
                }
#pragma unroll
                for (int j = 0; j < DV / 2; ++j) {
                    const float2 f = bf16x2_to_float2(vw[j]);
#pragma unroll
                    for (int h = 0; h < G; ++h) acc[h][j] = __ffma2_rn(make_float2(pv[h], pv[h]), f, acc[h][j]);
                }
            }
        }
        __syncwarp();  // pbuf is rewritten by this warp's next stage; the stage is read
        if (lane == 0) mbar_arrive(&sm.empty[s]);  // one arrival per consumer warp and stage
    }
    // finish: per head, m and l are uniform over its lanes; lane h*HL holds them.
    // The producer raises poison before it arms the stage with the bad block,
    // so after the last stage's wait the flag is final.
    const bool pois = sm.poison[si] != 0;
    if (active) {
        float mh[G], lh[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            mh[h] = __shfl_sync(kFull, m_run, h * HL);
            lh[h] = __shfl_sync(kFull, l_run, h * HL);
        }
        if (d.nparts == 1) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const long long orow = (long long)d.q_row0 * p.n_q + (long long)kvh * G + h;
                const float inv = 1.0f / lh[h];
                uint32_t w[DV / 2];
#pragma unroll
                for (int j = 0; j < DV / 2; ++j)
                    w[j] = pois ? 0x7fc07fc0u : float2_to_bf16x2(acc[h][j].x * inv, acc[h][j].y * inv);
                __nv_bfloat16* dst = p.out + orow * D + DV * lane;
                if constexpr (DV == 4)
                    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
                else
                    *reinterpret_cast<uint32_t*>(dst) = w[0];
            }
        } else {
            const float qnan = __int_as_float(0x7fc00000);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const long long orow = (long long)d.q_row0 * p.n_q + (long long)kvh * G + h;
                float* dst = p.part_o + (orow * p.np_max + d.part) * D + DV * lane;
#pragma unroll
                for (int j = 0; j < DV / 2; ++j) {
                    const float2 v = pois ? make_float2(qnan, qnan) : acc[h][j];
                    __stcg(reinterpret_cast<float2*>(dst + 2 * j), v);
                }
                if (lane == 0) __stcg(p.part_ml + orow * p.np_max + d.part, make_float2(mh[h], lh[h]));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Decode and short multi-query items on tensor cores: warp w < hps owns kv
// head hg * hps + w.  The product is taken transposed, tokens on the M axis
// and the columns -- (query, q head) pairs of the query tile, 8 per n-tile,
// NTN n-tiles -- on N:
//   S^T[16 x 8 NTN]  = K_tile[16 x D] . Q^T[D x 8 NTN]      (NTN D/16 mma m16n8k16)
//   O^T[D x 8 NTN]  += V_tile^T[D x 16] . P^T[16 x 8 NTN]   (NTN D/16 mma)
// A decode row (q_len = 1) is a tile of one query: its g <= 8 heads fill one
// n-tile, so g = 4 pads half of N instead of three quarters of M.  A short
// multi-query row of q_len <= 24 / g queries is one tile of up to three
// n-tiles, so every kv head of a block still shares one stage (32 KB copies of
// K and of V at the 8B shape) and each column applies its query's causal
// limit.  Three n-tiles hold 48 registers of Q^T fragments and 96 of O^T
// accumulators: they fit the consumer warpgroups' 224 registers (at the
// launch's 168 they spilled, and a speculative verification ran twice as slow
// as on mma.sync row tiles).  P^T's B fragments are the S^T accumulators
// transposed in registers (movmatrix).
// ---------------------------------------------------------------------------
template <int D, int NTN>
__device__ __forceinline__ void decode_tc_item(Smem<D, false>& sm, const AttnParams& p, const Desc& d, int warp, int lane,
                                               uint32_t gbase, int ntiles, int si, volatile int* abort) {
    constexpr int NB = D / 64;
    constexpr int NT = D / 16;
    const int G = p.G;
    const bool active = warp < d.hps;
    const int lb = log2i(p.bs < kTileT ? p.bs : kTileT);
    const int hps_lb = d.hps << lb, h_lb = warp << lb;
    const int kvh = d.hg * d.hps + warp;
    const int qd = lane & 3, qr = lane >> 2;
    // columns c < nq * G are (query c / G of the tile, q head c % G)
    const int ncols = d.nq * G;
    // Q^T as B fragments: n = column 8 nt + qr, k = dims
    uint32_t qb[NTN][NT][2];
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt) {
        const int c = 8 * nt + qr;
        const uint32_t* qrow =
            (active && c < ncols)
                ? reinterpret_cast<const uint32_t*>(
                      p.q + ((long long)(d.q_row0 + c / G) * p.n_q + (long long)kvh * G + c % G) * D)
                : nullptr;
#pragma unroll
        for (int ks = 0; ks < NT; ++ks) {
            qb[nt][ks][0] = qrow ? qrow[8 * ks + qd] : 0u;
            qb[nt][ks][1] = qrow ? qrow[8 * ks + 4 + qd] : 0u;
        }
    }
    float o[NT][NTN][4];  // O^T tile (mt, nt): (dim 16 mt + qr [+8], column 8 nt + 2 qd [+1])
#pragma unroll
    for (int mt = 0; mt < NT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
    // per column (8 nt + 2 qd + j): reference maximum, partial sum, last visible position
    float m[NTN][2], l[NTN][2];
    int lim[NTN][2];
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = 8 * nt + 2 * qd + j;
            m[nt][j] = -INFINITY;
            l[nt][j] = 0.f;
            lim[nt][j] = c < ncols ? d.t_vis - d.nq + c / G : -1;
        }
    const int mi = lane >> 3, mr = lane & 7;
    const int a_tok = ((mi & 1) << 3) + mr, a_hi = mi >> 1;   // K: (t0-7,lo) (t8-15,lo) (t0-7,hi) (t8-15,hi)
    const int v_tok = ((mi >> 1) << 3) + mr, v_hi = mi & 1;   // V: (t0-7,lo) (t0-7,hi) (t8-15,lo) (t8-15,hi)
    const int tb = d.t_begin / kTileT;
    for (int i = 0; i < ntiles; ++i) {
        const uint32_t gi = gbase + i;
        const int s = (int)(gi % kRingSlots);
        mbar_wait(&sm.full[s], (gi / kRingSlots) & 1, abort);
        if (!active) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
            continue;
        }
        const uint32_t kb = smem_u32(&sm.kv[s][0][0]);
        const uint32_t vb = smem_u32(&sm.kv[s][1][0]);
        const int t0 = (tb + i) * kTileT;
        const int nvalid = min(kTileT, d.t_end - t0);
        // S^T; with one n-tile, two accumulators halve the dependent mma chain
        float ca[NTN][4], cb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) ca[nt][0] = ca[nt][1] = ca[nt][2] = ca[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < NT; ++ks) {
            const int chunk = 2 * ks + a_hi;
            const int R = srow(h_lb, a_tok, chunk >> 3, hps_lb, lb, NB);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(kb + R * 128 + (((chunk & 7) ^ (R & 7)) << 4), a0, a1, a2, a3);
            if constexpr (NTN == 1) {
                mma_bf16_16816((ks & 1) ? cb : ca[0], a0, a1, a2, a3, qb[0][ks][0], qb[0][ks][1]);
            } else {
#pragma unroll
                for (int nt = 0; nt < NTN; ++nt) mma_bf16_16816(ca[nt], a0, a1, a2, a3, qb[nt][ks][0], qb[nt][ks][1]);
            }
        }
        if constexpr (NTN == 1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) ca[0][j] += cb[j];
        }
        // (token qr, column 2qd), (qr, 2qd+1), (qr+8, 2qd), (qr+8, 2qd+1) of each n-tile
        const bool va = qr < nvalid, vb8 = qr + 8 < nvalid;
        const int ta = t0 + qr, tb8 = t0 + qr + 8;
        float sv[NTN][4];
        bool fits = true;
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
            sv[nt][0] = va && ta <= lim[nt][0] ? ca[nt][0] * p.scale_log2 : -INFINITY;
            sv[nt][1] = va && ta <= lim[nt][1] ? ca[nt][1] * p.scale_log2 : -INFINITY;
            sv[nt][2] = vb8 && tb8 <= lim[nt][0] ? ca[nt][2] * p.scale_log2 : -INFINITY;
            sv[nt][3] = vb8 && tb8 <= lim[nt][1] ? ca[nt][3] * p.scale_log2 : -INFINITY;
            fits = fits && fmaxf(sv[nt][0], sv[nt][2]) <= m[nt][0] + kRescaleSlack &&
                   fmaxf(sv[nt][1], sv[nt][3]) <= m[nt][1] + kRescaleSlack;
        }
        // The reference maxima move only when a new score exceeds them by more
        // than kRescaleSlack (base-2 units), so most stages need no max
        // reduction and no rescale of O; probabilities stay <= 2^slack.  The
        // softmax is unchanged: O and l are relative to the same m.
        if (!__all_sync(kFull, fits)) {
#pragma unroll
            for (int nt = 0; nt < NTN; ++nt) {
                float x0 = fmaxf(sv[nt][0], sv[nt][2]), x1 = fmaxf(sv[nt][1], sv[nt][3]);
#pragma unroll
                for (int o8 = 4; o8 < 32; o8 <<= 1) {
                    x0 = fmaxf(x0, __shfl_xor_sync(kFull, x0, o8));
                    x1 = fmaxf(x1, __shfl_xor_sync(kFull, x1, o8));
                }
                const float n0 = fmaxf(m[nt][0], x0), n1 = fmaxf(m[nt][1], x1);
                const float c0 = n0 == -INFINITY ? 1.f : exp2f(m[nt][0] - n0);
                const float c1 = n1 == -INFINITY ? 1.f : exp2f(m[nt][1] - n1);
                l[nt][0] *= c0;
                l[nt][1] *= c1;
#pragma unroll
                for (int mt = 0; mt < NT; ++mt) {
                    o[mt][nt][0] *= c0;
                    o[mt][nt][1] *= c1;
                    o[mt][nt][2] *= c0;
                    o[mt][nt][3] *= c1;
                }
                m[nt][0] = n0;
                m[nt][1] = n1;
            }
        }
        uint32_t pb0[NTN], pb1[NTN];
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
            const float u0 = m[nt][0] == -INFINITY ? 0.f : m[nt][0], u1 = m[nt][1] == -INFINITY ? 0.f : m[nt][1];
            const float p0 = exp2f(sv[nt][0] - u0), p1 = exp2f(sv[nt][1] - u1);
            const float p2 = exp2f(sv[nt][2] - u0), p3 = exp2f(sv[nt][3] - u1);
            // l stays a per-lane partial sum (this lane's tokens); reduced once at the end
            l[nt][0] += p0 + p2;
            l[nt][1] += p1 + p3;
            pb0[nt] = movmatrix_trans(float2_to_bf16x2(p0, p1));  // (tokens 2qd, 2qd+1; column qr)
            pb1[nt] = movmatrix_trans(float2_to_bf16x2(p2, p3));  // (tokens 8+2qd, 9+2qd; column qr)
        }
        // V rows past the valid tokens may hold anything (even NaN): zero them
        const bool part = nvalid < kTileT;
        const uint32_t klo =
            part ? (2 * qd < nvalid ? 0x0000ffffu : 0u) | (2 * qd + 1 < nvalid ? 0xffff0000u : 0u) : 0xffffffffu;
        const uint32_t khi =
            part ? (8 + 2 * qd < nvalid ? 0x0000ffffu : 0u) | (9 + 2 * qd < nvalid ? 0xffff0000u : 0u) : 0xffffffffu;
#pragma unroll
        for (int mt = 0; mt < NT; ++mt) {
            const int chunk = 2 * mt + v_hi;
            const int R = srow(h_lb, v_tok, chunk >> 3, hps_lb, lb, NB);
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(vb + R * 128 + (((chunk & 7) ^ (R & 7)) << 4), a0, a1, a2, a3);
            if (part) {
                a0 &= klo;
                a1 &= klo;
                a2 &= khi;
                a3 &= khi;
            }
#pragma unroll
            for (int nt = 0; nt < NTN; ++nt) mma_bf16_16816(o[mt][nt], a0, a1, a2, a3, pb0[nt], pb1[nt]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);  // one arrival per consumer warp and stage
    }
    if (!active) return;
    const bool poisoned = sm.poison[si] != 0;  // final after the last stage's wait
    const float qnan = __int_as_float(0x7fc00000);
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float lj = l[nt][j];
#pragma unroll
            for (int o8 = 4; o8 < 32; o8 <<= 1) lj += __shfl_xor_sync(kFull, lj, o8);
            const int c = 8 * nt + 2 * qd + j;
            if (c >= ncols) continue;
            const long long orow = (long long)(d.q_row0 + c / G) * p.n_q + (long long)kvh * G + c % G;
            if (d.nparts == 1) {
                const float inv = 1.0f / lj;
                __nv_bfloat16* dst = p.out + orow * D + qr;
#pragma unroll
                for (int mt = 0; mt < NT; ++mt) {
                    dst[16 * mt] = poisoned ? __float2bfloat16_rn(qnan) : __float2bfloat16_rn(o[mt][nt][j] * inv);
                    dst[16 * mt + 8] =
                        poisoned ? __float2bfloat16_rn(qnan) : __float2bfloat16_rn(o[mt][nt][2 + j] * inv);
                }
            } else {
                float* dst = p.part_o + (orow * p.np_max + d.part) * D + qr;
#pragma unroll
                for (int mt = 0; mt < NT; ++mt) {
                    __stcg(dst + 16 * mt, poisoned ? qnan : o[mt][nt][j]);
                    __stcg(dst + 16 * mt + 8, poisoned ? qnan : o[mt][nt][2 + j]);
                }
                if (qr == 0) __stcg(p.part_ml + orow * p.np_max + d.part, make_float2(m[nt][j], lj));
            }
        }
    }
}

// Per-lane constants of a multi-query warp: causal limits of its rows A and
// B, shared-memory row indexing of the stage, ldmatrix lane roles.
struct MqLanes {
    int limA, limB, h_lb, hps_lb, lb, k_tok, k_hi, v_tok, v_hi, qd;
};

// One 16-token stage of a multi-query item (K at kb, V at vb, tokens t0 ..
// t0 + 15; positions at or past t_end are not part of the item): S = Q K^T,
// causal / tail mask, lazy reference maxima, O += P V.
template <int D>
__device__ __forceinline__ void mq_stage(uint32_t kb, uint32_t vb, int t0, int t_end, float scale_log2,
                                         const uint32_t (&qf)[D / 16][4], float (&o)[D / 8][4], float& mA, float& mB,
                                         float& lA, float& lB, const MqLanes& ml) {
    constexpr int NB = D / 64;
    const int qd = ml.qd;
    float sf[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const int chunk = 2 * ks + ml.k_hi;
        const int R = srow(ml.h_lb, ml.k_tok, chunk >> 3, ml.hps_lb, ml.lb, NB);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + R * 128 + (((chunk & 7) ^ (R & 7)) << 4), b0, b1, b2, b3);
        mma_bf16_16816(sf[0], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b0, b1);
        mma_bf16_16816(sf[1], qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3], b2, b3);
    }
    // scale, causal / tail mask (a stage whose 16 tokens every row of the warp
    // sees needs no mask: all stages but a partition's last ones)
    float mxA = -INFINITY, mxB = -INFINITY;
    if (__all_sync(kFull, t0 + kTileT <= t_end && t0 + kTileT - 1 <= min(ml.limA, ml.limB))) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float v = sf[nt][j] * scale_log2;
                sf[nt][j] = v;
                if (j < 2) mxA = fmaxf(mxA, v); else mxB = fmaxf(mxB, v);
            }
    } else {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int t = t0 + 8 * nt + 2 * qd + (j & 1);
                const int lim = j < 2 ? ml.limA : ml.limB;
                const bool vis = t < t_end && t <= lim;
                const float v = vis ? sf[nt][j] * scale_log2 : -INFINITY;
                sf[nt][j] = v;
                if (j < 2) mxA = fmaxf(mxA, v); else mxB = fmaxf(mxB, v);
            }
    }
    // lazy reference maxima (as in decode_tc_item): rows move theirs only when
    // a score exceeds it by more than kRescaleSlack
    if (!__all_sync(kFull, mxA <= mA + kRescaleSlack && mxB <= mB + kRescaleSlack)) {
        mxA = fmaxf(mxA, __shfl_xor_sync(kFull, mxA, 1));
        mxA = fmaxf(mxA, __shfl_xor_sync(kFull, mxA, 2));
        mxB = fmaxf(mxB, __shfl_xor_sync(kFull, mxB, 1));
        mxB = fmaxf(mxB, __shfl_xor_sync(kFull, mxB, 2));
        const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
        const float cA = nA == -INFINITY ? 1.f : exp2f(mA - nA), cB = nB == -INFINITY ? 1.f : exp2f(mB - nB);
        lA *= cA;
        lB *= cB;
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
            o[nt][0] *= cA;
            o[nt][1] *= cA;
            o[nt][2] *= cB;
            o[nt][3] *= cB;
        }
        mA = nA;
        mB = nB;
    }
    const float uA = mA == -INFINITY ? 0.f : mA, uB = mB == -INFINITY ? 0.f : mB;
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
    // l stays a per-lane partial sum (this lane's tokens); reduced once at the end
    lA += sA;
    lB += sB;
    const uint32_t pa0 = float2_to_bf16x2(sf[0][0], sf[0][1]);
    const uint32_t pa1 = float2_to_bf16x2(sf[0][2], sf[0][3]);
    const uint32_t pa2 = float2_to_bf16x2(sf[1][0], sf[1][1]);
    const uint32_t pa3 = float2_to_bf16x2(sf[1][2], sf[1][3]);
    if (t0 + kTileT <= t_end) {
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
            const int chunk = 2 * dp + ml.v_hi;
            const int R = srow(ml.h_lb, ml.v_tok, chunk >> 3, ml.hps_lb, ml.lb, NB);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vb + R * 128 + (((chunk & 7) ^ (R & 7)) << 4), b0, b1, b2, b3);
            mma_bf16_16816(o[2 * dp], pa0, pa1, pa2, pa3, b0, b1);
            mma_bf16_16816(o[2 * dp + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
    } else {
        // V rows past the valid tokens may hold anything (even NaN): zero them
        const int nvalid = t_end - t0;
        const uint32_t keep0 = (2 * qd < nvalid ? 0x0000ffffu : 0u) | (2 * qd + 1 < nvalid ? 0xffff0000u : 0u);
        const uint32_t keep1 =
            (8 + 2 * qd < nvalid ? 0x0000ffffu : 0u) | (8 + 2 * qd + 1 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
            const int chunk = 2 * dp + ml.v_hi;
            const int R = srow(ml.h_lb, ml.v_tok, chunk >> 3, ml.hps_lb, ml.lb, NB);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vb + R * 128 + (((chunk & 7) ^ (R & 7)) << 4), b0, b1, b2, b3);
            mma_bf16_16816(o[2 * dp], pa0, pa1, pa2, pa3, b0 & keep0, b1 & keep1);
            mma_bf16_16816(o[2 * dp + 1], pa0, pa1, pa2, pa3, b2 & keep0, b3 & keep1);
        }
    }
}

// ---------------------------------------------------------------------------
// Multi-query item on tensor cores (mma.sync m16n8k16, bf16 in, fp32 acc).
// Warp w serves kv head hw = w / wph of the group and its rows
// [16 rw, 16 rw + 16), rw = w % wph, of the query tile (rows are (query,
// q head) pairs of that kv head).
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void mq_item(Smem<D, false>& sm, const AttnParams& p, const Desc& d, int warp, int lane,
                                        uint32_t gbase, int ntiles, int si, volatile int* abort) {
    const int G = p.G;
    const int per = d.nq * G;                      // rows per kv head in this tile
    const int hw = warp / d.wph, rw = warp - hw * d.wph;
    const bool active = hw < d.hps && rw * 16 < per;
    const int lb = log2i(p.bs < kTileT ? p.bs : kTileT);
    const int hps_lb = d.hps << lb, h_lb = hw << lb;
    const int kvh = d.hg * d.hps + hw;
    const int qd = lane & 3, qr = lane >> 2;
    const int rA = rw * 16 + qr, rB = rA + 8;
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
            if (!active || qi >= d.nq) return nullptr;
            return reinterpret_cast<const uint32_t*>(
                p.q + ((long long)(d.q_row0 + qi) * p.n_q + (long long)kvh * G + hh) * D);
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
    // ldmatrix row addresses (per lane) inside a stage
    const int mi = lane >> 3, mrow = lane & 7;
    const int k_tok = ((mi >> 1) << 3) + mrow;  // K: (tok 0-7, d lo), (tok 0-7, d hi), (tok 8-15, d lo), ...
    const int k_hi = mi & 1;
    const int v_tok = ((mi & 1) << 3) + mrow;   // V: (tok 0-7, d lo), (tok 8-15, d lo), (tok 0-7, d hi), ...
    const int v_hi = mi >> 1;
    const MqLanes ml{limA, limB, h_lb, hps_lb, lb, k_tok, k_hi, v_tok, v_hi, qd};
    for (int i = 0; i < ntiles; ++i) {
        const uint32_t gi = gbase + i;
        const int s = (int)(gi % kRingSlots);
        mbar_wait(&sm.full[s], (gi / kRingSlots) & 1, abort);
        if (active)
            mq_stage<D>(smem_u32(&sm.kv[s][0][0]), smem_u32(&sm.kv[s][1][0]), (tb + i) * kTileT, d.t_end,
                        p.scale_log2, qf, o, mA, mB, lA, lB, ml);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);  // one arrival per consumer warp and stage
    }
    if (!active) return;
    lA += __shfl_xor_sync(kFull, lA, 1);
    lA += __shfl_xor_sync(kFull, lA, 2);
    lB += __shfl_xor_sync(kFull, lB, 1);
    lB += __shfl_xor_sync(kFull, lB, 2);
    const bool poisoned = sm.poison[si] != 0;  // final after the last stage's wait
    // finish from registers: rows rA, rB of kv head kvh
    const float qnan = __int_as_float(0x7fc00000);
    const float mfin[2] = {mA, mB}, lfin[2] = {lA, lB};
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = half ? rB : rA;
        const int qi = r / G, hh = r - qi * G;
        if (qi >= d.nq) continue;
        const long long orow = (long long)(d.q_row0 + qi) * p.n_q + (long long)kvh * G + hh;
        if (d.nparts == 1) {
            const float inv = 1.0f / lfin[half];
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                const uint32_t w = poisoned ? 0x7fc07fc0u
                                            : float2_to_bf16x2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
                *reinterpret_cast<uint32_t*>(p.out + orow * D + 8 * nt + 2 * qd) = w;
            }
        } else {
            float* dst = p.part_o + (orow * p.np_max + d.part) * D;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                const float2 v = poisoned ? make_float2(qnan, qnan) : make_float2(o[nt][2 * half], o[nt][2 * half + 1]);
                __stcg(reinterpret_cast<float2*>(dst + 8 * nt + 2 * qd), v);
            }
            if (qd == 0) __stcg(p.part_ml + orow * p.np_max + d.part, make_float2(mfin[half], lfin[half]));
        }
    }
}

// ---------------------------------------------------------------------------
// Query tile on the 5th-generation tensor cores (tcgen05, accumulators in
// tensor memory): the FlashAttention block loop of "Inference at Scale"
// section 07 for 128 rows = (query, q head) pairs of one kv head.
//   S_k  = Q K_k^T      (M 128, N 128 tokens, K = D): A = Q (shared memory,
//                        K-major), B = the stage's K slabs (K-major)
//   O_h += P_h V_k,h     (M 128, N = D, K 64 tokens): A = P (tensor memory,
//                        bf16), B = the stage's V slabs (MN-major)
// The two warpgroups split every stage's 128 tokens: warpgroup h (warps 4h ..
// 4h + 3) takes tokens [64 h, 64 h + 64) of each stage with its own running
// maximum, sum and accumulator O_h -- two independent online softmaxes over
// interleaved halves of the keys, merged once at the end with the same
// log-sum-exp rescaling as split-KV partitions (section 07, Flash-Decoding).
// So a stage needs no exchange between warps.  Thread (warp w, lane l) owns
// row r = 32 (w % 4) + l, the tensor-memory lane its warp may access.  It
// reads its 64 scores of S_k, writes its 64 probabilities (bf16) over the
// first 32 of those columns, and rescales its O_h only when its maximum moves
// by more than kRescaleSlack (lazy reference maximum, as in the other items).
// A dedicated MMA warp issues every tcgen05.mma (tc_mma): S_{k+1} once PV_{k-1}
// has read the S buffer it reuses, PV_k per half once that half's P is
// written; the PV commit releases the ring slot.  Every wait is a bounded
// mbarrier wait: a stalled warp can make the tile time out, never hang it.
// Tensor-memory columns: S0 [0, 128), S1 [128, 256), O_0 [256, 384),
// O_1 [384, 512).
// ---------------------------------------------------------------------------
struct TcState {
    uint32_t tmem;   // tensor-memory base
    uint32_t k;      // tcgen05 stages processed by this CTA (S / O buffer parity)
    uint32_t x;      // half-row exchanges done
    uint32_t tiles;  // tcgen05 tiles processed (entry / Q barrier parity)
};

// 2^x by the hardware approximation (MUFU), subnormal results flushed to 0:
// a probability below 2^-126 of the row maximum is 0 in the bf16 P anyway.
__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Softmax side of a tile (the eight consumer warps).
template <int D>
__device__ __forceinline__ void tc_item(Smem<D, false>& sm, const AttnParams& p, const Desc& d, int warp, int lane,
                                        uint32_t gbase, int ntiles, int si, TcState& st, volatile int* abort) {
    static_assert(D == 128, "tcgen05 tiles are built for head_dim 128");
    constexpr int kSlab = kTcT * 128;  // bytes of one 64-column slab of a stage
    const int G = p.G;
    const int quarter = warp & 3, hh = warp >> 2;
    const int r = quarter * 32 + lane;
    const int qi = r / G, hq = r - qi * G;
    const uint32_t tl = st.tmem + ((uint32_t)(quarter * 32) << 16);  // this warp's lanes
    const uint32_t tpar = st.tiles & 1;
    // every consumer warp has left its previous item (qbuf aliases pbuf, and
    // the previous tile's output reads are done)
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.ebar);
    mbar_wait(&sm.ebar, tpar, abort);
    // Q tile -> qbuf: 16-byte chunk j of row rr (slab x) at rr * 128 + ((j ^ (rr & 7)) << 4)
    for (int c = warp * 32 + lane; c < kTcRows * 16; c += kCThreads) {
        const int rr = c >> 4, c16 = c & 15, xs = c16 >> 3, jj = c16 & 7;
        const int qq = rr / G, h2 = rr - qq * G;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (qq < d.nq) v = ld_nc_v4(p.q + ((long long)(d.q_row0 + qq) * p.n_q + (long long)d.hg * G + h2) * D + c16 * 8);
        *reinterpret_cast<uint4*>(sm.qbuf + xs * kSlab + rr * 128 + ((jj ^ (rr & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.qbar);

    const int tb = d.t_begin / kTcT;
    // last visible position of this row (rows past the tile's queries take the last query's)
    const int lim = d.t_vis - d.nq + min(qi, d.nq - 1);
    const int last = min(lim, d.t_end - 1);
    const float sl2 = p.scale_log2;
    const bool pair = p.tc_pair != 0;
    const uint32_t ocol = kTmemO + (uint32_t)hh * D;  // this half's accumulator
    float m_ref = -INFINITY, l = 0.f;                 // this half's reference maximum and sum
    bool poisoned = false;
    for (int i = 0; i < ntiles; ++i) {
        const uint32_t k = st.k + i;
        const int b = (int)(k & 1);
        const uint32_t scol = kTmemS + (uint32_t)hh * 64;
        const uint32_t pcol = kTmemP + (uint32_t)b * (kTcT / 2) + (uint32_t)hh * 32;
        mbar_wait(&sm.sbar, k & 1, abort);
        __syncwarp();  // tcgen05.ld/st are warp-collective: reconverge after the polling wait
        tc_fence_after();
        uint32_t sv[64];
        tmem_ld32(tl + scol, sv);
        tmem_ld32(tl + scol + 32, sv + 32);
        tmem_wait_ld();
        // S_k is in registers: the MMA warp may overwrite the S buffer with S_{k+1}
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.sfree);
        // column j of this half holds stage token 64 hh + j, visible iff 64 hh + j <= lr
        const int lr = last - (tb + i) * kTcT;
        const bool full = lr >= 64 * hh + 63;
        float mx = -INFINITY;
        if (full) {
            // max of the scaled scores from the raw ones (the scale's sign picks max or min)
            float a = __uint_as_float(sv[0]);
            if (sl2 >= 0.f) {
#pragma unroll
                for (int j = 1; j < 64; ++j) a = fmaxf(a, __uint_as_float(sv[j]));
            } else {
#pragma unroll
                for (int j = 1; j < 64; ++j) a = fminf(a, __uint_as_float(sv[j]));
            }
            mx = a * sl2;
        } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const float v = 64 * hh + j <= lr ? __uint_as_float(sv[j]) * sl2 : -INFINITY;
                sv[j] = __float_as_uint(v);
                mx = fmaxf(mx, v);
            }
        }
        // O_h and l are relative to m_ref.  A row whose maximum moved rescales
        // its O_h once PV_{k-1} is done; the tensor-memory accesses are
        // warp-collective, so the whole warp takes the path (factor 1, exact,
        // for the rows that keep their reference)
        const bool move = mx > m_ref + kRescaleSlack;
        const float c = move && m_ref != -INFINITY ? ex2_fast(m_ref - mx) : 1.f;
        if (__any_sync(kFull, c != 1.f)) {
            const uint32_t kp = k - 1;  // i >= 1 here: a finite m_ref was set by an earlier stage
            mbar_wait(&sm.obar[kp & 1], (kp >> 1) & 1, abort);
            __syncwarp();
            tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t ov[32];
                tmem_ld32(tl + ocol + cc * 32, ov);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * c);
                tmem_st32(tl + ocol + cc * 32, ov);
            }
            tmem_wait_st();
        }
        if (move) {
            l *= c;
            m_ref = mx;  // (while m_ref was -inf every p was 0, so O_h and l are 0)
        }
        const float u = m_ref == -INFINITY ? 0.f : m_ref;
        float ls = 0.f;
        if (full) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {  // pair j overwrites sv[j], already consumed
                const float p0 = ex2_fast(fmaf(__uint_as_float(sv[2 * j]), sl2, -u));
                const float p1 = ex2_fast(fmaf(__uint_as_float(sv[2 * j + 1]), sl2, -u));
                ls += p0 + p1;
                sv[j] = float2_to_bf16x2(p0, p1);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float p0 = ex2_fast(__uint_as_float(sv[2 * j]) - u);
                const float p1 = ex2_fast(__uint_as_float(sv[2 * j + 1]) - u);
                ls += p0 + p1;
                sv[j] = float2_to_bf16x2(p0, p1);
            }
        }
        l += ls;
        // P_k into P buffer k & 1, once PV_{k-2} has read that buffer (within a
        // tile; an earlier tile's last PVs completed before its end)
        if (i >= 2) {
            const uint32_t k2 = k - 2;
            mbar_wait(&sm.obar[k2 & 1], (k2 >> 1) & 1, abort);
            __syncwarp();
            tc_fence_after();
        }
        tmem_st32(tl + pcol, sv);
        tmem_wait_st();
        if (i == ntiles - 1) {
            // the last V stage has landed (its slot is released only by PV_k):
            // the item's block checks are final, and this half's V rows past
            // the item's last position -- unfetched, or stale, possibly NaN --
            // are zeroed
            const uint32_t gv = gbase + i + 1;
            const int sv_ = (int)(gv % kRingSlots);
            mbar_wait(&sm.full[sv_], (gv / kRingSlots) & 1, abort);
            poisoned = sm.poison[si] != 0;
            const int nvalid = d.t_end - (tb + i) * kTcT;
            if (nvalid < kTcT) {
                uint8_t* vz = &sm.kv[sv_][1][0];
                // this half's 64 tokens x (2 slabs x 8 chunks of 16 B)
                for (int cz = quarter * 32 + lane; cz < 64 * 16; cz += 128) {
                    const int j = cz >> 4, xs = (cz >> 3) & 1, ch = cz & 7;
                    const int tok = 64 * hh + j;
                    if (tok < nvalid) continue;
                    const int off = pair ? (tok >> 4) * 4096 + xs * 2048 + (tok & 15) * 128 : xs * kSlab + tok * 128;
                    *reinterpret_cast<uint4*>(vz + off + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.pready[hh][k & 1]);
    }
    st.k += ntiles;
    ++st.tiles;
    // merge the two halves of each row: (m, l) through shared memory, then
    // O = O_0 c_0 + O_1 c_1 with c_h = 2^(m_h - m), l = l_0 c_0 + l_1 c_1
    sm.red[0][hh][r] = m_ref;
    sm.red[1][hh][r] = l;
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.xbar);
    mbar_wait(&sm.xbar, st.x & 1, abort);
    ++st.x;
    const float m_o = sm.red[0][hh ^ 1][r], l_o = sm.red[1][hh ^ 1][r];
    const float m0 = hh == 0 ? m_ref : m_o, m1 = hh == 0 ? m_o : m_ref;
    const float l0 = hh == 0 ? l : l_o, l1 = hh == 0 ? l_o : l;
    const float m = fmaxf(m0, m1);
    const float c0 = m0 == -INFINITY ? 0.f : ex2_fast(m0 - m), c1 = m1 == -INFINITY ? 0.f : ex2_fast(m1 - m);
    const float lrow = l0 * c0 + l1 * c1;
    const uint32_t kl = st.k - 1;
    mbar_wait(&sm.obar[kl & 1], (kl >> 1) & 1, abort);
    __syncwarp();
    tc_fence_after();
    const bool row_ok = qi < d.nq;
    const long long orow = (long long)(d.q_row0 + min(qi, d.nq - 1)) * p.n_q + (long long)d.hg * G + hq;
    const float inv = 1.0f / lrow;
    const float qnan = __int_as_float(0x7fc00000);
    // this thread writes output columns [64 hh, 64 hh + 64), in 32-column pieces
#pragma unroll 1
    for (int cc = 0; cc < 2; ++cc) {
        const int col0 = hh * 64 + cc * 32;
        uint32_t oa[32], ob[32];
        tmem_ld32(tl + kTmemO + col0, oa);
        tmem_ld32(tl + kTmemO + D + col0, ob);
        tmem_wait_ld();
        if (!row_ok) continue;
        float o[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = __uint_as_float(oa[j]) * c0 + __uint_as_float(ob[j]) * c1;
        if (d.nparts == 1) {
            uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D + col0);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint4 w;
                w.x = float2_to_bf16x2(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv);
                w.y = float2_to_bf16x2(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv);
                w.z = float2_to_bf16x2(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv);
                w.w = float2_to_bf16x2(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv);
                if (poisoned) w = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
                dst[q4] = w;
            }
        } else {
            float4* dst = reinterpret_cast<float4*>(p.part_o + (orow * p.np_max + d.part) * D + col0);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 v = poisoned ? make_float4(qnan, qnan, qnan, qnan)
                                          : make_float4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
                __stcg(dst + q4, v);
            }
        }
    }
    tc_fence_before();  // the next tile's first PV overwrites O after these reads
    if (row_ok && d.nparts > 1 && hh == 0) __stcg(p.part_ml + orow * p.np_max + d.part, make_float2(m, lrow));
}

// MMA side of a tile (the MMA warp; lane 0 issues).  K_i is in ring slot
// gbase + i, V_i in slot gbase + i + 1 (skewed slots, see produce_tc).
template <int D>
__device__ __forceinline__ void tc_mma(Smem<D, false>& sm, const Desc& d, int lane, uint32_t gbase, int ntiles,
                                       TcState& st, volatile int* abort, bool pair) {
    constexpr uint32_t kIdS = umma_idesc_bf16(kTcRows, kTcT, false);
    constexpr uint32_t kIdPV = umma_idesc_bf16(kTcRows, D, true);
    constexpr int kSlab = kTcT * 128;
    if (lane == 0) {
        // One thread issues every MMA, so the per-MMA work is kept to a few
        // adds: each operand's shared-memory descriptor is built once (per
        // tile for Q, per slot for K and V) and the k-step offsets are added
        // to its address field (address >> 4, 14 bits; every offset stays
        // inside its buffer, so no carry leaves the field).
        const uint64_t qdesc = umma_desc_sw128(smem_u32(sm.qbuf), 0);
        // S_i = Q K_i^T into the S buffer
        auto issue_s = [&](int i) -> bool {
            const uint32_t gi = gbase + i;
            const int s = (int)(gi % kRingSlots);
            if (!mbar_wait(&sm.full[s], (gi / kRingSlots) & 1, abort)) return false;
            tc_fence_after();
            const uint64_t kdesc = umma_desc_sw128(smem_u32(&sm.kv[s][0][0]), 0);
            const uint32_t dst = st.tmem + kTmemS;
#pragma unroll
            for (int xs = 0; xs < 2; ++xs)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t off = (uint64_t)((xs * kSlab + kk * 32) >> 4);
                    umma_ss(dst, qdesc + off, kdesc + off, kIdS, (xs | kk) != 0);
                }
            umma_commit(&sm.sbar);
            return true;
        };
        // Q written; the softmax warps wrote it after their previous tile had
        // ended, so they no longer need the S buffer S_0 overwrites
        bool ok = mbar_wait(&sm.qbar, st.tiles & 1, abort) && issue_s(0);
        if (ok) {
            // slot gbase holds K_0 alone: free once S_0 has read it
            const int s0 = (int)(gbase % kRingSlots);
            mbar_arrive(&sm.empty[s0], kCWarps - 1);
            umma_commit(&sm.empty[s0]);
        }
        for (int i = 0; ok && i < ntiles; ++i) {
            const uint32_t k = st.k + i;
            const int b = (int)(k & 1);
            if (i + 1 < ntiles) {
                // S_{k+1} overwrites S_k once every softmax warp holds S_k in
                // registers -- early in the softmax of stage k, so the tensor pipe
                // runs S_{k+1} beside it and PV_{k-1} (P lives in its own buffers)
                ok = mbar_wait(&sm.sfree, k & 1, abort);
                ok = ok && issue_s(i + 1);
            }
            const uint32_t gv = gbase + i + 1;
            const int sv = (int)(gv % kRingSlots);
            ok = ok && mbar_wait(&sm.full[sv], (gv / kRingSlots) & 1, abort);
            if (!ok) break;
            const uint32_t vb = smem_u32(&sm.kv[sv][1][0]);
            const uint64_t vdesc = pair ? umma_desc_sw128(vb, 2048) : umma_desc_sw128(vb, kSlab);
            // PV_k, each half once its four warps have written P
            for (int h = 0; h < 2; ++h) {
                ok = mbar_wait(&sm.pready[h][k & 1], (k >> 1) & 1, abort);
                if (!ok) break;
                tc_fence_after();
                // k-step kk of half h: tokens 64 h + 16 kk .. + 15 -- block
                // 4 h + kk of a paired V stage ([slab][16 rows] at 4 KB steps)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t bd =
                        vdesc + (uint64_t)((pair ? (4 * h + kk) * 4096 : (64 * h + 16 * kk) * 128) >> 4);
                    umma_ts(st.tmem + kTmemO + h * D, st.tmem + kTmemP + b * (kTcT / 2) + 32 * h + 8 * kk, bd,
                            kIdPV, i > 0 || kk > 0);
                }
            }
            if (!ok) break;
            umma_commit(&sm.obar[b]);
            // the slot's last arrival: once PV_k has read V_k (S_{k+1}, issued
            // earlier, has read K_{k+1})
            mbar_arrive(&sm.empty[sv], kCWarps - 1);
            umma_commit(&sm.empty[sv]);
        }
    }
    st.k += ntiles;
    ++st.tiles;
    __syncwarp();
}

// The MMA warp's item loop: it follows the item sequence (and the ring's
// stage count) and serves the tcgen05 tiles.
template <int D, bool F8>
__device__ __forceinline__ void mma_warp(Smem<D, F8>& sm, const AttnParams& p, int lane, TcState& tc) {
    volatile int* abort = &sm.abort;
    uint32_t g = 0;
    for (int islot = 0;; ++islot) {
        const int si = islot % kSlots;
        if (!mbar_wait(&sm.ifull[si], (islot / kSlots) & 1, abort)) break;
        const Desc d = sm.desc[si];
        if (d.kind == KIND_END) break;
        const int T = d.kind == KIND_TC ? kTcT : kTileT;
        const int ntiles = (d.t_end + T - 1) / T - d.t_begin / T;
        if constexpr (!F8) {
            if (d.kind == KIND_TC) tc_mma<D>(sm, d, lane, g, ntiles, tc, abort, p.tc_pair != 0);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.iempty[si]);
        g += (uint32_t)(d.kind == KIND_TC ? ntiles + 1 : ntiles);
    }
}

// The helper TMA warp's item loop: it follows the item sequence (and the
// ring's stage count) and issues the V copies of the tcgen05 tiles.
template <int D, bool F8>
__device__ __forceinline__ void helper_warp(Smem<D, F8>& sm, const TMaps* tm, const AttnParams& p, int lane) {
    volatile int* abort = &sm.abort;
    uint32_t g = 0;
    int unused = 0;
    bool aborted = false;
    for (int islot = 0;; ++islot) {
        const int si = islot % kSlots;
        if (!mbar_wait(&sm.ifull[si], (islot / kSlots) & 1, abort)) {
            aborted = true;
            break;
        }
        const Desc d = sm.desc[si];
        if (d.kind == KIND_END) break;
        const int T = d.kind == KIND_TC ? kTcT : kTileT;
        const int ntiles = (d.t_end + T - 1) / T - d.t_begin / T;
        if (d.kind == KIND_TC) {
            uint32_t gg = g;
            if (!produce_tc<D, F8>(sm, tm, p, d, si, lane, gg, unused, true)) {
                g = gg;  // stages up to the last one this warp copied into
                aborted = true;
                break;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.iempty[si]);
        g += (uint32_t)(d.kind == KIND_TC ? ntiles + 1 : ntiles);
    }
    // This warp's copies land on the producer's barriers.  After the last item
    // g is the producer's own stage count, so the drain waits for the latest
    // phase of every slot -- the one the producer's drain waits for too (an
    // older phase of a slot could alias the parity of a newer one).  After an
    // abort it waits for the stages this warp copied into, bounded by time
    // only: the producer may never have armed the last of them, and the wait
    // then gives up after the time limit, by which the copies have landed.
    if (lane == 0 && (aborted || g > 0)) drain_ring<Geo<D, F8>::kSlots>(sm.full, g);
}

// Four FP8 codes of one register -> (codes 0, 1) and (codes 2, 3) as f16x2
// (exact): e4m3 through the conversion instruction; an e5m2 code is the upper
// byte of the f16 of the same value, so e5m2 needs only a byte permute.
template <int FMT>
__device__ __forceinline__ void fp8x4_to_f16x2x2(uint32_t four, uint32_t& lo, uint32_t& hi) {
    if constexpr (FMT == 0) {
        e4m3x4_to_f16x2x2(four, lo, hi);
    } else {
        lo = __byte_perm(four, 0u, 0x1404);
        hi = __byte_perm(four, 0u, 0x3424);
    }
}

// V rows: bytes (t0 d0, t0 d1, t1 d0, t1 d1) of ldmatrix.trans -> the f16x2
// (t0 d0, t1 d0) and (t0 d1, t1 d1).
template <int FMT>
__device__ __forceinline__ void fp8x4_v_to_f16x2x2(uint32_t four, uint32_t& d0, uint32_t& d1) {
    if constexpr (FMT == 0) {
        e4m3x4_to_f16x2x2(__byte_perm(four, 0u, 0x3120), d0, d1);
    } else {
        d0 = __byte_perm(four, 0u, 0x2404);
        d1 = __byte_perm(four, 0u, 0x3414);
    }
}

// ---------------------------------------------------------------------------
// Item over an e4m3 pool ("Inference at Scale" section 03, KV cache
// quantization), any query tile of nq <= 8 * NTN / g queries: warp w < hps owns
// kv head hg * hps + w, in the transposed form of decode_tc_item with the
// columns N = (query, q head) pairs of the tile, 8 per n-tile, each with its
// own causal limit:
//   S^T[16 x 8 NTN] = K_tile[16 x D] . Q^T,   O^T[D x 8 NTN] += V_tile^T . P^T
// on f16 tensor cores (e4m3 -> f16 is exact; Q is rounded from bf16 to f16).
//   K: an ldmatrix row of 16 codes gives a lane 4 consecutive dims (4 qd ..
//      4 qd + 3) of its token; the two f16 pairs feed the k slots (2 qd, 2 qd + 1)
//      and (2 qd + 8, 2 qd + 9), and Q^T's fragments use the same permutation
//      of the dims, so the dot products are unchanged.
//   V: ldmatrix.trans of the byte pairs gives a lane tokens (2 qd, 2 qd + 1) x
//      dims (2 qr, 2 qr + 1); byte permutes split them into the m-rows qr
//      (dim 2 qr) and qr + 8 (dim 2 qr + 1), so O^T row r of chunk c holds dim
//      16 c + 2 (r mod 8) + r / 8.
// The per-head scales fold into the score scale (K) and the output (V).
// ---------------------------------------------------------------------------
// NS consecutive stages (i0, i0 + 1, ...) of a swap8 item: their S products
// are independent, so a warp running two at once hides more of the ldmatrix
// and MMA latency.
// FQ: bit 0 = e5m2 codes (else e4m3), bit 1 = a scale per (block, kv head)
// tile, read from the stage's scale rows (token qr's block and token qr + 8's;
// else the item's kv-head scale ksc, with V's applied at the end).
template <int D, int NTN, int NS, int FQ>
__device__ __forceinline__ void swap8_stages(Smem<D, true>& sm, const Desc& d, int i0, uint32_t gbase,
                                             const uint32_t (&qb)[NTN][D / 16][2], const int (&lim)[NTN][2],
                                             float (&o)[D / 16][NTN][4], float (&m)[NTN][2], float (&l)[NTN][2],
                                             float ksc, int R, int a_ch, int lane, volatile int* abort, int warp,
                                             int lb, float sl2) {
    constexpr int FMT = FQ & 1;
    constexpr bool PB = (FQ & 2) != 0;
    constexpr int RS = Geo<D, true>::kSlots;
    constexpr int NC = D / 16;
    const int qd = lane & 3, qr = lane >> 2;
    const int tb = d.t_begin / kTileT;
    int slot[NS], nvalid[NS], t0[NS];
#pragma unroll
    for (int u = 0; u < NS; ++u) {
        const uint32_t gi = gbase + i0 + u;
        slot[u] = (int)(gi % RS);
        mbar_wait(&sm.full[slot[u]], (gi / RS) & 1, abort);
        t0[u] = (tb + i0 + u) * kTileT;
        nvalid[u] = min(kTileT, d.t_end - t0[u]);
    }
    // S^T of every stage
    float sc[NS][2][NTN][4];
#pragma unroll
    for (int u = 0; u < NS; ++u)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int nt = 0; nt < NTN; ++nt) sc[u][h][nt][0] = sc[u][h][nt][1] = sc[u][h][nt][2] = sc[u][h][nt][3] = 0.f;
#pragma unroll
    for (int kc2 = 0; kc2 < NC / 2; ++kc2) {
        const int chunk = 2 * kc2 + a_ch;
#pragma unroll
        for (int u = 0; u < NS; ++u) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4(smem_u32(&sm.kv[slot[u]][0][0]) + R * 128 + (((chunk & 7) ^ (R & 7)) << 4), r0, r1, r2, r3);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t rA = h ? r2 : r0, rB = h ? r3 : r1;
                uint32_t a0, a1, a2, a3;
                fp8x4_to_f16x2x2<FMT>(rA, a0, a2);
                fp8x4_to_f16x2x2<FMT>(rB, a1, a3);
                const int kc = 2 * kc2 + h;
#pragma unroll
                for (int nt = 0; nt < NTN; ++nt)
                    mma_f16_16816(sc[u][h][nt], a0, a1, a2, a3, qb[nt][kc][0], qb[nt][kc][1]);
            }
        }
    }
    // scores (token qr / qr + 8, column 2 qd / 2 qd + 1) with the partition end
    // and each column's causal limit; lazy reference maxima as in decode_tc_item
    float sv[NS][NTN][4];
    // per-block scales of this lane's two tokens (qr, qr + 8) in each stage
    float kA[NS], kB[NS], vA[NS], vB[NS];
#pragma unroll
    for (int u = 0; u < NS; ++u) {
        if constexpr (PB) {
            const int eA = qr >> lb, eB = (qr + 8) >> lb;  // the tokens' blocks within the stage
            kA[u] = sm.scl[slot[u]][0][eA][warp] * sl2;
            kB[u] = sm.scl[slot[u]][0][eB][warp] * sl2;
            vA[u] = sm.scl[slot[u]][1][eA][warp];
            vB[u] = sm.scl[slot[u]][1][eB][warp];
        } else {
            kA[u] = kB[u] = ksc;
            vA[u] = vB[u] = 1.0f;
        }
    }
    bool fits = true;
#pragma unroll
    for (int u = 0; u < NS; ++u) {
        const int ta = t0[u] + qr, tb8 = t0[u] + qr + 8;
        const bool in_a = qr < nvalid[u], in_b = qr + 8 < nvalid[u];
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
            sv[u][nt][0] = in_a && ta <= lim[nt][0] ? (sc[u][0][nt][0] + sc[u][1][nt][0]) * kA[u] : -INFINITY;
            sv[u][nt][1] = in_a && ta <= lim[nt][1] ? (sc[u][0][nt][1] + sc[u][1][nt][1]) * kA[u] : -INFINITY;
            sv[u][nt][2] = in_b && tb8 <= lim[nt][0] ? (sc[u][0][nt][2] + sc[u][1][nt][2]) * kB[u] : -INFINITY;
            sv[u][nt][3] = in_b && tb8 <= lim[nt][1] ? (sc[u][0][nt][3] + sc[u][1][nt][3]) * kB[u] : -INFINITY;
            fits = fits && fmaxf(sv[u][nt][0], sv[u][nt][2]) <= m[nt][0] + kRescaleSlack &&
                   fmaxf(sv[u][nt][1], sv[u][nt][3]) <= m[nt][1] + kRescaleSlack;
        }
    }
    if (!__all_sync(kFull, fits)) {
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) {
            float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
            for (int u = 0; u < NS; ++u) {
                x0 = fmaxf(x0, fmaxf(sv[u][nt][0], sv[u][nt][2]));
                x1 = fmaxf(x1, fmaxf(sv[u][nt][1], sv[u][nt][3]));
            }
#pragma unroll
            for (int o8 = 4; o8 < 32; o8 <<= 1) {
                x0 = fmaxf(x0, __shfl_xor_sync(kFull, x0, o8));
                x1 = fmaxf(x1, __shfl_xor_sync(kFull, x1, o8));
            }
            const float n0 = fmaxf(m[nt][0], x0), n1 = fmaxf(m[nt][1], x1);
            const float c0 = n0 == -INFINITY ? 1.f : exp2f(m[nt][0] - n0);
            const float c1 = n1 == -INFINITY ? 1.f : exp2f(m[nt][1] - n1);
            l[nt][0] *= c0;
            l[nt][1] *= c1;
#pragma unroll
            for (int mc = 0; mc < NC; ++mc) {
                o[mc][nt][0] *= c0;
                o[mc][nt][1] *= c1;
                o[mc][nt][2] *= c0;
                o[mc][nt][3] *= c1;
            }
            m[nt][0] = n0;
            m[nt][1] = n1;
        }
    }
    uint32_t pb0[NS][NTN], pb1[NS][NTN];
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt) {
        const float u0 = m[nt][0] == -INFINITY ? 0.f : m[nt][0], u1 = m[nt][1] == -INFINITY ? 0.f : m[nt][1];
#pragma unroll
        for (int u = 0; u < NS; ++u) {
            const float p0 = exp2f(sv[u][nt][0] - u0), p1 = exp2f(sv[u][nt][1] - u1);
            const float p2 = exp2f(sv[u][nt][2] - u0), p3 = exp2f(sv[u][nt][3] - u1);
            l[nt][0] += p0 + p2;
            l[nt][1] += p1 + p3;
            // with per-block scales each token's V scale rides on its
            // probability in the P V product (the sum l stays unscaled)
            if constexpr (PB) {
                pb0[u][nt] = movmatrix_trans(float2_to_f16x2(p0 * vA[u], p1 * vA[u]));
                pb1[u][nt] = movmatrix_trans(float2_to_f16x2(p2 * vB[u], p3 * vB[u]));
            } else {
                pb0[u][nt] = movmatrix_trans(float2_to_f16x2(p0, p1));  // (tokens 2qd, 2qd+1; column qr)
                pb1[u][nt] = movmatrix_trans(float2_to_f16x2(p2, p3));  // (tokens 8+2qd, 9+2qd; column qr)
            }
        }
    }
    // V rows past the valid tokens may hold anything (even NaN): zero them
    uint32_t klo[NS], khi[NS];
#pragma unroll
    for (int u = 0; u < NS; ++u) {
        const int nv = nvalid[u];
        klo[u] = nv == kTileT ? 0xffffffffu
                              : (2 * qd < nv ? 0x0000ffffu : 0u) | (2 * qd + 1 < nv ? 0xffff0000u : 0u);
        khi[u] = nv == kTileT ? 0xffffffffu
                              : (8 + 2 * qd < nv ? 0x0000ffffu : 0u) | (9 + 2 * qd < nv ? 0xffff0000u : 0u);
    }
    bool partial = false;
#pragma unroll
    for (int u = 0; u < NS; ++u) partial = partial || nvalid[u] < kTileT;
#pragma unroll
    for (int kc2 = 0; kc2 < NC / 2; ++kc2) {
        const int chunk = 2 * kc2 + a_ch;
#pragma unroll
        for (int u = 0; u < NS; ++u) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_t(smem_u32(&sm.kv[slot[u]][1][0]) + R * 128 + (((chunk & 7) ^ (R & 7)) << 4), r0, r1, r2, r3);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t rA = h ? r2 : r0, rB = h ? r3 : r1;
                // bytes (t0 d0, t0 d1, t1 d0, t1 d1) -> (t0 d0, t1 d0 | t0 d1, t1 d1): one
                // permute, then each half converts to the f16 pair of one dim
                uint32_t a0, a1, a2, a3;
                fp8x4_v_to_f16x2x2<FMT>(rA, a0, a1);
                fp8x4_v_to_f16x2x2<FMT>(rB, a2, a3);
                if (partial) {
                    a0 &= klo[u];
                    a1 &= klo[u];
                    a2 &= khi[u];
                    a3 &= khi[u];
                }
                const int mc = 2 * kc2 + h;
#pragma unroll
                for (int nt = 0; nt < NTN; ++nt) mma_f16_16816(o[mc][nt], a0, a1, a2, a3, pb0[u][nt], pb1[u][nt]);
            }
        }
    }
    __syncwarp();
    if (lane == 0) {
#pragma unroll
        for (int u = 0; u < NS; ++u) mbar_arrive(&sm.empty[slot[u]]);  // one arrival per consumer warp and stage
    }
}

template <int D, int NTN, int FQ>
__device__ __forceinline__ void swap8_item(Smem<D, true>& sm, const AttnParams& p, const Desc& d, int warp, int lane,
                                           uint32_t gbase, int ntiles, int si, volatile int* abort) {
    constexpr bool PB = (FQ & 2) != 0;
    constexpr int RS = Geo<D, true>::kSlots;
    constexpr int NC = D / 16;  // 16-code chunks per row: k-steps of S, m-tiles of O
    static_assert(Geo<D, true>::kNB == 1, "e4m3 rows are one 128-byte box");
    const int G = p.G;
    const bool active = warp < d.hps;
    const int lb = log2i(p.bs < kTileT ? p.bs : kTileT);
    const int hps_lb = d.hps << lb, h_lb = warp << lb;
    const int kvh = d.hg * d.hps + warp;
    const int qd = lane & 3, qr = lane >> 2;
    const int ncols = d.nq * G;
    if (!active) {
        for (int i = 0; i < ntiles; ++i) {
            const uint32_t gi = gbase + i;
            mbar_wait(&sm.full[gi % RS], (gi / RS) & 1, abort);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[gi % RS]);
        }
        return;
    }
    uint32_t qb[NTN][NC][2];
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt) {
        const int c = 8 * nt + qr;
        const __nv_bfloat16* qrow =
            c < ncols ? p.q + ((long long)(d.q_row0 + c / G) * p.n_q + (long long)kvh * G + c % G) * D : nullptr;
#pragma unroll
        for (int kc = 0; kc < NC; ++kc) {
            uint2 raw = make_uint2(0u, 0u);
            if (qrow) raw = *reinterpret_cast<const uint2*>(qrow + 16 * kc + 4 * qd);
            const float2 x01 = bf16x2_to_float2(raw.x), x23 = bf16x2_to_float2(raw.y);
            qb[nt][kc][0] = float2_to_f16x2(x01.x, x01.y);
            qb[nt][kc][1] = float2_to_f16x2(x23.x, x23.y);
        }
    }
    // a scale per kv head: folded into the scores (K) and the output (V); per
    // block: read with each stage (swap8_stages)
    const float ksc = PB ? p.scale_log2 : __ldg(p.k_scale + kvh) * p.scale_log2;
    const float vsc = PB ? 1.0f : __ldg(p.v_scale + kvh);
    // last visible position of the two columns (2 qd, 2 qd + 1) of each n-tile
    int lim[NTN][2];
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = 8 * nt + 2 * qd + j;
            lim[nt][j] = c < ncols ? d.t_vis - d.nq + c / G : -1;
        }
    float o[NC][NTN][4];
#pragma unroll
    for (int mc = 0; mc < NC; ++mc)
#pragma unroll
        for (int nt = 0; nt < NTN; ++nt) o[mc][nt][0] = o[mc][nt][1] = o[mc][nt][2] = o[mc][nt][3] = 0.f;
    float m[NTN][2], l[NTN][2];
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt) m[nt][0] = m[nt][1] = -INFINITY, l[nt][0] = l[nt][1] = 0.f;
    const int mi = lane >> 3, mr = lane & 7;
    const int a_tok = ((mi & 1) << 3) + mr, a_ch = mi >> 1;  // (t0-7, c) (t8-15, c) (t0-7, c+1) (t8-15, c+1)
    const int R = srow(h_lb, a_tok, 0, hps_lb, lb, 1);
    int i = 0;
    if constexpr (NTN == 1) {
        for (; i + 1 < ntiles; i += 2)
            swap8_stages<D, NTN, 2, FQ>(sm, d, i, gbase, qb, lim, o, m, l, ksc, R, a_ch, lane, abort, warp, lb,
                                        p.scale_log2);
    }
    for (; i < ntiles; ++i)
        swap8_stages<D, NTN, 1, FQ>(sm, d, i, gbase, qb, lim, o, m, l, ksc, R, a_ch, lane, abort, warp, lb,
                                    p.scale_log2);
    const bool poisoned = sm.poison[si] != 0;  // final after the last stage's wait
    const float qnan = __int_as_float(0x7fc00000);
#pragma unroll
    for (int nt = 0; nt < NTN; ++nt) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float lj = l[nt][j];
#pragma unroll
            for (int o8 = 4; o8 < 32; o8 <<= 1) lj += __shfl_xor_sync(kFull, lj, o8);
            const int c = 8 * nt + 2 * qd + j;
            if (c >= ncols) continue;
            const long long orow = (long long)(d.q_row0 + c / G) * p.n_q + (long long)kvh * G + c % G;
            if (d.nparts == 1) {
                const float inv = vsc / lj;
                __nv_bfloat16* dst = p.out + orow * D + 2 * qr;
#pragma unroll
                for (int mc = 0; mc < NC; ++mc) {
                    const uint32_t v = poisoned ? 0x7fc07fc0u
                                                : float2_to_bf16x2(o[mc][nt][j] * inv, o[mc][nt][2 + j] * inv);
                    *reinterpret_cast<uint32_t*>(dst + 16 * mc) = v;
                }
            } else {
                float* dst = p.part_o + (orow * p.np_max + d.part) * D + 2 * qr;
#pragma unroll
                for (int mc = 0; mc < NC; ++mc)
                    __stcg(reinterpret_cast<float2*>(dst + 16 * mc),
                           poisoned ? make_float2(qnan, qnan)
                                    : make_float2(o[mc][nt][j] * vsc, o[mc][nt][2 + j] * vsc));
                if (qr == 0) __stcg(p.part_ml + orow * p.np_max + d.part, make_float2(m[nt][j], lj));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Combine kernel: one warp per (query row, q head) whose row was split into
// np > 1 partitions.  With M = max_p m_p and w_p = 2^(m_p - M),
//   O = (sum_p w_p O_p) / (sum_p w_p l_p)
// summed in partition order ("Chapter 31 Serving Efficiency", Example 31.2;
// "Inference at Scale", section 07, Flash-Decoding's log-sum-exp merge).
// ---------------------------------------------------------------------------
struct CombineParams {
    __nv_bfloat16* out;
    const float* part_o;
    const float2* part_ml;
    const int* row_np;   // [total_q] partitions of each query row (0 or 1: nothing to merge; -1: invalid
                         // sequence, the row is written NaN)
    int* hdr;            // workspace header: key check, queue head reset
    int32_t* status;
    int total_q, n_q, np_max, plan_key;
};

constexpr int kCombineThreads = 128;

template <int D>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const __grid_constant__ CombineParams c) {
    constexpr int V = D / 32;  // output dims per lane (4 or 2)
    constexpr int U = 8;       // partitions whose loads are in flight together
    pdl_wait();                // the attention grid has finished and its partials are visible
    pdl_launch();
    const int lane = threadIdx.x & 31;
    const long long nwarps = (long long)gridDim.x * (kCombineThreads / 32);
    const long long rows = (long long)c.total_q * c.n_q;
    const bool planned = c.hdr[HDR_KEY] == c.plan_key;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (planned) c.hdr[HDR_HEAD] = 0;  // the next call over this plan starts its queue at 0
        else report(c.status, PKV_STATUS_BAD_PLAN);
    }
    for (long long orow = (long long)blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5); orow < rows;
         orow += nwarps) {
        const int np = planned ? __ldg(c.row_np + orow / c.n_q) : -1;
        if (np < 0) {
            // a row of an invalid sequence, or a workspace without a plan for this shape
            __nv_bfloat16* dst = c.out + orow * D + lane * V;
            if constexpr (V == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(0x7fc07fc0u, 0x7fc07fc0u);
            else *reinterpret_cast<uint32_t*>(dst) = 0x7fc07fc0u;
            continue;
        }
        if (np <= 1) continue;
        const float2* ml = c.part_ml + orow * c.np_max;
        const float* src = c.part_o + orow * c.np_max * D + lane * V;
        // the first U partitions' outputs are loaded together with the
        // statistics (they do not depend on them): two dependent rounds of
        // loads for rows of up to U partitions
        float a[U][V];
        auto load_o = [&](int p0) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (p0 + u < np) {
                    const float* sp = src + (long long)(p0 + u) * D;
                    if constexpr (V == 4) {
                        const float4 t = __ldcg(reinterpret_cast<const float4*>(sp));
                        a[u][0] = t.x;
                        a[u][1] = t.y;
                        a[u][2] = t.z;
                        a[u][3] = t.w;
                    } else {
                        const float2 t = __ldcg(reinterpret_cast<const float2*>(sp));
                        a[u][0] = t.x;
                        a[u][1] = t.y;
                    }
                }
            }
        };
        // statistics: lane j holds partitions j, j + 32, ... (the first 32 kept in registers)
        const float2 s0 = lane < np ? __ldcg(ml + lane) : make_float2(-INFINITY, 0.f);
        load_o(0);
        float M = s0.x;
        for (int pp = lane + 32; pp < np; pp += 32) M = fmaxf(M, __ldcg(&ml[pp].x));
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        const float mu = M == -INFINITY ? 0.f : M;
        float acc[V];
#pragma unroll
        for (int j = 0; j < V; ++j) acc[j] = 0.f;
        float L = 0.f;
        for (int p0 = 0; p0 < np; p0 += 32) {
            float w = 0.f;
            if (p0 + lane < np) {
                const float2 s = p0 == 0 ? s0 : __ldcg(ml + p0 + lane);
                w = exp2f(s.x - mu);
                L += s.y * w;
            }
            const int n = min(32, np - p0);
            for (int u0 = 0; u0 < n; u0 += U) {
                if (p0 + u0 > 0) load_o(p0 + u0);  // (the first batch is in flight already)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float wu = __shfl_sync(kFull, w, (u0 + u) & 31);
                    if (u0 + u < n) {
#pragma unroll
                        for (int j = 0; j < V; ++j) acc[j] += wu * a[u][j];
                    }
                }
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(kFull, L, o);
        const float inv = 1.0f / L;
        __nv_bfloat16* dst = c.out + orow * D + lane * V;
        if constexpr (V == 4) {
            uint2 v;
            v.x = float2_to_bf16x2(acc[0] * inv, acc[1] * inv);
            v.y = float2_to_bf16x2(acc[2] * inv, acc[3] * inv);
            *reinterpret_cast<uint2*>(dst) = v;
        } else {
            *reinterpret_cast<uint32_t*>(dst) = float2_to_bf16x2(acc[0] * inv, acc[1] * inv);
        }
    }
}

template <int D>
int launch_combine(const CombineParams& c, cudaStream_t st) {
    const long long warps = (long long)c.total_q * c.n_q;
    long long grid = (warps + kCombineThreads / 32 - 1) / (kCombineThreads / 32);
    const long long cap = (long long)host::sm_count() * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    const cudaError_t e =
        host::launch_pdl(combine_kernel<D>, dim3((unsigned)grid), dim3(kCombineThreads), 0, st, c);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Consumer warps
// ---------------------------------------------------------------------------
// NTN: most n-tiles (8 columns each) of the transposed tensor-core items this
// kernel variant holds code for; a variant built for decode batches alone
// (NTN = 1) keeps its register allocation free of the wider items'.
// FQ (FP8 pools): bit 0 = e5m2 codes, bit 1 = per-block scales.
template <int D, int GD, bool F8, bool TC, int NTN, int FQ>
__device__ __forceinline__ void consumer(Smem<D, F8>& sm, const AttnParams& p, int warp, int lane, TcState& tc) {
    volatile int* abort = &sm.abort;
    uint32_t g = 0;
    for (int islot = 0;; ++islot) {
        const int si = islot % kSlots;
        if (!mbar_wait(&sm.ifull[si], (islot / kSlots) & 1, abort)) break;  // timed out: abort is set
        const Desc d = sm.desc[si];
        if (d.kind == KIND_END) break;
        const int T = d.kind == KIND_TC ? kTcT : kTileT;  // tokens per stage
        const int ntiles = (d.t_end + T - 1) / T - d.t_begin / T;
        const int nslots = d.kind == KIND_TC ? ntiles + 1 : ntiles;  // tcgen05 tiles: skewed K/V slots
        if (d.kind == KIND_TC) {
            if constexpr (TC) tc_item<D>(sm, p, d, warp, lane, g, ntiles, si, tc, abort);
        } else if constexpr (F8) {
            if (d.nq * p.G > 8) swap8_item<D, 2, FQ>(sm, p, d, warp, lane, g, ntiles, si, abort);
            else swap8_item<D, 1, FQ>(sm, p, d, warp, lane, g, ntiles, si, abort);
        } else {
            if (d.kind == KIND_DEC) {
                // columns of the tile: g heads of each of its nq queries, 8 per n-tile
                const int ncols = d.nq * p.G;
                if (NTN == 1 || ncols <= 8) decode_tc_item<D, 1>(sm, p, d, warp, lane, g, ntiles, si, abort);
                else if (NTN == 2 || ncols <= 16) {
                    if constexpr (NTN > 1) decode_tc_item<D, 2>(sm, p, d, warp, lane, g, ntiles, si, abort);
                } else {
                    if constexpr (NTN > 2) decode_tc_item<D, 3>(sm, p, d, warp, lane, g, ntiles, si, abort);
                }
            } else if (d.kind == KIND_MQ) {
                mq_item<D>(sm, p, d, warp, lane, g, ntiles, si, abort);
            } else {
                if constexpr (GD > 0) decode_item<D, GD>(sm, p, d, warp, lane, g, ntiles, si, abort);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.iempty[si]);  // this warp is done with the descriptor
        g += (uint32_t)nslots;
    }
}

__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
    uint32_t n;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(n));
    return n;
}

// Tensor memory of the tcgen05 variant, set up by the consumer warps and the
// MMA warp together: allocated (by consumer warp 0) only when the plan made
// tiles -- one CTA per SM, so the allocation never waits -- then one named
// barrier over those nine warps.  Returns whether tensor memory is in use.
template <int D, bool F8>
__device__ __forceinline__ bool tc_begin(Smem<D, F8>& sm, const AttnParams& p, int warp, TcState& tc) {
    const bool use_tc = p.tc != 0 && p.hdr[HDR_TC] != 0 && p.hdr[HDR_KEY] == p.plan_key;
    if (use_tc) {
        if (warp == 0) tmem_alloc(&sm.tmem, kTmemCols);
        tc_fence_before();
        named_bar(1, kCThreads + 32);  // consumers + the MMA warp, once
        tc_fence_after();
        tc.tmem = sm.tmem;
    }
    return use_tc;
}

// Release of the tensor memory once every MMA has completed and every warp is
// done with it (bounded by time alone: an abort must not skip the release).
template <int D, bool F8>
__device__ __forceinline__ void tc_end(Smem<D, F8>& sm, int warp, int lane, bool mma, const TcState& tc) {
    if (mma && lane == 0) {
        umma_commit(&sm.tdone);
        if (!mbar_wait_ns(&sm.tdone, 0)) sm.abort = 1;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.dbar);
    if (warp == 0) {
        if (!mbar_wait_ns(&sm.dbar, 0)) sm.abort = 1;
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tc.tmem, kTmemCols);
    }
}

// TC: the variant with tcgen05 tiles (head_dim 128, bf16), launched only for
// batches that may hold a tile (a row of more than kTcMinCols columns) -- the
// other variant carries none of the tile code.  Both launch kThreads threads:
// eight consumer warps and the side warpgroup (producer, MMA and helper warps
// of the tile variant, V warp).

template <int D, int GD, bool F8, bool TC, int NTN, int FQ>
__global__ void __launch_bounds__(kThreads, 1)
    paged_attention_kernel(const __grid_constant__ TMaps tm, const __grid_constant__ AttnParams p) {
    static_assert(!TC || Smem<D, F8>::kTC, "tcgen05 tiles need the head_dim 128 bf16 layout");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    using SM = Smem<D, F8>;
    constexpr int RS = Geo<D, F8>::kSlots;
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    if (base - reinterpret_cast<uintptr_t>(smem_raw) + sizeof(SM) > dynamic_smem_bytes()) {
        // the shared window is not 1024-byte aligned and the launch left no slack
        if (threadIdx.x == 0) report(p.status, PKV_STATUS_TIMEOUT);
        return;
    }
    SM& sm = *reinterpret_cast<SM*>(base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < RS; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kCWarps);
        }
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&sm.ifull[i], 1);
            mbar_init(&sm.iempty[i], kCWarps + 1 + (TC ? 2 : 0));  // + the V warp, the MMA and helper warps
        }
        if constexpr (TC) {
            mbar_init(&sm.sbar, 1);
            mbar_init(&sm.sfree, kCWarps);
            mbar_init(&sm.obar[0], 1);
            mbar_init(&sm.obar[1], 1);
            for (int h = 0; h < 2; ++h)
                for (int e = 0; e < 2; ++e) mbar_init(&sm.pready[h][e], kCWarps / 2);
            mbar_init(&sm.xbar, kCWarps);
            mbar_init(&sm.ebar, kCWarps);
            mbar_init(&sm.qbar, kCWarps);
            mbar_init(&sm.tdone, 1);
            mbar_init(&sm.dbar, kCWarps + 1);
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();    // the planning kernel's records are complete and visible
    pdl_launch();  // the combine kernel may be scheduled; it waits for this grid to finish
    // Register budgets per warpgroup: each role's code sits wholly inside the
    // branch that set its budget (code reached from both branches would be
    // held to the smaller one).
    if (warp >= kCWarps) {
        setmaxnreg_dec<kSideRegs>();
        if (warp == kCWarps) {
            producer<D, F8>(sm, &tm, p, lane);
        } else if (warp == kCWarps + 3) {
            v_warp<D, F8>(sm, &tm, p, lane);
        } else if constexpr (TC) {
            if (warp == kCWarps + 2) {
                helper_warp<D, F8>(sm, &tm, p, lane);
            } else if (warp == kCWarps + 1) {
                TcState tc{0u, 0u, 0u, 0u};
                const bool use_tc = tc_begin<D, F8>(sm, p, warp, tc);
                mma_warp<D, F8>(sm, p, lane, tc);
                if (use_tc) tc_end<D, F8>(sm, warp, lane, true, tc);
            }
        }
        // warps kCWarps + 1 and + 2 of the variant without tiles: no role
    } else {
        setmaxnreg_inc<kConsumerRegs>();
        TcState tc{0u, 0u, 0u, 0u};
        bool use_tc = false;
        if constexpr (TC) use_tc = tc_begin<D, F8>(sm, p, warp, tc);
        consumer<D, GD, F8, TC, NTN, FQ>(sm, p, warp, lane, tc);
        if constexpr (TC) {
            if (use_tc) tc_end<D, F8>(sm, warp, lane, false, tc);
        }
    }
    if (threadIdx.x == 0 && sm.abort) report(p.status, PKV_STATUS_TIMEOUT);
}

template <int D, int GD, bool F8 = false, bool TC = false, int NTN = 3, int FQ = 0>
int launch_attention(const TMaps& tm, const AttnParams& p, long long max_items, cudaStream_t st) {
    static int configured[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    // 1 KB of slack aligns the ring to 1024 bytes where the budget allows; the
    // shared window itself is 1024-byte aligned, which the kernel checks
    constexpr size_t kMaxSmem = 227 * 1024;
    const size_t smem = sizeof(Smem<D, F8>) + 1024 <= kMaxSmem ? sizeof(Smem<D, F8>) + 1024 : sizeof(Smem<D, F8>);
    static_assert(sizeof(Smem<D, F8>) <= kMaxSmem, "shared-memory budget");
    if (dev < 0 || dev >= 64) return PKV_ERR_CUDA;
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(paged_attention_kernel<D, GD, F8, TC, NTN, FQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return PKV_ERR_CUDA;
        // the warpgroups' setmaxnreg counts add up to kLaunchRegs a thread:
        // a build that launched with fewer would leave the consumers' request
        // waiting for registers the CTA does not have, so it is never launched
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, paged_attention_kernel<D, GD, F8, TC, NTN, FQ>) != cudaSuccess ||
            fa.numRegs != kLaunchRegs || fa.maxThreadsPerBlock < kThreads)
            return PKV_ERR_CUDA;
        configured[dev] = 1;
    }
    long long grid = host::sm_count();
    if (grid > max_items) grid = max_items;
    if (grid < 1) grid = 1;
    const cudaError_t e =
        host::launch_pdl(paged_attention_kernel<D, GD, F8, TC, NTN, FQ>, dim3((unsigned)grid), dim3(kThreads), smem, st,
                         tm, p);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// wide: the batch may hold transposed items of more than 8 columns (q_len * g
// > 8, at most kDecCols); otherwise the variant with decode items only runs.
template <int D>
int dispatch_g(int GD, bool wide, const TMaps& tm, const AttnParams& p, long long mi, cudaStream_t st) {
    switch (GD) {
        case 1: return launch_attention<D, 1>(tm, p, mi, st);
        case 2: return launch_attention<D, 2>(tm, p, mi, st);
        case 4: return launch_attention<D, 4>(tm, p, mi, st);
        case 8: return launch_attention<D, 8>(tm, p, mi, st);
        default:
            return wide ? launch_attention<D, 0, false, false, 3>(tm, p, mi, st)
                        : launch_attention<D, 0, false, false, 1>(tm, p, mi, st);
    }
}

int dispatch_attention_d64(int GD, bool wide, const TMaps& tm, const AttnParams& p, long long mi, cudaStream_t st);
int dispatch_attention_d128(int GD, bool tc, bool wide, const TMaps& tm, const AttnParams& p, long long mi,
                            cudaStream_t st);
int combine_d64(const CombineParams& c, cudaStream_t st);
int dispatch_attention_fp8_d128(int fq, const TMaps& tm, const AttnParams& p, long long mi, cudaStream_t st);
int combine_d128(const CombineParams& c, cudaStream_t st);

}  // namespace pkv
