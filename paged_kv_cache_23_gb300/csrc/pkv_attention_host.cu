// pkv_attention_host.cu -- planning kernel, workspace layout and the C entry
// points of the paged attention (kernels in pkv_attention.cuh).
#include "pkv_attention.cuh"

namespace pkv {

// ---------------------------------------------------------------------------
// Planning kernel
// ---------------------------------------------------------------------------
__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ int mq_items_of(int L, int ql, int G, int P) {
    const int QT = G >= kMqRows ? 1 : kMqRows / G;
    int n = 0;
    for (int qt = 0; qt * QT < ql; ++qt) {
        const int last = min(ql, (qt + 1) * QT);
        n += ceil_div(L - ql + last, P);
    }
    return n;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ PlanParams pp) {
    __shared__ int tmp[32];
    __shared__ int s_total_mq;
    const int tid = threadIdx.x;
    int bits = 0;
    // pass A: query row offsets and validity
    long long carry = 0;
    for (int base = 0; base < pp.num_seqs; base += kPlanThreads) {
        const int b = base + tid;
        int qlc = 0, flag = 0;
        if (b < pp.num_seqs) {
            const int L = pp.seq_lens[b], ql = pp.q_lens[b];
            if (L < 0 || (long long)L > (long long)pp.max_blocks * pp.bs || L > pp.max_seq_len)
                flag |= PKV_STATUS_BAD_SEQLEN;
            if (ql < 0 || ql > L) flag |= PKV_STATUS_BAD_QLEN;
            // clamp so the scan cannot overflow (total_q <= 2^20 is checked on the host)
            qlc = ql > 0 ? min(ql, pp.total_q + 1) : 0;
        }
        int tot;
        const int ex = block_exclusive_scan_1024(qlc, tmp, &tot);
        if (b < pp.num_seqs) {
            const long long q0 = carry + ex;
            if (q0 + qlc > pp.total_q) flag |= PKV_STATUS_BAD_QLEN;  // rows would overflow q/out
            pp.seq_q0[b] = (int)(q0 < pp.total_q ? q0 : pp.total_q);
            pp.seq_flag[b] = flag;
            bits |= flag;
        }
        carry += tot;
    }
    __syncthreads();
    // pass B: item counts
    int carry_mq = 0, carry_dec = 0;
    for (int base = 0; base < pp.num_seqs; base += kPlanThreads) {
        const int b = base + tid;
        int nmq = 0, ndec = 0;
        if (b < pp.num_seqs && pp.seq_flag[b] == 0) {
            const int L = pp.seq_lens[b], ql = pp.q_lens[b];
            if (ql == 1 && pp.decode_ok)
                ndec = ceil_div(L, pp.P) * pp.n_kv;
            else if (ql > 0)
                nmq = mq_items_of(L, ql, pp.G, pp.P) * pp.n_kv;
        }
        int tm, td;
        const int exm = block_exclusive_scan_1024(nmq, tmp, &tm);
        const int exd = block_exclusive_scan_1024(ndec, tmp, &td);
        if (b < pp.num_seqs) {
            pp.seq_mq_off[b] = carry_mq + exm;
            pp.seq_dec_off[b] = carry_dec + exd;
        }
        carry_mq += tm;
        carry_dec += td;
    }
    if (tid == 0) {
        s_total_mq = carry_mq;
        pp.hdr[0] = carry_mq + carry_dec;
        pp.hdr[1] = 0;
    }
    for (long long i = tid; i < (long long)pp.total_q * pp.n_kv; i += kPlanThreads) pp.tickets[i] = 0;
    __syncthreads();
    const int total_mq = s_total_mq;
    const int warp = tid >> 5, lane = tid & 31;
    const int QT = pp.G >= kMqRows ? 1 : kMqRows / pp.G;
    for (int b = warp; b < pp.num_seqs; b += kPlanThreads / 32) {
        const int flag = pp.seq_flag[b];
        const int L = pp.seq_lens[b], ql = pp.q_lens[b];
        const int q0 = pp.seq_q0[b];
        if (flag) {
            // rows of an invalid sequence are NaN (inside the q/out extent)
            const int qlc = ql > 0 ? min(ql, pp.total_q) : 0;
            const int rows = min(qlc, pp.total_q - q0);
            const long long n16 = (long long)rows * pp.n_q * pp.D / 8;
            uint4* o = reinterpret_cast<uint4*>(pp.out + (long long)q0 * pp.n_q * pp.D);
            for (long long e = lane; e < n16; e += 32) o[e] = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
            continue;
        }
        if (ql <= 0) continue;
        if (ql == 1 && pp.decode_ok) {
            const int nparts = ceil_div(L, pp.P);
            const int base = total_mq + pp.seq_dec_off[b];
            for (int it = lane; it < nparts * pp.n_kv; it += 32) {
                const int part = it / pp.n_kv, kvh = it - part * pp.n_kv;
                int4* d = pp.items + 3LL * (base + it);
                d[0] = make_int4(b, kvh, part, nparts);
                d[1] = make_int4(part * pp.P, min((part + 1) * pp.P, L), L, q0);
                d[2] = make_int4(1, KIND_DEC, 0, 0);
            }
        } else {
            int base = pp.seq_mq_off[b];
            for (int qt = 0; qt * QT < ql; ++qt) {
                const int nq = min(QT, ql - qt * QT);
                const int t_vis = L - ql + qt * QT + nq;
                const int nparts = ceil_div(t_vis, pp.P);
                for (int it = lane; it < nparts * pp.n_kv; it += 32) {
                    const int part = it / pp.n_kv, kvh = it - part * pp.n_kv;
                    int4* d = pp.items + 3LL * (base + it);
                    d[0] = make_int4(b, kvh, part, nparts);
                    d[1] = make_int4(part * pp.P, min((part + 1) * pp.P, t_vis), t_vis, q0 + qt * QT);
                    d[2] = make_int4(nq, KIND_MQ, 0, 0);
                }
                base += nparts * pp.n_kv;
            }
        }
    }
    if (bits) report(pp.status, bits);
}

struct WsLayout {
    size_t hdr, items, seq, tickets, ml, o, total;
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
    off = align256(off + (size_t)w.max_items * 48);
    w.seq = off;
    off = align256(off + (size_t)num_seqs * 4 * sizeof(int));
    w.tickets = off;
    off = align256(off + (size_t)total_q * n_kv * sizeof(int));
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

extern "C" int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                                          const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                                          const int32_t* q_lens, int num_seqs, int total_q, int max_seq_len,
                                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                          int num_blocks, float scale, int partition_tokens, int flags,
                                          void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
    if (num_seqs < 0 || total_q < 0 || max_blocks < 1 || max_seq_len < 0 || num_q_heads < 1 || num_kv_heads < 1 ||
        num_blocks < 1 || block_size < 1)
        return PKV_ERR_SIZE;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads) return PKV_ERR_UNSUPPORTED;
    const int G = num_q_heads / num_kv_heads;
    if (G > kMqRows) return PKV_ERR_UNSUPPORTED;
    if ((block_size & (block_size - 1)) || block_size > 256) return PKV_ERR_UNSUPPORTED;
    if ((long long)num_blocks * num_kv_heads * block_size >= (1LL << 31)) return PKV_ERR_SIZE;
    if (flags & ~PKV_ATTN_DECODE_TENSOR_CORES) return PKV_ERR_SIZE;
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

    CUtensorMap tmk, tmv;
    const uint64_t rows = (uint64_t)num_blocks * num_kv_heads * block_size;
    const uint32_t box_rows = block_size < kTileT ? (uint32_t)block_size : (uint32_t)kTileT;
    if (host::encode_tiled_2d(&tmk, k_cache, head_dim, rows, (uint64_t)head_dim * 2, 64, box_rows,
                              CU_TENSOR_MAP_SWIZZLE_128B) ||
        host::encode_tiled_2d(&tmv, v_cache, head_dim, rows, (uint64_t)head_dim * 2, 64, box_rows,
                              CU_TENSOR_MAP_SWIZZLE_128B))
        return PKV_ERR_CUDA;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* seq = reinterpret_cast<int*>(ws + w.seq);
    const int GD = (G == 1 || G == 2 || G == 4 || G == 8) ? G : 0;
    const bool decode_ok = GD > 0 && !(flags & PKV_ATTN_DECODE_TENSOR_CORES);

    PlanParams pp{};
    pp.seq_lens = seq_lens;
    pp.q_lens = q_lens;
    pp.items = reinterpret_cast<int4*>(ws + w.items);
    pp.hdr = reinterpret_cast<int*>(ws + w.hdr);
    pp.seq_q0 = seq;
    pp.seq_flag = seq + num_seqs;
    pp.seq_mq_off = seq + 2 * num_seqs;
    pp.seq_dec_off = seq + 3 * num_seqs;
    pp.tickets = reinterpret_cast<int*>(ws + w.tickets);
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
    pp.decode_ok = decode_ok ? 1 : 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    plan_kernel<<<1, kPlanThreads, 0, st>>>(pp);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;

    AttnParams ap{};
    ap.out = static_cast<__nv_bfloat16*>(out);
    ap.q = static_cast<const __nv_bfloat16*>(q);
    ap.block_tables = block_tables;
    ap.items = pp.items;
    ap.hdr = pp.hdr;
    ap.tickets = pp.tickets;
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
    ap.flags = flags;
    ap.scale_log2 = scale * 1.4426950408889634f;
    if (head_dim == 128) return dispatch_attention_d128(decode_ok ? GD : 0, tmk, tmv, ap, w.max_items, st);
    return dispatch_attention_d64(decode_ok ? GD : 0, tmk, tmv, ap, w.max_items, st);
}
