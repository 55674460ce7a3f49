// pkv_cache_ops.cu -- cache maintenance kernels of libpkv:
//   slot mapping, KV append, copy-on-write block copy, block-table gather.
//
// "Inference at Scale: KV Cache, Prefill, and Decode", section 05 ("The
// block table", "Block sharing and copy-on-write") and section 02 (decode
// appends one K/V row per new token); "Chapter 31 Serving Efficiency", 31.3.
//
// All four are byte movers: 16-byte vector loads and stores, grid-stride loops
// sized to the SM count.  Their cost is small next to the attention reread.
// They are launched as programmatic dependents (each waits for the previous
// kernel of the stream before touching memory), so back-to-back launches
// overlap their launch latency.
#include "pkv_common.cuh"
#include "pkv_host.h"

namespace pkv {

// ---------------------------------------------------------------------------
// Slot mapping: one CTA of 1024 threads; append_lens are scanned in shared
// memory, then every output slot finds its sequence by binary search.
// ---------------------------------------------------------------------------
constexpr int kSlotMaxSeqs = 16384;

__global__ void __launch_bounds__(1024) slot_mapping_kernel(int64_t* __restrict__ slots,
                                                            const int32_t* __restrict__ block_tables,
                                                            int max_blocks, const int32_t* __restrict__ seq_lens,
                                                            const int32_t* __restrict__ append_lens, int num_seqs,
                                                            int num_slots, int block_size, int num_blocks,
                                                            int32_t* status) {
    extern __shared__ int sh[];
    int* start = sh;                   // [num_seqs + 1] first output slot of each sequence
    int* bad = sh + num_seqs + 1;      // [num_seqs] invalid-length flag
    __shared__ int tmp[32];
    pdl_wait();  // programmatic dependent launch: the previous kernel's writes are visible
    pdl_launch();
    int bits = 0;
    int carry = 0;
    for (int base = 0; base < num_seqs; base += 1024) {
        const int b = base + threadIdx.x;
        int A = 0;
        if (b < num_seqs) {
            const int L = seq_lens[b];
            const int a = append_lens[b];
            int flag = 0;
            if (L < 0 || (long long)L > (long long)max_blocks * block_size) flag |= PKV_STATUS_BAD_SEQLEN;
            if (a < 0 || a > L) flag |= PKV_STATUS_BAD_QLEN;
            bad[b] = flag;
            bits |= flag;
            A = a > 0 ? a : 0;
        }
        int tot;
        const int ex = block_exclusive_scan_1024(A, tmp, &tot);
        if (b < num_seqs) start[b] = carry + ex;
        carry += tot;
    }
    if (threadIdx.x == 0) start[num_seqs] = carry;
    if (carry != num_slots) bits |= PKV_STATUS_BAD_QLEN;
    __syncthreads();
    const int n = carry < num_slots ? carry : num_slots;
    for (int o = threadIdx.x; o < num_slots; o += 1024) {
        if (o >= n) {
            slots[o] = -1;
            continue;
        }
        int lo = 0, hi = num_seqs - 1;  // last b with start[b] <= o
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (start[mid] <= o) lo = mid; else hi = mid - 1;
        }
        const int b = lo;
        if (bad[b]) {
            slots[o] = -1;
            continue;
        }
        const int L = seq_lens[b];
        const int A = start[b + 1] - start[b];
        const int pos = L - A + (o - start[b]);
        const int32_t blk = block_tables[(long long)b * max_blocks + pos / block_size];
        if (blk < 0 || blk >= num_blocks) {
            bits |= PKV_STATUS_BAD_BLOCK;
            slots[o] = -1;
            continue;
        }
        slots[o] = (int64_t)blk * block_size + pos % block_size;
    }
    report(status, bits);
}

// ---------------------------------------------------------------------------
// KV append: one 16-byte chunk per thread-iteration, K and V together.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) kv_append_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                        const uint4* __restrict__ k_new,
                                                        const uint4* __restrict__ v_new,
                                                        const int64_t* __restrict__ slots, int num_tokens,
                                                        int num_blocks, int block_size, int num_kv_heads,
                                                        int chunks_per_row, int32_t* status) {
    pdl_wait();
    pdl_launch();
    const long long per_tok = (long long)num_kv_heads * chunks_per_row;
    const long long total = (long long)num_tokens * per_tok;
    const long long cap = (long long)num_blocks * block_size;
    int bits = 0;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long t = i / per_tok;
        const long long rem = i - t * per_tok;
        const int h = (int)(rem / chunks_per_row);
        const int c = (int)(rem - (long long)h * chunks_per_row);
        const int64_t s = slots[t];
        if (s < 0) continue;
        if (s >= cap) {
            bits |= PKV_STATUS_BAD_SLOT;
            continue;
        }
        const long long blk = s / block_size;
        const int row = (int)(s - blk * block_size);
        const long long dst = ((blk * num_kv_heads + h) * block_size + row) * chunks_per_row + c;
        k_cache[dst] = ld_nc_v4(k_new + i);
        v_cache[dst] = ld_nc_v4(v_new + i);
    }
    report(status, bits);
}

// ---------------------------------------------------------------------------
// Slot mapping fused with the append: every 1024-thread CTA scans the
// append lengths into shared memory (batches up to kFusedMaxSeqs sequences),
// then each 16-byte chunk of a new row finds its sequence by binary search,
// forms the slot (as slot_mapping_kernel) and is copied (as kv_append_kernel).
// One launch instead of two.
// ---------------------------------------------------------------------------
constexpr int kFusedMaxSeqs = 2048;

__global__ void __launch_bounds__(1024) kv_append_paged_kernel(
    uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const uint4* __restrict__ k_new,
    const uint4* __restrict__ v_new, const int32_t* __restrict__ block_tables, int max_blocks,
    const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ append_lens, int num_seqs, int num_tokens,
    int num_blocks, int block_size, int num_kv_heads, int chunks_per_row, int64_t* __restrict__ slots,
    int32_t* status) {
    __shared__ int start[kFusedMaxSeqs + 1];
    __shared__ int bad[kFusedMaxSeqs];
    __shared__ int tmp[32];
    pdl_wait();
    pdl_launch();
    int bits = 0;
    int carry = 0;
    for (int base = 0; base < num_seqs; base += 1024) {
        const int b = base + threadIdx.x;
        int A = 0;
        if (b < num_seqs) {
            const int L = seq_lens[b];
            const int a = append_lens[b];
            int flag = 0;
            if (L < 0 || (long long)L > (long long)max_blocks * block_size) flag |= PKV_STATUS_BAD_SEQLEN;
            if (a < 0 || a > L) flag |= PKV_STATUS_BAD_QLEN;
            bad[b] = flag;
            if (blockIdx.x == 0) bits |= flag;
            A = a > 0 ? min(a, num_tokens + 1) : 0;
        }
        int tot;
        const int ex = block_exclusive_scan_1024(A, tmp, &tot);
        if (b < num_seqs) start[b] = carry + ex;
        carry += tot;
    }
    if (threadIdx.x == 0) start[num_seqs] = carry;
    if (blockIdx.x == 0 && threadIdx.x == 0 && carry != num_tokens) bits |= PKV_STATUS_BAD_QLEN;
    __syncthreads();
    const int n = carry < num_tokens ? carry : num_tokens;
    const long long cap = (long long)num_blocks * block_size;
    const long long per_tok = (long long)num_kv_heads * chunks_per_row;
    const long long total = (long long)num_tokens * per_tok;
    for (long long i = blockIdx.x * 1024LL + threadIdx.x; i < total; i += (long long)gridDim.x * 1024) {
        const int o = (int)(i / per_tok);
        const long long rem = i - (long long)o * per_tok;
        int64_t slot = -1;
        if (o < n) {
            int lo = 0, hi = num_seqs - 1;  // last b with start[b] <= o
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (start[mid] <= o) lo = mid; else hi = mid - 1;
            }
            const int b = lo;
            if (!bad[b]) {
                const int L = seq_lens[b];
                const int pos = L - (start[b + 1] - start[b]) + (o - start[b]);
                const int32_t blk = block_tables[(long long)b * max_blocks + pos / block_size];
                if (blk < 0 || blk >= num_blocks) {
                    if (rem == 0) bits |= PKV_STATUS_BAD_BLOCK;
                } else {
                    slot = (int64_t)blk * block_size + pos % block_size;
                }
            }
        }
        if (rem == 0) slots[o] = slot;
        if (slot < 0 || slot >= cap) continue;
        const int h = (int)(rem / chunks_per_row);
        const int c = (int)(rem - (long long)h * chunks_per_row);
        const long long blk = slot / block_size;
        const int row = (int)(slot - blk * block_size);
        const long long dst = ((blk * num_kv_heads + h) * block_size + row) * chunks_per_row + c;
        k_cache[dst] = ld_nc_v4(k_new + i);
        v_cache[dst] = ld_nc_v4(v_new + i);
    }
    if (bits) report(status, bits);
}

// ---------------------------------------------------------------------------
// KV append into e4m3 pools ("Inference at Scale" section 03, KV cache
// quantization): code = e4m3(x * (1 / scale[head])), the reciprocal and the
// product rounded to fp32 (nearest even), the conversion rounding to nearest
// even and saturating to +-448.  8 values (16 bytes in, 8 out) per thread.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(uint2* __restrict__ k_cache, uint2* __restrict__ v_cache,
                                                            const uint4* __restrict__ k_new,
                                                            const uint4* __restrict__ v_new,
                                                            const int64_t* __restrict__ slots,
                                                            const float* __restrict__ k_scale,
                                                            const float* __restrict__ v_scale, int num_tokens,
                                                            int num_blocks, int block_size, int num_kv_heads,
                                                            int chunks_per_row, int32_t* status) {
    pdl_wait();
    pdl_launch();
    const long long per_tok = (long long)num_kv_heads * chunks_per_row;
    const long long total = (long long)num_tokens * per_tok;
    const long long cap = (long long)num_blocks * block_size;
    int bits = 0;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long t = i / per_tok;
        const long long rem = i - t * per_tok;
        const int h = (int)(rem / chunks_per_row);
        const int c = (int)(rem - (long long)h * chunks_per_row);
        const int64_t s = slots[t];
        if (s < 0) continue;
        if (s >= cap) {
            bits |= PKV_STATUS_BAD_SLOT;
            continue;
        }
        const long long blk = s / block_size;
        const int row = (int)(s - blk * block_size);
        const long long dst = ((blk * num_kv_heads + h) * block_size + row) * chunks_per_row + c;
        const float ik = __fdiv_rn(1.0f, __ldg(k_scale + h)), iv = __fdiv_rn(1.0f, __ldg(v_scale + h));
        const uint4 a = ld_nc_v4(k_new + i), b = ld_nc_v4(v_new + i);
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
        uint32_t ck[4], cv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 xk = bf16x2_to_float2(wa[u]), xv = bf16x2_to_float2(wb[u]);
            ck[u] = f32x2_to_e4m3x2(__fmul_rn(xk.x, ik), __fmul_rn(xk.y, ik));
            cv[u] = f32x2_to_e4m3x2(__fmul_rn(xv.x, iv), __fmul_rn(xv.y, iv));
        }
        k_cache[dst] = make_uint2(ck[0] | (ck[1] << 16), ck[2] | (ck[3] << 16));
        v_cache[dst] = make_uint2(cv[0] | (cv[1] << 16), cv[2] | (cv[3] << 16));
    }
    report(status, bits);
}

// ---------------------------------------------------------------------------
// FP8 pools of either format ("Inference at Scale" section 03: e4m3 or e5m2),
// with a dequantisation scale per kv head or per (block, kv head) tile.
//
// Per-block scales are set when a block is opened: the append that writes a
// block's row 0 first sets, from that row's values of each kv head, the
// smallest power of two s = 2^e (e in [-120, 120]) with max|x| <= s * FMAX / 2
// (FMAX = 448 for e4m3, 57344 for e5m2; NaN values ignored; s = 1 for an
// all-zero or infinite row), so the opening row uses at most half of the range
// and later rows may grow to twice its magnitude before they saturate.  A
// first kernel sets the scales of the blocks this call opens (one warp per
// (opening token, kv head)); the quantising kernel, its programmatic
// dependent, then stores every row with its block's scales.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float open_block_scale(float amax, int fmt) {
    if (!(amax > 0.0f) || isinf(amax)) return 1.0f;
    const float half = fmt ? 28672.0f : 224.0f;
    // start from the exponent difference, then settle by exact comparisons
    int e = ilogbf(amax) - ilogbf(half);
    e = max(-120, min(120, e));
    while (e < 120 && ldexpf(half, e) < amax) ++e;
    while (e > -120 && ldexpf(half, e - 1) >= amax) --e;
    return ldexpf(1.0f, e);
}

__global__ void __launch_bounds__(256) fp8_open_blocks_kernel(const uint4* __restrict__ k_new,
                                                              const uint4* __restrict__ v_new,
                                                              const int64_t* __restrict__ slots,
                                                              float* __restrict__ k_scale,
                                                              float* __restrict__ v_scale, int num_tokens,
                                                              int num_blocks, int block_size, int num_kv_heads,
                                                              int chunks_per_row, int fmt) {
    pdl_wait();
    pdl_launch();
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    const long long cap = (long long)num_blocks * block_size;
    for (long long wi = blockIdx.x * (long long)(blockDim.x >> 5) + (threadIdx.x >> 5);
         wi < (long long)num_tokens * num_kv_heads; wi += warps) {
        const long long t = wi / num_kv_heads;
        const int h = (int)(wi - t * num_kv_heads);
        const int64_t s = slots[t];
        if (s < 0 || s >= cap || s % block_size != 0) continue;  // not a block's opening row
        float ak = 0.0f, av = 0.0f;
        const uint4* kr = k_new + (t * num_kv_heads + h) * chunks_per_row;
        const uint4* vr = v_new + (t * num_kv_heads + h) * chunks_per_row;
        for (int c = lane; c < chunks_per_row; c += 32) {
            const uint4 a = ld_nc_v4(kr + c), b = ld_nc_v4(vr + c);
            const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 xk = bf16x2_to_float2(wa[u]), xv = bf16x2_to_float2(wb[u]);
                // fmaxf ignores a NaN operand: NaN values do not enter the maximum
                ak = fmaxf(ak, fmaxf(fabsf(xk.x), fabsf(xk.y)));
                av = fmaxf(av, fmaxf(fabsf(xv.x), fabsf(xv.y)));
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            ak = fmaxf(ak, __shfl_xor_sync(kFull, ak, o));
            av = fmaxf(av, __shfl_xor_sync(kFull, av, o));
        }
        if (lane == 0) {
            const long long blk = s / block_size;
            k_scale[blk * num_kv_heads + h] = open_block_scale(ak, fmt);
            v_scale[blk * num_kv_heads + h] = open_block_scale(av, fmt);
        }
    }
}

// fp32 pair -> two FP8 codes of format fmt (round to nearest even, saturating
// to the largest finite value, NaN kept), lo in the lower byte.
__device__ __forceinline__ uint32_t f32x2_to_fp8x2(float lo, float hi, int fmt) {
    return fmt ? (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E5M2)
               : f32x2_to_e4m3x2(lo, hi);
}

// Quantising append of either format and scale granularity: code =
// fp8(x * (1 / scale)), the reciprocal and the product rounded to fp32.
// 8 values (16 bytes in, 8 out) per thread.
__global__ void __launch_bounds__(256) kv_append_fp8_ex_kernel(uint2* __restrict__ k_cache,
                                                               uint2* __restrict__ v_cache,
                                                               const uint4* __restrict__ k_new,
                                                               const uint4* __restrict__ v_new,
                                                               const int64_t* __restrict__ slots,
                                                               const float* __restrict__ k_scale,
                                                               const float* __restrict__ v_scale, int num_tokens,
                                                               int num_blocks, int block_size, int num_kv_heads,
                                                               int chunks_per_row, int fmt, int per_block,
                                                               int32_t* status) {
    pdl_wait();  // the scales of the blocks this call opens are set and visible
    pdl_launch();
    const long long per_tok = (long long)num_kv_heads * chunks_per_row;
    const long long total = (long long)num_tokens * per_tok;
    const long long cap = (long long)num_blocks * block_size;
    int bits = 0;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long t = i / per_tok;
        const long long rem = i - t * per_tok;
        const int h = (int)(rem / chunks_per_row);
        const int c = (int)(rem - (long long)h * chunks_per_row);
        const int64_t s = slots[t];
        if (s < 0) continue;
        if (s >= cap) {
            bits |= PKV_STATUS_BAD_SLOT;
            continue;
        }
        const long long blk = s / block_size;
        const int row = (int)(s - blk * block_size);
        const long long dst = ((blk * num_kv_heads + h) * block_size + row) * chunks_per_row + c;
        const long long si = per_block ? blk * num_kv_heads + h : h;
        const float ik = __fdiv_rn(1.0f, k_scale[si]), iv = __fdiv_rn(1.0f, v_scale[si]);
        const uint4 a = ld_nc_v4(k_new + i), b = ld_nc_v4(v_new + i);
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
        uint32_t ck[4], cv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 xk = bf16x2_to_float2(wa[u]), xv = bf16x2_to_float2(wb[u]);
            ck[u] = f32x2_to_fp8x2(__fmul_rn(xk.x, ik), __fmul_rn(xk.y, ik), fmt);
            cv[u] = f32x2_to_fp8x2(__fmul_rn(xv.x, iv), __fmul_rn(xv.y, iv), fmt);
        }
        k_cache[dst] = make_uint2(ck[0] | (ck[1] << 16), ck[2] | (ck[3] << 16));
        v_cache[dst] = make_uint2(cv[0] | (cv[1] << 16), cv[2] | (cv[3] << 16));
    }
    report(status, bits);
}

// The scales of the copied blocks: pair i copies row src of k_scale / v_scale
// ([num_blocks][n_kv]) to row dst.
__global__ void copy_block_scales_kernel(float* __restrict__ k_scale, float* __restrict__ v_scale,
                                         const int32_t* __restrict__ src_dst, int num_pairs, int num_blocks,
                                         int num_kv_heads) {
    pdl_wait();
    pdl_launch();
    const long long n = (long long)num_pairs * num_kv_heads;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x) {
        const int pr = (int)(i / num_kv_heads), h = (int)(i - (long long)pr * num_kv_heads);
        const int32_t s = src_dst[2 * pr], d = src_dst[2 * pr + 1];
        if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) continue;  // reported by the block copy
        k_scale[(long long)d * num_kv_heads + h] = k_scale[(long long)s * num_kv_heads + h];
        v_scale[(long long)d * num_kv_heads + h] = v_scale[(long long)s * num_kv_heads + h];
    }
}

// ---------------------------------------------------------------------------
// Copy blocks: blockIdx.y = pair, grid-stride over the block's 16-byte chunks.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                                          const int32_t* __restrict__ src_dst, int num_blocks,
                                                          long long chunks_per_block, int32_t* status) {
    pdl_wait();
    pdl_launch();
    const int pair = blockIdx.y;
    const int32_t s = src_dst[2 * pair], d = src_dst[2 * pair + 1];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
        if (blockIdx.x == 0 && threadIdx.x == 0) report(status, PKV_STATUS_BAD_PAIR);
        return;
    }
    const uint4* ks = k_cache + (long long)s * chunks_per_block;
    const uint4* vs = v_cache + (long long)s * chunks_per_block;
    uint4* kd = k_cache + (long long)d * chunks_per_block;
    uint4* vd = v_cache + (long long)d * chunks_per_block;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < chunks_per_block;
         i += (long long)gridDim.x * blockDim.x) {
        const uint4 a = ks[i];
        const uint4 b = vs[i];
        kd[i] = a;
        vd[i] = b;
    }
}

// ---------------------------------------------------------------------------
// Gather: blockIdx.x = logical block, blockIdx.y = sequence.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gather_kv_kernel(uint4* __restrict__ k_out, uint4* __restrict__ v_out,
                                                        const uint4* __restrict__ k_cache,
                                                        const uint4* __restrict__ v_cache,
                                                        const int32_t* __restrict__ block_tables, int max_blocks,
                                                        const int32_t* __restrict__ seq_lens,
                                                        const int64_t* __restrict__ out_offsets, int num_blocks,
                                                        int block_size, int num_kv_heads, int chunks_per_row,
                                                        int32_t* status) {
    pdl_wait();
    pdl_launch();
    const int b = blockIdx.y;
    const int L = seq_lens[b];
    if (L < 0 || (long long)L > (long long)max_blocks * block_size) {
        if (blockIdx.x == 0 && threadIdx.x == 0) report(status, PKV_STATUS_BAD_SEQLEN);
        return;
    }
    for (int lb = blockIdx.x; (long long)lb * block_size < L; lb += gridDim.x) {
        const int rows = min(block_size, L - lb * block_size);
        const int32_t blk = block_tables[(long long)b * max_blocks + lb];
        const bool ok = blk >= 0 && blk < num_blocks;
        if (!ok && threadIdx.x == 0) report(status, PKV_STATUS_BAD_BLOCK);
        const long long row0 = out_offsets[b] + (long long)lb * block_size;
        const int per_row = num_kv_heads * chunks_per_row;
        const int n = rows * per_row;
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const int r = i / per_row;
            const int rem = i - r * per_row;
            const int h = rem / chunks_per_row;
            const int c = rem - h * chunks_per_row;
            const long long dst = (row0 + r) * per_row + rem;
            if (!ok) {
                const uint4 nan = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
                k_out[dst] = nan;
                v_out[dst] = nan;
                continue;
            }
            const long long src = (((long long)blk * num_kv_heads + h) * block_size + r) * chunks_per_row + c;
            k_out[dst] = k_cache[src];
            v_out[dst] = v_cache[src];
        }
    }
}

}  // namespace pkv

using namespace pkv;

extern "C" int pkv_slot_mapping(int64_t* slots, const int32_t* block_tables, int max_blocks,
                                const int32_t* seq_lens, const int32_t* append_lens, int num_seqs,
                                int num_slots, int block_size, int num_blocks, int32_t* status,
                                void* stream) {
    if (num_seqs < 0 || num_slots < 0 || num_seqs > kSlotMaxSeqs || max_blocks < 1 || block_size < 1 ||
        num_blocks < 1)
        return PKV_ERR_SIZE;
    if (num_seqs == 0 || num_slots == 0) return PKV_OK;
    if (!slots || !block_tables || !seq_lens || !append_lens) return PKV_ERR_NULL;
    const int rc = host::check_device();
    if (rc) return rc;
    const size_t smem = sizeof(int) * (2 * (size_t)num_seqs + 1);
    if (smem > 48 * 1024) {
        if (cudaFuncSetAttribute(slot_mapping_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return PKV_ERR_CUDA;
    }
    const cudaError_t e = host::launch_pdl(slot_mapping_kernel, dim3(1), dim3(1024), smem, (cudaStream_t)stream,
                                           slots, block_tables, max_blocks, seq_lens, append_lens, num_seqs,
                                           num_slots, block_size, num_blocks, status);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_kv_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                             const int64_t* slots, int num_tokens, int num_blocks, int block_size,
                             int num_kv_heads, int head_dim, int32_t* status, void* stream) {
    if (num_tokens < 0 || num_blocks < 1 || block_size < 1 || num_kv_heads < 1 || head_dim < 8) return PKV_ERR_SIZE;
    if (head_dim % 8) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k_cache || !v_cache || !k_new || !v_new || !slots) return PKV_ERR_NULL;
    if (!host::aligned16(k_cache) || !host::aligned16(v_cache) || !host::aligned16(k_new) || !host::aligned16(v_new))
        return PKV_ERR_ALIGN;
    const int rc = host::check_device();
    if (rc) return rc;
    const int cpr = head_dim / 8;
    const long long total = (long long)num_tokens * num_kv_heads * cpr;
    const long long want = (total + 255) / 256;
    const int grid = (int)(want < host::sm_count() * 8LL ? want : host::sm_count() * 8LL);
    const cudaError_t e = host::launch_pdl(kv_append_kernel, dim3(grid), dim3(256), 0, (cudaStream_t)stream,
                                           (uint4*)k_cache, (uint4*)v_cache, (const uint4*)k_new,
                                           (const uint4*)v_new, slots, num_tokens, num_blocks, block_size,
                                           num_kv_heads, cpr, status);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_kv_append_paged(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                                   const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                                   const int32_t* append_lens, int num_seqs, int num_tokens, int num_blocks,
                                   int block_size, int num_kv_heads, int head_dim, int64_t* slots, int32_t* status,
                                   void* stream) {
    if (num_seqs < 0 || num_tokens < 0 || max_blocks < 1 || num_blocks < 1 || block_size < 1 || num_kv_heads < 1 ||
        head_dim < 8)
        return PKV_ERR_SIZE;
    if (head_dim % 8) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 || num_tokens == 0) return PKV_OK;
    if (!k_cache || !v_cache || !k_new || !v_new || !block_tables || !seq_lens || !append_lens || !slots)
        return PKV_ERR_NULL;
    if (!host::aligned16(k_cache) || !host::aligned16(v_cache) || !host::aligned16(k_new) || !host::aligned16(v_new))
        return PKV_ERR_ALIGN;
    if (num_seqs > kFusedMaxSeqs) {
        // larger batches: the two-kernel path
        const int rc = pkv_slot_mapping(slots, block_tables, max_blocks, seq_lens, append_lens, num_seqs, num_tokens,
                                        block_size, num_blocks, status, stream);
        if (rc) return rc;
        return pkv_kv_append(k_cache, v_cache, k_new, v_new, slots, num_tokens, num_blocks, block_size, num_kv_heads,
                             head_dim, status, stream);
    }
    const int rc = host::check_device();
    if (rc) return rc;
    const int cpr = head_dim / 8;
    const long long total = (long long)num_tokens * num_kv_heads * cpr;
    const long long want = (total + 1023) / 1024;
    const int grid = (int)(want < host::sm_count() * 2LL ? want : host::sm_count() * 2LL);
    const cudaError_t e = host::launch_pdl(kv_append_paged_kernel, dim3(grid), dim3(1024), 0, (cudaStream_t)stream,
                                           (uint4*)k_cache, (uint4*)v_cache, (const uint4*)k_new,
                                           (const uint4*)v_new, block_tables, max_blocks, seq_lens, append_lens,
                                           num_seqs, num_tokens, num_blocks, block_size, num_kv_heads, cpr, slots,
                                           status);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_kv_append_fp8(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                                 const int64_t* slots, const float* k_scale, const float* v_scale, int num_tokens,
                                 int num_blocks, int block_size, int num_kv_heads, int head_dim, int32_t* status,
                                 void* stream) {
    if (num_tokens < 0 || num_blocks < 1 || block_size < 1 || num_kv_heads < 1 || head_dim < 8) return PKV_ERR_SIZE;
    if (head_dim % 8) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k_cache || !v_cache || !k_new || !v_new || !slots || !k_scale || !v_scale) return PKV_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(k_cache) & 7) || (reinterpret_cast<uintptr_t>(v_cache) & 7) ||
        !host::aligned16(k_new) || !host::aligned16(v_new))
        return PKV_ERR_ALIGN;
    const int rc = host::check_device();
    if (rc) return rc;
    const int cpr = head_dim / 8;
    const long long total = (long long)num_tokens * num_kv_heads * cpr;
    const long long want = (total + 255) / 256;
    const int grid = (int)(want < host::sm_count() * 8LL ? want : host::sm_count() * 8LL);
    const cudaError_t e = host::launch_pdl(kv_append_fp8_kernel, dim3(grid), dim3(256), 0, (cudaStream_t)stream,
                                           (uint2*)k_cache, (uint2*)v_cache, (const uint4*)k_new,
                                           (const uint4*)v_new, slots, k_scale, v_scale, num_tokens, num_blocks,
                                           block_size, num_kv_heads, cpr, status);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_dst, int num_pairs,
                               int num_blocks, int block_size, int num_kv_heads, int head_dim,
                               int32_t* status, void* stream) {
    if (num_pairs < 0 || num_pairs > 65535 || num_blocks < 1 || block_size < 1 || num_kv_heads < 1 ||
        head_dim < 8)
        return PKV_ERR_SIZE;
    if (head_dim % 8) return PKV_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !src_dst) return PKV_ERR_NULL;
    if (!host::aligned16(k_cache) || !host::aligned16(v_cache)) return PKV_ERR_ALIGN;
    const int rc = host::check_device();
    if (rc) return rc;
    const long long cpb = (long long)num_kv_heads * block_size * head_dim / 8;
    long long gx = (cpb + 255) / 256;
    const long long cap = (host::sm_count() * 8LL + num_pairs - 1) / num_pairs;
    if (gx > cap) gx = cap;
    if (gx < 1) gx = 1;
    dim3 grid((unsigned)gx, (unsigned)num_pairs);
    const cudaError_t e = host::launch_pdl(copy_blocks_kernel, grid, dim3(256), 0, (cudaStream_t)stream,
                                           (uint4*)k_cache, (uint4*)v_cache, src_dst, num_blocks, cpb, status);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_gather_kv(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                             const int64_t* out_offsets, int num_seqs, int num_blocks, int block_size,
                             int num_kv_heads, int head_dim, int32_t* status, void* stream) {
    if (num_seqs < 0 || num_seqs > 65535 || max_blocks < 1 || num_blocks < 1 || block_size < 1 ||
        num_kv_heads < 1 || head_dim < 8)
        return PKV_ERR_SIZE;
    if (head_dim % 8) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!k_out || !v_out || !k_cache || !v_cache || !block_tables || !seq_lens || !out_offsets) return PKV_ERR_NULL;
    if (!host::aligned16(k_out) || !host::aligned16(v_out) || !host::aligned16(k_cache) || !host::aligned16(v_cache))
        return PKV_ERR_ALIGN;
    const int rc = host::check_device();
    if (rc) return rc;
    const int gx = max_blocks < 1024 ? max_blocks : 1024;
    dim3 grid(gx, num_seqs);
    const cudaError_t e = host::launch_pdl(gather_kv_kernel, grid, dim3(256), 0, (cudaStream_t)stream,
                                           (uint4*)k_out, (uint4*)v_out, (const uint4*)k_cache,
                                           (const uint4*)v_cache, block_tables, max_blocks, seq_lens, out_offsets,
                                           num_blocks, block_size, num_kv_heads, head_dim / 8, status);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_kv_append_fp8_ex(void* k_cache, void* v_cache, float* k_scale, float* v_scale, const void* k_new,
                                    const void* v_new, const int64_t* slots, int num_tokens, int num_blocks,
                                    int block_size, int num_kv_heads, int head_dim, int kv_format, int scale_mode,
                                    int32_t* status, void* stream) {
    if (num_tokens < 0 || num_blocks < 1 || block_size < 1 || num_kv_heads < 1 || head_dim < 8) return PKV_ERR_SIZE;
    if (kv_format != PKV_FP8_E4M3 && kv_format != PKV_FP8_E5M2) return PKV_ERR_UNSUPPORTED;
    if (scale_mode != PKV_FP8_SCALE_PER_HEAD && scale_mode != PKV_FP8_SCALE_PER_BLOCK) return PKV_ERR_UNSUPPORTED;
    if (head_dim % 8) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k_cache || !v_cache || !k_new || !v_new || !slots || !k_scale || !v_scale) return PKV_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(k_cache) & 7) || (reinterpret_cast<uintptr_t>(v_cache) & 7) ||
        !host::aligned16(k_new) || !host::aligned16(v_new))
        return PKV_ERR_ALIGN;
    const int rc = host::check_device();
    if (rc) return rc;
    const int cpr = head_dim / 8;
    cudaStream_t st = (cudaStream_t)stream;
    const bool pb = scale_mode == PKV_FP8_SCALE_PER_BLOCK;
    if (pb) {
        const long long warps = (long long)num_tokens * num_kv_heads;
        const long long want = (warps + 7) / 8;
        const int grid = (int)(want < host::sm_count() * 8LL ? want : host::sm_count() * 8LL);
        if (host::launch_pdl(fp8_open_blocks_kernel, dim3(grid), dim3(256), 0, st, (const uint4*)k_new,
                             (const uint4*)v_new, slots, k_scale, v_scale, num_tokens, num_blocks, block_size,
                             num_kv_heads, cpr, kv_format) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    const long long total = (long long)num_tokens * num_kv_heads * cpr;
    const long long want = (total + 255) / 256;
    const int grid = (int)(want < host::sm_count() * 8LL ? want : host::sm_count() * 8LL);
    const cudaError_t e = host::launch_pdl(kv_append_fp8_ex_kernel, dim3(grid), dim3(256), 0, st, (uint2*)k_cache,
                                           (uint2*)v_cache, (const uint4*)k_new, (const uint4*)v_new, slots,
                                           (const float*)k_scale, (const float*)v_scale, num_tokens, num_blocks,
                                           block_size, num_kv_heads, cpr, kv_format, pb ? 1 : 0, status);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_copy_blocks_fp8_ex(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                                      const int32_t* src_dst, int num_pairs, int num_blocks, int block_size,
                                      int num_kv_heads, int head_dim, int scale_mode, int32_t* status, void* stream) {
    if (scale_mode != PKV_FP8_SCALE_PER_HEAD && scale_mode != PKV_FP8_SCALE_PER_BLOCK) return PKV_ERR_UNSUPPORTED;
    if (scale_mode == PKV_FP8_SCALE_PER_BLOCK && num_pairs > 0 && (!k_scale || !v_scale)) return PKV_ERR_NULL;
    const int rc = pkv_copy_blocks_fp8(k_cache, v_cache, src_dst, num_pairs, num_blocks, block_size, num_kv_heads,
                                       head_dim, status, stream);
    if (rc || scale_mode != PKV_FP8_SCALE_PER_BLOCK || num_pairs == 0) return rc;
    const long long n = (long long)num_pairs * num_kv_heads;
    const int grid = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    const cudaError_t e = host::launch_pdl(copy_block_scales_kernel, dim3(grid), dim3(256), 0, (cudaStream_t)stream,
                                           k_scale, v_scale, src_dst, num_pairs, num_blocks, num_kv_heads);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_copy_blocks_fp8(void* k_cache, void* v_cache, const int32_t* src_dst, int num_pairs,
                                   int num_blocks, int block_size, int num_kv_heads, int head_dim, int32_t* status,
                                   void* stream) {
    // a block of 1-byte values is a block of 2-byte values of half the head_dim
    if (head_dim % 16) return PKV_ERR_UNSUPPORTED;
    return pkv_copy_blocks(k_cache, v_cache, src_dst, num_pairs, num_blocks, block_size, num_kv_heads, head_dim / 2,
                           status, stream);
}
