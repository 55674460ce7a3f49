/*
 * pkv_oracle.c -- plain, slow, fp64 CPU oracle for paged-KV decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this library.  The product
 * path (the CUDA library and its Python binding) never calls it, and this file
 * shares no code, header, table or helper with the CUDA sources.
 *
 * Every function below is the plain definition of one step of the path, written
 * out with loops and no blocking, fusion or reordering beyond what the
 * definition states.  Floating point is fp64 throughout; bf16 inputs are
 * widened exactly (a bf16 bit pattern is the top half of an IEEE fp32).
 *
 * Sources (web pages the method is taken from):
 *   [KVC]  "Inference at Scale: KV Cache, Prefill, and Decode"
 *          (blog.truongducdung.dev), sections 02, 03, 05, 07, 08.
 *   [SE]   "Chapter 31 Serving Efficiency" (imbrooklyn.dev), 31.3, 31.4
 *          (Example 31.2), 31.5.
 *   [SI]   "Spending the Idle" (derivingsystems.com), 12.4.
 *   ([SE] 31.5 with Example 31.3 for the rejection-sampling acceptance.)
 *
 * Cache layout (a choice; the pages only say K/V are read through the block
 * table): k_cache, v_cache are [num_blocks][num_kv_heads][block_size][head_dim]
 * bf16.  Logical token t of a sequence lives in physical block
 * block_tables[b][t / block_size] at row t % block_size ([KVC] 05, "The block
 * table").
 *
 * Status bits returned (same meaning as the CUDA library's, defined here
 * independently):
 *   1  a block id outside [0, num_blocks) was needed
 *   2  a seq_len outside [0, max_blocks * block_size]
 *   4  a q_len outside [0, seq_len]
 *   8  a slot outside [-1.., num_blocks * block_size)  (negative = skip)
 *   64 a copy pair outside [0, num_blocks)
 *   128 a draft token outside [0, vocab)
 *   256 a sampling distribution with no positive weight
 * Output rows affected by bits 1, 2 or 4 are written as NaN.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ST_BAD_BLOCK 1
#define ST_BAD_SEQLEN 2
#define ST_BAD_QLEN 4
#define ST_BAD_SLOT 8
#define ST_BAD_PAIR 64

static double widen_bf16(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Offset (in elements) of row `row` of kv head `head` in physical block `blk`. */
static int64_t cache_offset(int64_t blk, int head, int row, int n_kv, int bs, int d) {
    return ((blk * n_kv + head) * (int64_t)bs + row) * (int64_t)d;
}

/*
 * Slot mapping ([KVC] 05 "The block table"): the new tokens of sequence b are
 * its last append_lens[b] positions; position pos goes to
 * slot = block_tables[b][pos / bs] * bs + pos % bs.  Output is packed in
 * sequence order.  Returns status bits.
 */
int oracle_slot_mapping(int64_t *slots, const int32_t *block_tables, int max_blocks,
                        const int32_t *seq_lens, const int32_t *append_lens, int num_seqs,
                        int block_size, int num_blocks) {
    int status = 0;
    int64_t o = 0;
    for (int b = 0; b < num_seqs; b++) {
        int L = seq_lens[b], A = append_lens[b];
        int bad = 0;
        if (L < 0 || (int64_t)L > (int64_t)max_blocks * block_size) { status |= ST_BAD_SEQLEN; bad = 1; }
        if (A < 0 || A > L) { status |= ST_BAD_QLEN; bad = 1; }
        if (A < 0) continue;
        for (int i = 0; i < A; i++, o++) {
            if (bad) { slots[o] = -1; continue; }
            int pos = L - A + i;
            int32_t blk = block_tables[(int64_t)b * max_blocks + pos / block_size];
            if (blk < 0 || blk >= num_blocks) { status |= ST_BAD_BLOCK; slots[o] = -1; continue; }
            slots[o] = (int64_t)blk * block_size + pos % block_size;
        }
    }
    return status;
}

/*
 * KV append ([KVC] 02 "The two phases of a request": a decode step appends one
 * K/V row per new token).  k_new/v_new are [num_tokens][n_kv][d].  A negative
 * slot means "skip"; a slot past the pool is an error and is skipped.
 */
int oracle_kv_append(uint16_t *k_cache, uint16_t *v_cache, const uint16_t *k_new,
                     const uint16_t *v_new, const int64_t *slots, int num_tokens,
                     int num_blocks, int block_size, int n_kv, int d) {
    int status = 0;
    for (int t = 0; t < num_tokens; t++) {
        int64_t s = slots[t];
        if (s < 0) continue;
        if (s >= (int64_t)num_blocks * block_size) { status |= ST_BAD_SLOT; continue; }
        int64_t blk = s / block_size;
        int row = (int)(s % block_size);
        for (int h = 0; h < n_kv; h++) {
            for (int c = 0; c < d; c++) {
                int64_t dst = cache_offset(blk, h, row, n_kv, block_size, d) + c;
                int64_t src = ((int64_t)t * n_kv + h) * d + c;
                k_cache[dst] = k_new[src];
                v_cache[dst] = v_new[src];
            }
        }
    }
    return status;
}

/*
 * Copy-on-write block copy ([SE] 31.3: share blocks, copy a block when a
 * branch appends; [KVC] 05 "Block sharing and copy-on-write").  src_dst is
 * [n][2]; every byte of K and V of block src is copied to block dst, pairs in
 * order.
 */
int oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, const int32_t *src_dst, int n,
                       int num_blocks, int block_size, int n_kv, int d) {
    int status = 0;
    int64_t per_block = (int64_t)n_kv * block_size * d;
    for (int i = 0; i < n; i++) {
        int32_t s = src_dst[2 * i], t = src_dst[2 * i + 1];
        if (s < 0 || s >= num_blocks || t < 0 || t >= num_blocks) { status |= ST_BAD_PAIR; continue; }
        for (int64_t e = 0; e < per_block; e++) {
            k_cache[(int64_t)t * per_block + e] = k_cache[(int64_t)s * per_block + e];
            v_cache[(int64_t)t * per_block + e] = v_cache[(int64_t)s * per_block + e];
        }
    }
    return status;
}

/*
 * Block-table gather ([KVC] 05 "The block table"): the K/V of each sequence,
 * read through its block table, laid out contiguously as
 * [sum seq_len][n_kv][d] in sequence order.
 */
int oracle_gather_kv(uint16_t *k_out, uint16_t *v_out, const uint16_t *k_cache,
                     const uint16_t *v_cache, const int32_t *block_tables, int max_blocks,
                     const int32_t *seq_lens, int num_seqs, int num_blocks, int block_size,
                     int n_kv, int d) {
    int status = 0;
    int64_t o = 0;
    for (int b = 0; b < num_seqs; b++) {
        int L = seq_lens[b];
        if (L < 0 || (int64_t)L > (int64_t)max_blocks * block_size) { status |= ST_BAD_SEQLEN; continue; }
        for (int t = 0; t < L; t++, o++) {
            int32_t blk = block_tables[(int64_t)b * max_blocks + t / block_size];
            for (int h = 0; h < n_kv; h++) {
                for (int c = 0; c < d; c++) {
                    int64_t dst = (o * n_kv + h) * d + c;
                    if (blk < 0 || blk >= num_blocks) {
                        k_out[dst] = 0x7fc0;  /* bf16 quiet NaN */
                        v_out[dst] = 0x7fc0;
                        status |= ST_BAD_BLOCK;
                        continue;
                    }
                    int64_t src = cache_offset(blk, h, t % block_size, n_kv, block_size, d) + c;
                    k_out[dst] = k_cache[src];
                    v_out[dst] = v_cache[src];
                }
            }
        }
    }
    return status;
}

/* Shared validation of one sequence for the attention functions. */
static int check_seq(int L, int ql, int max_blocks, int block_size) {
    int st = 0;
    if (L < 0 || (int64_t)L > (int64_t)max_blocks * block_size) st |= ST_BAD_SEQLEN;
    if (ql < 0 || ql > L) st |= ST_BAD_QLEN;
    return st;
}

/*
 * Softmax attention over K/V gathered through the block table -- the plain
 * definition that paged, online and split attention all reach exactly
 * ([KVC] 07 "Online softmax": the same computation with a different order of
 * additions; [SE] 31.4).
 *
 * For sequence b with seq_len L and q_len ql, query i (0 <= i < ql) sits at
 * position p = L - ql + i and sees positions 0..p (causal within the new
 * tokens, [KVC] 08: the verify pass is like a short prefill).  Query head h
 * uses kv head h / g, g = n_q / n_kv ([KVC] 04 "GQA").
 *   s_t = scale * <q, K_t>,  M = max_t s_t,  w_t = exp(s_t - M),
 *   o   = sum_t w_t V_t / sum_t w_t.
 * q is [sum ql][n_q][d]; out is [sum ql][n_q][d] fp64.
 */
int oracle_attention(double *out, const uint16_t *q, const uint16_t *k_cache,
                     const uint16_t *v_cache, const int32_t *block_tables, int max_blocks,
                     const int32_t *seq_lens, const int32_t *q_lens, int num_seqs, int n_q,
                     int n_kv, int d, int block_size, int num_blocks, double scale) {
    int status = 0;
    int g = n_q / n_kv;
    int64_t *row0 = (int64_t *)malloc(sizeof(int64_t) * (num_seqs + 1));
    row0[0] = 0;
    for (int b = 0; b < num_seqs; b++) row0[b + 1] = row0[b] + (q_lens[b] > 0 ? q_lens[b] : 0);
    for (int b = 0; b < num_seqs; b++) status |= check_seq(seq_lens[b], q_lens[b], max_blocks, block_size);

#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
    for (int b = 0; b < num_seqs; b++) {
        int L = seq_lens[b], ql = q_lens[b];
        if (ql <= 0) continue;
        int seq_bad = check_seq(L, ql, max_blocks, block_size);
        double *s = (double *)malloc(sizeof(double) * (L > 0 ? L : 1));
        for (int i = 0; i < ql; i++) {
            int64_t r = row0[b] + i;
            int p = L - ql + i;
            for (int h = 0; h < n_q; h++) {
                double *o = out + (r * n_q + h) * d;
                const uint16_t *qv = q + (r * n_q + h) * d;
                int j = h / g;
                int bad = seq_bad;
                for (int t = 0; t <= p && !bad; t++) {
                    int32_t blk = block_tables[(int64_t)b * max_blocks + t / block_size];
                    if (blk < 0 || blk >= num_blocks) { bad = 1; status |= ST_BAD_BLOCK; }
                }
                if (bad) {
                    for (int c = 0; c < d; c++) o[c] = NAN;
                    continue;
                }
                /* scores */
                for (int t = 0; t <= p; t++) {
                    int32_t blk = block_tables[(int64_t)b * max_blocks + t / block_size];
                    const uint16_t *kt = k_cache + cache_offset(blk, j, t % block_size, n_kv, block_size, d);
                    double acc = 0.0;
                    for (int c = 0; c < d; c++) acc += widen_bf16(qv[c]) * widen_bf16(kt[c]);
                    s[t] = scale * acc;
                }
                double M = -INFINITY;
                for (int t = 0; t <= p; t++) if (s[t] > M) M = s[t];
                double den = 0.0;
                for (int t = 0; t <= p; t++) { s[t] = exp(s[t] - M); den += s[t]; }
                for (int c = 0; c < d; c++) o[c] = 0.0;
                for (int t = 0; t <= p; t++) {
                    int32_t blk = block_tables[(int64_t)b * max_blocks + t / block_size];
                    const uint16_t *vt = v_cache + cache_offset(blk, j, t % block_size, n_kv, block_size, d);
                    for (int c = 0; c < d; c++) o[c] += s[t] * widen_bf16(vt[c]);
                }
                for (int c = 0; c < d; c++) o[c] /= den;
            }
        }
        free(s);
    }
    free(row0);
    return status;
}

/*
 * Split-KV attention with a log-sum-exp merge, in the order Flash-Decoding
 * describes it ([KVC] 07 "FlashAttention-2, FlashAttention-3, and
 * Flash-Decoding"): the visible positions of each query are cut into
 * partitions [k*P, (k+1)*P); each partition yields a partial result
 * (running max m_k, sum l_k = sum exp(s - m_k), normalised output o_k); the
 * partials are merged with the online-softmax rescaling:
 *   M = max_k m_k,  l = sum_k l_k exp(m_k - M),
 *   o = sum_k o_k l_k exp(m_k - M) / l.
 * A partition with no visible position has m = -inf, l = 0 and weight 0
 * ([SE] Example 31.2: combine tile statistics, not tile averages).
 *
 * part_o / part_m / part_l (may be NULL) receive the partials for every
 * (row, head, partition) as [sum ql][n_q][nparts_max](*d), where
 * nparts_max = ceil(max over sequences of seq_len / P); unused entries are
 * set to o = 0, m = -inf, l = 0.
 */
int oracle_attention_split(double *out, double *part_o, double *part_m, double *part_l,
                           int nparts_max, const uint16_t *q, const uint16_t *k_cache,
                           const uint16_t *v_cache, const int32_t *block_tables, int max_blocks,
                           const int32_t *seq_lens, const int32_t *q_lens, int num_seqs, int n_q,
                           int n_kv, int d, int block_size, int num_blocks, double scale,
                           int partition_tokens) {
    int status = 0;
    int g = n_q / n_kv;
    int P = partition_tokens;
    int64_t *row0 = (int64_t *)malloc(sizeof(int64_t) * (num_seqs + 1));
    row0[0] = 0;
    for (int b = 0; b < num_seqs; b++) row0[b + 1] = row0[b] + (q_lens[b] > 0 ? q_lens[b] : 0);
    for (int b = 0; b < num_seqs; b++) status |= check_seq(seq_lens[b], q_lens[b], max_blocks, block_size);

#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
    for (int b = 0; b < num_seqs; b++) {
        int L = seq_lens[b], ql = q_lens[b];
        if (ql <= 0) continue;
        int seq_bad = check_seq(L, ql, max_blocks, block_size);
        double *po = (double *)malloc(sizeof(double) * (size_t)nparts_max * d);
        double *pm = (double *)malloc(sizeof(double) * (size_t)nparts_max);
        double *pl = (double *)malloc(sizeof(double) * (size_t)nparts_max);
        for (int i = 0; i < ql; i++) {
            int64_t r = row0[b] + i;
            int p = L - ql + i; /* last visible position */
            for (int h = 0; h < n_q; h++) {
                double *o = out + (r * n_q + h) * d;
                const uint16_t *qv = q + (r * n_q + h) * d;
                int j = h / g;
                int bad = seq_bad;
                for (int t = 0; t <= p && !bad; t++) {
                    int32_t blk = block_tables[(int64_t)b * max_blocks + t / block_size];
                    if (blk < 0 || blk >= num_blocks) { bad = 1; status |= ST_BAD_BLOCK; }
                }
                for (int k = 0; k < nparts_max; k++) {
                    pm[k] = -INFINITY;
                    pl[k] = 0.0;
                    for (int c = 0; c < d; c++) po[(size_t)k * d + c] = 0.0;
                }
                if (!bad) {
                    /* one partial per partition */
                    for (int k = 0; k < nparts_max; k++) {
                        int lo = k * P, hi = (k + 1) * P - 1;
                        if (hi > p) hi = p;
                        if (lo > hi) continue; /* nothing visible: m=-inf, l=0 */
                        double m = -INFINITY;
                        for (int t = lo; t <= hi; t++) {
                            int32_t blk = block_tables[(int64_t)b * max_blocks + t / block_size];
                            const uint16_t *kt = k_cache + cache_offset(blk, j, t % block_size, n_kv, block_size, d);
                            double acc = 0.0;
                            for (int c = 0; c < d; c++) acc += widen_bf16(qv[c]) * widen_bf16(kt[c]);
                            double st = scale * acc;
                            if (st > m) m = st;
                        }
                        double l = 0.0;
                        double *ok = po + (size_t)k * d;
                        for (int t = lo; t <= hi; t++) {
                            int32_t blk = block_tables[(int64_t)b * max_blocks + t / block_size];
                            const uint16_t *kt = k_cache + cache_offset(blk, j, t % block_size, n_kv, block_size, d);
                            const uint16_t *vt = v_cache + cache_offset(blk, j, t % block_size, n_kv, block_size, d);
                            double acc = 0.0;
                            for (int c = 0; c < d; c++) acc += widen_bf16(qv[c]) * widen_bf16(kt[c]);
                            double w = exp(scale * acc - m);
                            l += w;
                            for (int c = 0; c < d; c++) ok[c] += w * widen_bf16(vt[c]);
                        }
                        for (int c = 0; c < d; c++) ok[c] /= l;
                        pm[k] = m;
                        pl[k] = l;
                    }
                    /* merge */
                    double M = -INFINITY;
                    for (int k = 0; k < nparts_max; k++) if (pm[k] > M) M = pm[k];
                    double lsum = 0.0;
                    for (int c = 0; c < d; c++) o[c] = 0.0;
                    for (int k = 0; k < nparts_max; k++) {
                        if (pm[k] == -INFINITY) continue; /* empty partition, weight 0 */
                        double wk = pl[k] * exp(pm[k] - M);
                        lsum += wk;
                        for (int c = 0; c < d; c++) o[c] += po[(size_t)k * d + c] * wk;
                    }
                    for (int c = 0; c < d; c++) o[c] /= lsum;
                } else {
                    for (int c = 0; c < d; c++) o[c] = NAN;
                }
                if (part_o) {
                    for (int k = 0; k < nparts_max; k++) {
                        size_t idx = ((size_t)r * n_q + h) * nparts_max + k;
                        part_m[idx] = pm[k];
                        part_l[idx] = pl[k];
                        for (int c = 0; c < d; c++) part_o[idx * d + c] = po[(size_t)k * d + c];
                    }
                }
            }
        }
        free(po);
        free(pm);
        free(pl);
    }
    free(row0);
    return status;
}

/*
 * "a beats b" for the argmax: NaN is greater than every number and the first
 * index wins among equal values (numpy/torch argmax convention).
 */
static int beats(float a, int64_t ia, float b, int64_t ib) {
    int an = isnan(a), bn = isnan(b);
    if (an != bn) return an;
    if (!an && a != b) return a > b;
    return ia < ib;
}

/*
 * Greedy speculative acceptance ([SI] 12.4: accept the drafts that match what
 * the model would pick and stop at the first that does not; [KVC] 08: with
 * greedy decoding accept a draft token if it matches the target's argmax, and
 * always add one target token).
 *   logits [B][k+1][V] fp32, draft [B][k] int32.
 *   argmax[b][j]  = first index of the maximum of row (b, j)   (j = 0..k)
 *   accepted[b]   = number of leading j < k with draft[b][j] == argmax[b][j]
 *   next_token[b] = argmax[b][accepted[b]]   (the correction or bonus token)
 * argmax may be NULL.
 */
int oracle_spec_accept_greedy(int32_t *accepted, int32_t *next_token, int32_t *argmax,
                              const float *logits, const int32_t *draft, int B, int k, int V) {
    for (int b = 0; b < B; b++) {
        int32_t *rowmax = (int32_t *)malloc(sizeof(int32_t) * (k + 1));
        for (int j = 0; j <= k; j++) {
            const float *row = logits + ((int64_t)b * (k + 1) + j) * V;
            int64_t best = 0;
            for (int64_t v = 1; v < V; v++)
                if (beats(row[v], v, row[best], best)) best = v;
            rowmax[j] = (int32_t)best;
            if (argmax) argmax[b * (k + 1) + j] = (int32_t)best;
        }
        int a = 0;
        while (a < k && draft[b * k + a] == rowmax[a]) a++;
        accepted[b] = a;
        next_token[b] = rowmax[a];
        free(rowmax);
    }
    return 0;
}

/*
 * FP8 KV cache ([KVC] 03 "KV cache quantization": store K and V in FP8,
 * 1 byte per value, formats e4m3 and e5m2; this library takes e4m3).
 *
 * e4m3 (the "fn" variant: no infinities): sign bit, 4 exponent bits with bias
 * 7, 3 mantissa bits; exponent field 0 holds subnormals m * 2^-9; code
 * S.1111.111 is NaN; the largest finite magnitude is 1.75 * 2^8 = 448.
 * Encoding rounds to the nearest representable value, ties to the even code,
 * and saturates magnitudes above 448 to 448; NaN stays NaN (0x7f).
 *
 * Scales (a reading: the pages fix none): one fp32 dequantisation scale per kv
 * head for K and one for V, supplied by the caller.  Appending a bf16 row
 * stores e4m3(x * (1 / scale)), with 1 / scale and the product each rounded
 * to fp32 (round to nearest even); reading decodes e4m3 and multiplies by the
 * scale (exactly, in fp64 here).
 */
static double e4m3_value(uint8_t c) {
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return s ? -v : v;
}

static uint8_t e4m3_encode(float x) {
    if (isnan(x)) return 0x7f;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7e;
    /* largest finite code whose magnitude is <= a (magnitudes grow with the code) */
    int c = 0;
    while (c < 0x7e && e4m3_value((uint8_t)(c + 1)) <= a) c++;
    if (c < 0x7e) {
        const double lo = e4m3_value((uint8_t)c), hi = e4m3_value((uint8_t)(c + 1));
        if (a - lo > hi - a || (a - lo == hi - a && (c & 1))) c++;
    }
    return sign | (uint8_t)c;
}

int oracle_e4m3_encode(uint8_t *out, const float *in, int64_t n) {
    for (int64_t i = 0; i < n; i++) out[i] = e4m3_encode(in[i]);
    return 0;
}

int oracle_e4m3_decode(double *out, const uint8_t *in, int64_t n) {
    for (int64_t i = 0; i < n; i++) out[i] = e4m3_value(in[i]);
    return 0;
}

/* KV append into an e4m3 pool: as oracle_kv_append, each value quantised. */
int oracle_kv_append_fp8(uint8_t *k_cache, uint8_t *v_cache, const uint16_t *k_new, const uint16_t *v_new,
                         const int64_t *slots, int num_tokens, int num_blocks, int block_size, int n_kv, int d,
                         const float *k_scale, const float *v_scale) {
    int status = 0;
    for (int t = 0; t < num_tokens; t++) {
        int64_t s = slots[t];
        if (s < 0) continue;
        if (s >= (int64_t)num_blocks * block_size) { status |= ST_BAD_SLOT; continue; }
        int64_t blk = s / block_size;
        int row = (int)(s % block_size);
        for (int h = 0; h < n_kv; h++) {
            const float ik = 1.0f / k_scale[h], iv = 1.0f / v_scale[h];
            for (int c = 0; c < d; c++) {
                int64_t dst = cache_offset(blk, h, row, n_kv, block_size, d) + c;
                int64_t src = ((int64_t)t * n_kv + h) * d + c;
                const float xk = (float)widen_bf16(k_new[src]) * ik;
                const float xv = (float)widen_bf16(v_new[src]) * iv;
                k_cache[dst] = e4m3_encode(xk);
                v_cache[dst] = e4m3_encode(xv);
            }
        }
    }
    return status;
}

/*
 * The second FP8 format of [KVC] 03, e5m2: sign bit, 5 exponent bits with bias
 * 15, 2 mantissa bits; exponent field 0 holds subnormals m * 2^-16; field 31
 * holds the infinities (m = 0) and NaN (m != 0); the largest finite magnitude
 * is 1.75 * 2^15 = 57344.  Encoding rounds to the nearest representable value,
 * ties to the even code, and saturates magnitudes above 57344 (infinities
 * included) to 57344; NaN is stored as 0x7f.
 */
static double e5m2_value(uint8_t c) {
    const int s = c >> 7, e = (c >> 2) & 31, m = c & 3;
    double v;
    if (e == 31) v = m ? NAN : INFINITY;
    else v = e == 0 ? ldexp((double)m, -16) : ldexp((double)(4 + m), e - 17);
    return s ? -v : v;
}

static uint8_t e5m2_encode(float x) {
    if (isnan(x)) return 0x7f;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 57344.0) return sign | 0x7b;
    int c = 0;
    while (c < 0x7b && e5m2_value((uint8_t)(c + 1)) <= a) c++;
    if (c < 0x7b) {
        const double lo = e5m2_value((uint8_t)c), hi = e5m2_value((uint8_t)(c + 1));
        if (a - lo > hi - a || (a - lo == hi - a && (c & 1))) c++;
    }
    return sign | (uint8_t)c;
}

/* fmt 0 = e4m3, 1 = e5m2 */
static double fp8_value(uint8_t c, int fmt) { return fmt ? e5m2_value(c) : e4m3_value(c); }
static uint8_t fp8_encode(float x, int fmt) { return fmt ? e5m2_encode(x) : e4m3_encode(x); }

int oracle_fp8_encode(uint8_t *out, const float *in, int64_t n, int fmt) {
    for (int64_t i = 0; i < n; i++) out[i] = fp8_encode(in[i], fmt);
    return 0;
}

int oracle_fp8_decode(double *out, const uint8_t *in, int64_t n, int fmt) {
    for (int64_t i = 0; i < n; i++) out[i] = fp8_value(in[i], fmt);
    return 0;
}

/*
 * Scale of one (block, kv head) tile of an FP8 pool with per-block scales (a
 * reading: [KVC] 03 fixes no scaling).  It is set when the block is opened --
 * by the append that writes the block's row 0 -- from that row's values x of
 * the head: the smallest power of two s = 2^e (e in [-120, 120]) with
 *   amax <= s * FMAX / 2,   amax = max |x| over the row's non-NaN values,
 * FMAX the format's largest finite value (448 for e4m3, 57344 for e5m2).  The
 * opening row then uses at most half of the format's range, and the rows
 * appended after it may grow to twice its magnitude before they saturate.
 * s = 1 when amax is 0 (or every value is NaN) or infinite.  A power of two
 * makes 1 / s and x * (1 / s) exact in fp32.
 */
float oracle_block_scale(const float *row, int d, int fmt) {
    double amax = 0.0;
    for (int c = 0; c < d; c++)
        if (!isnan(row[c]) && fabs((double)row[c]) > amax) amax = fabs((double)row[c]);
    if (amax == 0.0 || isinf(amax)) return 1.0f;
    const double half = fmt ? 28672.0 : 224.0;
    int e = -120;
    while (e < 120 && ldexp(half, e) < amax) e++;
    return (float)ldexp(1.0, e);
}

/*
 * KV append into an FP8 pool of either format.  per_block = 0: one scale per
 * kv head, k_scale[n_kv] (read only), as oracle_kv_append_fp8.  per_block = 1:
 * k_scale and v_scale are [num_blocks][n_kv]; first every appended token whose
 * slot is row 0 of its block sets that block's scales from its own row
 * (oracle_block_scale), then every token is stored with its block's scales --
 * so rows appended in the same call as their block's row 0 use the scale that
 * row set.  Each value x is stored as fp8(x * (1 / scale)), the reciprocal and
 * the product rounded to fp32.
 */
int oracle_kv_append_fp8_ex(uint8_t *k_cache, uint8_t *v_cache, float *k_scale, float *v_scale, const uint16_t *k_new,
                            const uint16_t *v_new, const int64_t *slots, int num_tokens, int num_blocks,
                            int block_size, int n_kv, int d, int fmt, int per_block) {
    int status = 0;
    float *row = (float *)malloc(sizeof(float) * (d > 0 ? d : 1));
    if (per_block) {
        for (int t = 0; t < num_tokens; t++) {
            int64_t s = slots[t];
            if (s < 0 || s >= (int64_t)num_blocks * block_size || s % block_size != 0) continue;
            int64_t blk = s / block_size;
            for (int h = 0; h < n_kv; h++) {
                for (int c = 0; c < d; c++) row[c] = (float)widen_bf16(k_new[((int64_t)t * n_kv + h) * d + c]);
                k_scale[blk * n_kv + h] = oracle_block_scale(row, d, fmt);
                for (int c = 0; c < d; c++) row[c] = (float)widen_bf16(v_new[((int64_t)t * n_kv + h) * d + c]);
                v_scale[blk * n_kv + h] = oracle_block_scale(row, d, fmt);
            }
        }
    }
    for (int t = 0; t < num_tokens; t++) {
        int64_t s = slots[t];
        if (s < 0) continue;
        if (s >= (int64_t)num_blocks * block_size) { status |= ST_BAD_SLOT; continue; }
        int64_t blk = s / block_size;
        int r = (int)(s % block_size);
        for (int h = 0; h < n_kv; h++) {
            const int64_t si = per_block ? blk * n_kv + h : h;
            const float ik = 1.0f / k_scale[si], iv = 1.0f / v_scale[si];
            for (int c = 0; c < d; c++) {
                int64_t dst = cache_offset(blk, h, r, n_kv, block_size, d) + c;
                int64_t src = ((int64_t)t * n_kv + h) * d + c;
                const float xk = (float)widen_bf16(k_new[src]) * ik;
                const float xv = (float)widen_bf16(v_new[src]) * iv;
                k_cache[dst] = fp8_encode(xk, fmt);
                v_cache[dst] = fp8_encode(xv, fmt);
            }
        }
    }
    free(row);
    return status;
}

/*
 * Copy-on-write block copy in an FP8 pool ([SE] 31.3; [KVC] 05): every byte of
 * K and V of block src to block dst, and with per-block scales the block's
 * scales too.  A pair outside the pool sets ST_BAD_PAIR and is skipped.
 */
int oracle_copy_blocks_fp8(uint8_t *k_cache, uint8_t *v_cache, float *k_scale, float *v_scale,
                           const int32_t *src_dst, int n, int num_blocks, int block_size, int n_kv, int d,
                           int per_block) {
    int status = 0;
    const int64_t blk_bytes = (int64_t)n_kv * block_size * d;
    for (int i = 0; i < n; i++) {
        int32_t sb = src_dst[2 * i], tb = src_dst[2 * i + 1];
        if (sb < 0 || sb >= num_blocks || tb < 0 || tb >= num_blocks) { status |= ST_BAD_PAIR; continue; }
        for (int64_t e = 0; e < blk_bytes; e++) {
            k_cache[(int64_t)tb * blk_bytes + e] = k_cache[(int64_t)sb * blk_bytes + e];
            v_cache[(int64_t)tb * blk_bytes + e] = v_cache[(int64_t)sb * blk_bytes + e];
        }
        if (per_block)
            for (int h = 0; h < n_kv; h++) {
                k_scale[(int64_t)tb * n_kv + h] = k_scale[(int64_t)sb * n_kv + h];
                v_scale[(int64_t)tb * n_kv + h] = v_scale[(int64_t)sb * n_kv + h];
            }
    }
    return status;
}

/*
 * Attention over an FP8 pool of either format and scale granularity:
 * oracle_attention with K_t = fp8(K) * k_scale and V_t = fp8(V) * v_scale,
 * the scale of kv head j (per_block = 0) or of the (block of t, j) tile
 * (per_block = 1).
 */
int oracle_attention_fp8_ex(double *out, const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                            const float *k_scale, const float *v_scale, const int32_t *block_tables, int max_blocks,
                            const int32_t *seq_lens, const int32_t *q_lens, int num_seqs, int n_q, int n_kv, int d,
                            int block_size, int num_blocks, double scale, int fmt, int per_block) {
    int status = 0;
    int g = n_q / n_kv;
    double val[256]; /* value of every code, looked up below */
    for (int c = 0; c < 256; c++) val[c] = fp8_value((uint8_t)c, fmt);
    int64_t *row0 = (int64_t *)malloc(sizeof(int64_t) * (num_seqs + 1));
    row0[0] = 0;
    for (int b = 0; b < num_seqs; b++) row0[b + 1] = row0[b] + (q_lens[b] > 0 ? q_lens[b] : 0);
    for (int b = 0; b < num_seqs; b++) status |= check_seq(seq_lens[b], q_lens[b], max_blocks, block_size);

#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
    for (int b = 0; b < num_seqs; b++) {
        int L = seq_lens[b], ql = q_lens[b];
        if (ql <= 0) continue;
        int seq_bad = check_seq(L, ql, max_blocks, block_size);
        double *s = (double *)malloc(sizeof(double) * (L > 0 ? L : 1));
        for (int i = 0; i < ql; i++) {
            int64_t r = row0[b] + i;
            int p = L - ql + i;
            for (int h = 0; h < n_q; h++) {
                double *o = out + (r * n_q + h) * d;
                const uint16_t *qv = q + (r * n_q + h) * d;
                int j = h / g;
                int bad = seq_bad;
                for (int t = 0; t <= p && !bad; t++) {
                    int32_t blk = block_tables[(int64_t)b * max_blocks + t / block_size];
                    if (blk < 0 || blk >= num_blocks) { bad = 1; status |= ST_BAD_BLOCK; }
                }
                if (bad) {
                    for (int c = 0; c < d; c++) o[c] = NAN;
                    continue;
                }
                for (int t = 0; t <= p; t++) {
                    int32_t blk = block_tables[(int64_t)b * max_blocks + t / block_size];
                    const uint8_t *kt = k_cache + cache_offset(blk, j, t % block_size, n_kv, block_size, d);
                    const double ks = per_block ? (double)k_scale[(int64_t)blk * n_kv + j] : (double)k_scale[j];
                    double acc = 0.0;
                    for (int c = 0; c < d; c++) acc += widen_bf16(qv[c]) * (val[kt[c]] * ks);
                    s[t] = scale * acc;
                }
                double M = -INFINITY;
                for (int t = 0; t <= p; t++) if (s[t] > M) M = s[t];
                double den = 0.0;
                for (int t = 0; t <= p; t++) { s[t] = exp(s[t] - M); den += s[t]; }
                for (int c = 0; c < d; c++) o[c] = 0.0;
                for (int t = 0; t <= p; t++) {
                    int32_t blk = block_tables[(int64_t)b * max_blocks + t / block_size];
                    const uint8_t *vt = v_cache + cache_offset(blk, j, t % block_size, n_kv, block_size, d);
                    const double vs = per_block ? (double)v_scale[(int64_t)blk * n_kv + j] : (double)v_scale[j];
                    for (int c = 0; c < d; c++) o[c] += s[t] * (val[vt[c]] * vs);
                }
                for (int c = 0; c < d; c++) o[c] /= den;
            }
        }
        free(s);
    }
    free(row0);
    return status;
}

/*
 * Attention over an e4m3 pool: oracle_attention with K_t = e4m3(K) * k_scale[j]
 * and V_t = e4m3(V) * v_scale[j] for kv head j.
 */
int oracle_attention_fp8(double *out, const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                         const float *k_scale, const float *v_scale, const int32_t *block_tables, int max_blocks,
                         const int32_t *seq_lens, const int32_t *q_lens, int num_seqs, int n_q, int n_kv, int d,
                         int block_size, int num_blocks, double scale) {
    int status = 0;
    int g = n_q / n_kv;
    double val[256]; /* e4m3_value of every code, looked up below */
    for (int c = 0; c < 256; c++) val[c] = e4m3_value((uint8_t)c);
    int64_t *row0 = (int64_t *)malloc(sizeof(int64_t) * (num_seqs + 1));
    row0[0] = 0;
    for (int b = 0; b < num_seqs; b++) row0[b + 1] = row0[b] + (q_lens[b] > 0 ? q_lens[b] : 0);
    for (int b = 0; b < num_seqs; b++) status |= check_seq(seq_lens[b], q_lens[b], max_blocks, block_size);

#pragma omp parallel for schedule(dynamic, 1) reduction(| : status)
    for (int b = 0; b < num_seqs; b++) {
        int L = seq_lens[b], ql = q_lens[b];
        if (ql <= 0) continue;
        int seq_bad = check_seq(L, ql, max_blocks, block_size);
        double *s = (double *)malloc(sizeof(double) * (L > 0 ? L : 1));
        for (int i = 0; i < ql; i++) {
            int64_t r = row0[b] + i;
            int p = L - ql + i;
            for (int h = 0; h < n_q; h++) {
                double *o = out + (r * n_q + h) * d;
                const uint16_t *qv = q + (r * n_q + h) * d;
                int j = h / g;
                int bad = seq_bad;
                for (int t = 0; t <= p && !bad; t++) {
                    int32_t blk = block_tables[(int64_t)b * max_blocks + t / block_size];
                    if (blk < 0 || blk >= num_blocks) { bad = 1; status |= ST_BAD_BLOCK; }
                }
                if (bad) {
                    for (int c = 0; c < d; c++) o[c] = NAN;
                    continue;
                }
                for (int t = 0; t <= p; t++) {
                    int32_t blk = block_tables[(int64_t)b * max_blocks + t / block_size];
                    const uint8_t *kt = k_cache + cache_offset(blk, j, t % block_size, n_kv, block_size, d);
                    double acc = 0.0;
                    for (int c = 0; c < d; c++) acc += widen_bf16(qv[c]) * (val[kt[c]] * (double)k_scale[j]);
                    s[t] = scale * acc;
                }
                double M = -INFINITY;
                for (int t = 0; t <= p; t++) if (s[t] > M) M = s[t];
                double den = 0.0;
                for (int t = 0; t <= p; t++) { s[t] = exp(s[t] - M); den += s[t]; }
                for (int c = 0; c < d; c++) o[c] = 0.0;
                for (int t = 0; t <= p; t++) {
                    int32_t blk = block_tables[(int64_t)b * max_blocks + t / block_size];
                    const uint8_t *vt = v_cache + cache_offset(blk, j, t % block_size, n_kv, block_size, d);
                    for (int c = 0; c < d; c++) o[c] += s[t] * (val[vt[c]] * (double)v_scale[j]);
                }
                for (int c = 0; c < d; c++) o[c] /= den;
            }
        }
        free(s);
    }
    free(row0);
    return status;
}

/*
 * Stochastic speculative acceptance -- modified rejection sampling
 * ([SE] 31.5 and Example 31.3; [SI] 12.4; [KVC] 08 "Why the output keeps the
 * exact distribution").
 *
 * For each sequence b, the drafts x_j ~ q_j, j = 0..k-1, are checked in order:
 * x_j is accepted with probability min(1, p_j(x_j) / q_j(x_j)), decided with
 * the caller's uniform r_j as  r_j * q_j(x_j) < p_j(x_j)  (fp32 multiply and
 * compare: the decision is an integer, so it is taken in the precision the
 * GPU kernel uses).  At the first rejection j* the round ends and the next
 * token is drawn from the normalised positive part max(0, p_j* - q_j*); when
 * all k drafts are accepted it is drawn from p_k (the extra target position).
 *
 * The draw is inverse-CDF sampling with the caller's uniform s_b over the
 * distribution quantised to units of 2^-32: w_t = quant(value_t), where the
 * residual value is the fp32 difference p - q, quant(x) = 0 for x <= 0 or NaN,
 * 2^32 for x >= 1, else floor(x * 2^32); T = floor(s * sum w) exactly; the
 * token is the smallest t whose inclusive prefix sum of w exceeds T.  Integer
 * sums make the draw independent of summation order.  If every weight of the
 * chosen distribution is zero, the residual falls back to p_j*; if that is
 * zero too, next = -1 and status bit 256 is set.  A draft outside [0, V) is
 * rejected and sets status bit 128.
 *
 * p  [B][k+1][V] fp32, q [B][k][V] fp32, draft [B][k], r [B][k], s [B].
 * Outputs accepted [B] (0..k) and next_token [B].  Returns the status bits.
 */
static uint64_t quant32(float x) {
    if (!(x > 0.0f)) return 0;            /* <= 0 or NaN */
    if (x >= 1.0f) return (uint64_t)1 << 32;
    return (uint64_t)(x * 4294967296.0f); /* exact scaling by 2^32, truncation */
}

/* floor(s * total) for s in [0, 1): s = m * 2^(e - 24) with integer m < 2^24 */
static uint64_t scaled_floor(float s, uint64_t total) {
    if (!(s > 0.0f)) return 0;
    if (s >= 1.0f) return total ? total - 1 : 0;
    int e;
    const double f = frexp((double)s, &e);          /* s = f * 2^e, f in [0.5, 1) */
    const uint64_t m = (uint64_t)ldexp(f, 24);       /* exact: s has 24 significant bits */
    const unsigned __int128 prod = (unsigned __int128)m * total;
    const int sh = 24 - e;                           /* s = m * 2^-sh, sh >= 25 */
    return sh >= 128 ? 0 : (uint64_t)(prod >> sh);
}

static int64_t inverse_cdf(const uint64_t *w, int64_t V, float s) {
    uint64_t total = 0;
    for (int64_t t = 0; t < V; t++) total += w[t];
    if (total == 0) return -1;
    const uint64_t T = scaled_floor(s, total);
    uint64_t c = 0;
    for (int64_t t = 0; t < V; t++) {
        c += w[t];
        if (c > T) return t;
    }
    return V - 1; /* not reached: T < total */
}

int oracle_spec_accept_sample(int32_t *accepted, int32_t *next_token, const float *p, const float *q,
                              const int32_t *draft, const float *r, const float *s, int B, int k, int V) {
    int status = 0;
    uint64_t *w = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(V > 0 ? V : 1));
    for (int b = 0; b < B; b++) {
        int j = 0;
        for (; j < k; j++) {
            const int32_t x = draft[(int64_t)b * k + j];
            if (x < 0 || x >= V) {
                status |= 128;
                break;
            }
            const float px = p[((int64_t)b * (k + 1) + j) * V + x];
            const float qx = q[((int64_t)b * k + j) * V + x];
            const float rq = r[(int64_t)b * k + j] * qx; /* one fp32 rounding */
            if (!(rq < px)) break;
        }
        accepted[b] = j;
        const float *pj = p + ((int64_t)b * (k + 1) + j) * V;
        int64_t t;
        if (j < k) {
            const float *qj = q + ((int64_t)b * k + j) * V;
            for (int64_t u = 0; u < V; u++) w[u] = quant32(pj[u] - qj[u]);
            t = inverse_cdf(w, V, s[b]);
            if (t < 0) {
                for (int64_t u = 0; u < V; u++) w[u] = quant32(pj[u]);
                t = inverse_cdf(w, V, s[b]);
            }
        } else {
            for (int64_t u = 0; u < V; u++) w[u] = quant32(pj[u]);
            t = inverse_cdf(w, V, s[b]);
        }
        if (t < 0) status |= 256;
        next_token[b] = (int32_t)t;
    }
    free(w);
    return status;
}

/*
 * Prefix-cache block hashes ([KVC] 05 "Prefix caching": each full block is
 * identified by a hash of itself plus the hash of its parent block, i.e. of the
 * whole prefix up to that block; [SE] 31.3: the key must cover the token
 * content and the computation version, and only a shared beginning counts).
 *
 * The hash is this library's own definition (the pages fix none), 128 bits as two
 * 64-bit lanes L = 0, 1; salt = the caller's computation-version key:
 *   mix(x):  x ^= x >> 32; x *= M; x ^= x >> 29; x *= M; x ^= x >> 32,
 *            M = 0xD6E8FEB86659FD93 (arithmetic mod 2^64)
 *   content: c = S_L ^ salt; for i = 0..bs-1: c = mix(c + (uint32)tok_i + (i << 32));
 *            d_j = mix(c + 0x9E3779B97F4A7C15) mod P
 *   chain:   a_{-1} = S_L mod P;  a_j = (a_{j-1} * X_L + d_j) mod P,  P = 2^61 - 1
 *            (the parent's hash times X_L plus the block's own digest)
 *   key_j:   lane L = mix(a_j), except that a key whose lane 1 is 0 and lane 0
 *            is 0 or 1 takes lane 1 = 1 ((0, 0) and (1, 0) mark the table's
 *            empty and removed entries)
 * with S0 = 0x243F6A8885A308D3, S1 = 0x13198A2E03707344, X0 =
 * 0x0C3A5F1D2B4E6978, X1 = 0x15D3B7E9A1C4F286.  Only full blocks (j < len / bs)
 * are hashed.  hashes: [num_seqs][max_blocks][2] (lane 0, lane 1); entries
 * past a sequence's full blocks are left alone.
 */
static uint64_t hmix(uint64_t x) {
    const uint64_t M = 0xD6E8FEB86659FD93ull;
    x ^= x >> 32;
    x *= M;
    x ^= x >> 29;
    x *= M;
    x ^= x >> 32;
    return x;
}

static const uint64_t P61 = (1ull << 61) - 1;

static uint64_t mulmod61(uint64_t a, uint64_t b) {
    const unsigned __int128 p = (unsigned __int128)a * b;
    uint64_t r = (uint64_t)(p % P61);
    return r;
}

int oracle_prefix_hash(uint64_t *hashes, const int32_t *tokens, int max_tokens, const int32_t *lens, int num_seqs,
                       int block_size, int max_blocks, uint64_t salt) {
    const uint64_t seed[2] = {0x243F6A8885A308D3ull, 0x13198A2E03707344ull};
    const uint64_t X[2] = {0x0C3A5F1D2B4E6978ull, 0x15D3B7E9A1C4F286ull};
    for (int b = 0; b < num_seqs; b++) {
        int nfull = lens[b] / block_size;
        if (nfull > max_blocks) nfull = max_blocks;
        uint64_t a[2] = {seed[0] % P61, seed[1] % P61};
        for (int j = 0; j < nfull; j++) {
            uint64_t key[2];
            for (int L = 0; L < 2; L++) {
                uint64_t c = seed[L] ^ salt;
                for (int i = 0; i < block_size; i++) {
                    const uint32_t t = (uint32_t)tokens[(int64_t)b * max_tokens + (int64_t)j * block_size + i];
                    c = hmix(c + (uint64_t)t + ((uint64_t)i << 32));
                }
                const uint64_t d = hmix(c + 0x9E3779B97F4A7C15ull) % P61;
                a[L] = (mulmod61(a[L], X[L]) + d) % P61;
                key[L] = hmix(a[L]);
            }
            if (key[1] == 0 && key[0] < 2) key[1] = 1;
            hashes[((int64_t)b * max_blocks + j) * 2] = key[0];
            hashes[((int64_t)b * max_blocks + j) * 2 + 1] = key[1];
        }
    }
    return 0;
}

/* Threads for the oracle's parallel loops from now on (no effect without
 * OpenMP); the CPU-baseline timing runs the same step on all cores and on one. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Number of threads the oracle's parallel loops use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
#else
    return 1;
#endif
}
