/*
 * pkv.h -- C ABI of libpkv, paged-KV decode attention for GB300 (sm_103a).
 *
 * The operations follow these web pages:
 *   [KVC] "Inference at Scale: KV Cache, Prefill, and Decode"
 *         (blog.truongducdung.dev): section 02 (decode appends one K/V row and
 *         rereads the cache; GQA intensity), 03 (bytes per token), 05 (block
 *         table, block sharing and copy-on-write), 07 (online softmax,
 *         FlashAttention loop, Flash-Decoding split-KV + log-sum-exp merge),
 *         08 (speculative verification, greedy rule).
 *   [SE]  "Chapter 31 Serving Efficiency" (imbrooklyn.dev): 31.3 (shared
 *         prefix, copy a block when a branch appends), 31.4 (Example 31.2,
 *         combine tile statistics), 31.5 (greedy acceptance).
 *   [SI]  "Spending the Idle" (derivingsystems.com): 12.4 (accept the
 *         longest matching prefix, stop at the first miss).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is DEVICE memory on the current CUDA device,
 *   allocated and owned by the caller.  The library allocates no device
 *   memory; kernels that need scratch take a caller-provided workspace.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream).  Nothing synchronises the host.
 * - bf16 tensors hold raw bfloat16 values (2 bytes each), 16-byte aligned.
 * - Cache layout: k_cache and v_cache are separate pools
 *   [num_blocks][num_kv_heads][block_size][head_dim] bf16, so one
 *   (block, kv head) tile is block_size * head_dim * 2 contiguous bytes.
 *   Logical token t of sequence b is row t % block_size of physical block
 *   block_tables[b * max_blocks + t / block_size] ([KVC] 05).
 * - block_tables: int32 [num_seqs][max_blocks]; entries past a sequence's
 *   last block are never read.
 * - Query head h reads kv head h / g, g = num_q_heads / num_kv_heads
 *   ([KVC] 04, GQA: contiguous groups).
 * - Return value: PKV_OK (0) when the work was enqueued; a negative PKV_ERR_*
 *   when the host detected a bad argument (nothing was enqueued) or the launch
 *   failed.
 * - Device-detected input errors (block id out of range, bad lengths, bad
 *   slots) are OR-ed into *status (device int32, may be NULL) as
 *   PKV_STATUS_* bits; the affected outputs are written as NaN or skipped as
 *   documented per call.  No kernel traps, asserts or spins without a bound:
 *   a wait that runs out sets PKV_STATUS_TIMEOUT.
 * - Results are deterministic: no floating-point atomics, and the attention
 *   result does not depend on where the physical blocks sit in the pool.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_OK 0
#define PKV_ERR_NULL (-1)        /* a required pointer is NULL */
#define PKV_ERR_SIZE (-2)        /* a size or count argument is out of range */
#define PKV_ERR_UNSUPPORTED (-3) /* head_dim, block_size or head grouping not supported */
#define PKV_ERR_WORKSPACE (-4)   /* workspace missing or smaller than required */
#define PKV_ERR_ALIGN (-5)       /* a pointer is not 16-byte aligned */
#define PKV_ERR_CUDA (-6)        /* a CUDA runtime call or launch failed */
#define PKV_ERR_DEVICE (-7)      /* the current device is not an sm_103 GPU */
#define PKV_ERR_SCRATCH_LIMIT (-8) /* the problem needs more scratch than the fixed no-alloc buffer */

#define PKV_STATUS_BAD_BLOCK 1   /* a needed block id is outside [0, num_blocks) */
#define PKV_STATUS_BAD_SEQLEN 2  /* a seq_len is < 0, > max_blocks*block_size or > max_seq_len */
#define PKV_STATUS_BAD_QLEN 4    /* a q_len/append_len is < 0, > seq_len or > max_q_len, or rows overflow */
#define PKV_STATUS_BAD_SLOT 8    /* a slot is >= num_blocks*block_size */
#define PKV_STATUS_TIMEOUT 32    /* a bounded device wait ran out (library bug) */
#define PKV_STATUS_BAD_PAIR 64   /* a copy pair names a block outside the pool */
#define PKV_STATUS_BAD_TOKEN 128 /* a draft token is outside [0, vocab) */
#define PKV_STATUS_BAD_DIST 256  /* a sampling distribution has no positive weight */
#define PKV_STATUS_TABLE_FULL 512  /* a prefix-cache insert found no free entry */
#define PKV_STATUS_NOT_FOUND 1024  /* a prefix-cache release named a key not in the table */
#define PKV_STATUS_BAD_PLAN 2048   /* an attention run found no plan for its shape in the workspace */

/* Attention flags. */
#define PKV_ATTN_DECODE_CUDA_CORES 1 /* run q_len = 1 rows on the CUDA-core FMA path */
#define PKV_ATTN_NO_TCGEN05 2        /* run every multi-query tile on mma.sync (no tcgen05 tiles) */
#define PKV_ATTN_PLAN_FP8 4          /* pkv_attention_plan only: the runs are over e4m3 pools */

/* Library version, 100 * major + minor. */
int pkv_version(void);

/* Text for a PKV_ERR_* return code or a single PKV_STATUS_* bit. */
const char* pkv_error_string(int rc);
const char* pkv_status_string(int bit);

/*
 * a1. Slot mapping ([KVC] 05, "The block table").
 * The new tokens of sequence b are its last append_lens[b] positions
 * pos in [seq_lens[b] - append_lens[b], seq_lens[b]); each gets
 *   slots[o] = block_tables[b][pos / block_size] * block_size + pos % block_size
 * packed in sequence order (o runs over sequences, then positions).
 *   slots        int64 [num_slots] out; num_slots must equal sum(append_lens)
 *   seq_lens     int32 [num_seqs], append_lens int32 [num_seqs]
 * Invalid lengths (PKV_STATUS_BAD_SEQLEN / BAD_QLEN) or block ids
 * (BAD_BLOCK) give slot -1 ("skip" for pkv_kv_append).
 * num_seqs <= 16384.
 */
int pkv_slot_mapping(int64_t* slots, const int32_t* block_tables, int max_blocks,
                     const int32_t* seq_lens, const int32_t* append_lens, int num_seqs,
                     int num_slots, int block_size, int num_blocks, int32_t* status,
                     void* stream);

/*
 * a2. KV append ([KVC] 02: each decode step appends one K/V row per new
 * token before attention rereads the cache).
 *   k_new, v_new  bf16 [num_tokens][num_kv_heads][head_dim]
 *   slots         int64 [num_tokens]; slot < 0 skips the token,
 *                 slot >= num_blocks*block_size sets PKV_STATUS_BAD_SLOT and
 *                 skips it.
 * Row slots[t] % block_size of block slots[t] / block_size receives token t,
 * all kv heads.  Bit-exact copy.  Two tokens with the same slot race.
 * head_dim must be a multiple of 8.
 */
int pkv_kv_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                  const int64_t* slots, int num_tokens, int num_blocks, int block_size,
                  int num_kv_heads, int head_dim, int32_t* status, void* stream);

/*
 * a3. Copy-on-write block copy ([SE] 31.3: share physical blocks and copy a
 * block when a branch appends; [KVC] 05 "Block sharing and copy-on-write").
 *   src_dst  int32 [num_pairs][2]: every byte of K and V of block src is
 *            copied to block dst.
 * Destinations must be distinct and must not also be sources in the same
 * call (pairs run in parallel).  A pair outside [0, num_blocks) sets
 * PKV_STATUS_BAD_PAIR and is skipped.  Bit-exact.
 */
int pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* src_dst, int num_pairs,
                    int num_blocks, int block_size, int num_kv_heads, int head_dim,
                    int32_t* status, void* stream);

/*
 * a4 as a standalone utility: block-table gather ([KVC] 05: the kernel
 * reads K and V through the block table).  Writes each sequence's K/V
 * contiguously:
 *   k_out, v_out  bf16 [sum seq_lens][num_kv_heads][head_dim]
 *   out_offsets   int64 [num_seqs]: first output row of sequence b
 * A bad block id writes NaN rows and sets PKV_STATUS_BAD_BLOCK; a bad
 * seq_len skips the sequence and sets PKV_STATUS_BAD_SEQLEN.  Bit-exact.
 */
int pkv_gather_kv(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                  const int64_t* out_offsets, int num_seqs, int num_blocks, int block_size,
                  int num_kv_heads, int head_dim, int32_t* status, void* stream);

/*
 * Smallest partition length pkv_paged_attention_decode uses when
 * partition_tokens is 0, for a batch of num_seqs sequences no longer than
 * max_seq_len (512, doubled while a sequence would have more than 1024
 * partitions).  It sizes the workspace; the call itself gives each sequence
 * a partition length of its own, never shorter (see partition_tokens below).
 */
int pkv_attention_auto_partition(int num_seqs, int total_q, int num_kv_heads, int max_seq_len);

/*
 * Workspace bytes pkv_paged_attention_decode needs for these bounds
 * (total_q = sum of q_lens, max_seq_len >= every seq_len).  The same
 * workspace may be reused by calls on the same stream.
 */
size_t pkv_attention_workspace_bytes(int num_seqs, int total_q, int num_q_heads, int num_kv_heads,
                                     int head_dim, int max_seq_len, int partition_tokens);

/*
 * a4-a8. Paged attention for decode, speculative verification and chunked
 * prefill in one launch.
 *
 * Computes, for every sequence b, query i < q_lens[b] and query head h,
 * the softmax attention of q over the K/V of kv head h / g read through the
 * block table ([KVC] 05), causal within the new tokens: query i sits at
 * position p = seq_lens[b] - q_lens[b] + i and sees positions 0..p ([KVC] 08:
 * the verify pass is like a short prefill):
 *   s_t = scale * <q, K_t>,  o = sum_t softmax(s)_t V_t.
 * It is evaluated with the online-softmax recurrence ([KVC] 07: running max
 * m, running sum l, rescale O by exp(m_old - m_new)), split into partitions
 * of partition_tokens positions whose partial (O, m, l) are merged with the
 * log-sum-exp rescaling of Flash-Decoding ([KVC] 07; [SE] Example 31.2:
 * combine tile statistics, not tile averages).  Arithmetic is fp32 on bf16
 * inputs; out is bf16 (round to nearest even).
 *
 *   out, q        bf16 [total_q][num_q_heads][head_dim], sequences in batch
 *                 order (the first q_lens[0] rows belong to sequence 0, ...)
 *   seq_lens      int32 [num_seqs], INCLUDING the new tokens, whose K/V must
 *                 already be in the cache (pkv_kv_append)
 *   q_lens        int32 [num_seqs]: 1 = decode, k > 1 = speculative verify
 *                 or a prefill chunk, 0 = no rows
 *   max_q_len     host bound on every q_len (a larger q_len is BAD_QLEN);
 *                 the tcgen05 tile code runs only when max_q_len * g > 24
 *   max_seq_len   host bound on every seq_len (sizes the workspace)
 *   head_dim      64 or 128; block_size a power of two in [1, 256];
 *                 g = num_q_heads / num_kv_heads an integer in [1, 64]
 *   partition_tokens  multiple of 16, at most 1024 partitions per sequence,
 *                 every sequence cut at multiples of it; or 0: automatic --
 *                 the planning kernel cuts each sequence into nearly equal
 *                 partitions (whole 16-token stages; 32 for FP8 pools, 128
 *                 for tcgen05 tiles) of at least
 *                 P0 = pkv_attention_auto_partition(...): about
 *                 round(L / C) of them for a target length C of the batch's
 *                 work over two items per SM (up to 8192), or, for a batch
 *                 of up to 1024 sequences made mostly of multi-row
 *                 decode-style sequences (speculative verification), the
 *                 shortest length whose items fit on the SMs in one wave
 *                 (ceil(L / C) partitions of at most C); the target C is the int at byte offset 8 of
 *                 the workspace after the call
 *   flags         0, or an OR of PKV_ATTN_DECODE_CUDA_CORES (q_len = 1 rows
 *                 on the CUDA-core FMA path; by default every row uses the
 *                 tensor cores, measured faster on GB300) and
 *                 PKV_ATTN_NO_TCGEN05.  A sequence with q_len * g <= 24
 *                 (query, q head) columns per kv head -- decode rows, and
 *                 speculative verification of up to 6 tokens at g = 4 -- runs
 *                 on the transposed tensor-core item.  By default (head_dim
 *                 128, block_size >= 16, partition length a multiple of 128,
 *                 decode rows on tensor cores) a sequence with q_len * g > 24
 *                 runs as tiles of 128 (query, q head) rows
 *                 of one kv head on the tcgen05 tensor cores (accumulators in
 *                 tensor memory, 128-token stages); PKV_ATTN_NO_TCGEN05 keeps
 *                 it on the mma.sync multi-query path
 *   workspace     >= pkv_attention_workspace_bytes(...) bytes, 256-byte
 *                 aligned; scratch, contents need not be initialised
 * Rows of a sequence with a bad length, or that read a bad block id, are
 * NaN and set the matching PKV_STATUS_* bit.  Output rows are written once;
 * the result is bit-identical under any permutation of the physical blocks.
 */
int pkv_paged_attention_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                               const int32_t* q_lens, int num_seqs, int total_q, int max_q_len,
                               int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, float scale, int partition_tokens,
                               int flags, void* workspace, size_t workspace_bytes, int32_t* status,
                               void* stream);

/*
 * The two halves of pkv_paged_attention_decode, so that one plan serves many
 * calls.  A model calls attention once per layer over the same block tables
 * and lengths ([KVC] 03: the KV bytes a decode step reads are summed over
 * every layer; [KVC] 05: the block table is per sequence, not per layer), so
 * the work list -- which depends only on seq_lens and q_lens -- is built once
 * per decode step and each layer runs over it.
 *
 * pkv_attention_plan: the planning part (one small kernel): validates the
 * lengths (PKV_STATUS_BAD_SEQLEN / BAD_QLEN bits into *status, may be NULL),
 * picks the partition length and writes the work list into the workspace.
 * Arguments as in pkv_paged_attention_decode; flags may add
 * PKV_ATTN_PLAN_FP8 when the runs will be pkv_paged_attention_run_fp8 (then
 * no other flag).  The workspace (pkv_attention_workspace_bytes, 256-byte
 * aligned) then holds the plan until the next plan written into it.
 *
 * pkv_paged_attention_run / pkv_paged_attention_run_fp8: the attention over
 * a planned workspace (the attention and combine kernels): the same
 * computation, outputs and error behaviour as pkv_paged_attention_decode /
 * pkv_paged_attention_decode_fp8_ex (kv_format, scale_mode as there) for the
 * lengths the plan was made from.
 * Every size and flag argument must equal the plan's (num_blocks, scale,
 * the pools, block tables, q and out are the run's own); a workspace planned
 * for another shape makes the run write every output row NaN and set
 * PKV_STATUS_BAD_PLAN (the check is a key of the sizes the plan leaves in the
 * workspace, so it catches a mismatch, not a changed length array).  Runs and
 * the plan must be ordered on one stream; the lengths must not change between
 * the plan and its runs.  Any number of runs may follow one plan: each run
 * leaves the plan as it found it.
 */
int pkv_attention_plan(const int32_t* seq_lens, const int32_t* q_lens, int num_seqs, int total_q,
                       int max_q_len, int max_seq_len, int max_blocks, int num_q_heads, int num_kv_heads,
                       int head_dim, int block_size, int partition_tokens, int flags, void* workspace,
                       size_t workspace_bytes, int32_t* status, void* stream);
int pkv_paged_attention_run(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks, int num_seqs, int total_q,
                            int max_q_len, int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int num_blocks, float scale, int partition_tokens, int flags,
                            void* workspace, size_t workspace_bytes, int32_t* status, void* stream);
int pkv_paged_attention_run_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                const float* k_scale, const float* v_scale, int kv_format, int scale_mode,
                                const int32_t* block_tables, int max_blocks, int num_seqs, int total_q,
                                int max_q_len, int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int num_blocks, float scale, int partition_tokens, void* workspace,
                                size_t workspace_bytes, int32_t* status, void* stream);

/*
 * No-allocation variant of pkv_paged_attention_decode.  The source pages have
 * no counterpart to this entry point; it exists for callers that cannot
 * allocate device memory on the call path -- code running inside another
 * runtime's allocator or memory-pool hooks (a nested cudaMalloc would re-enter
 * it), latency-critical loops that must not block on the driver allocator,
 * and plugins that are handed only their inputs and outputs.
 *
 * Same arguments, semantics and results as pkv_paged_attention_decode, minus
 * the workspace: the scratch lives in a fixed device array inside the library
 * (pkv_noalloc_scratch_bytes() bytes, 32 MiB), which every GPU that loads the
 * library holds until the process exits.  The call allocates nothing.
 * - Returns PKV_ERR_SCRATCH_LIMIT, launching nothing, when
 *   pkv_attention_workspace_bytes(...) for these sizes exceeds that array.
 * - The first call on a device (with that device current) looks up the
 *   array's device address; make that first call before any stream capture.
 *   The address is cached per device and per CUDA context (its unique id):
 *   after cudaDeviceReset, or any other destruction and re-creation of the
 *   device's context, the next call looks it up again and is then a first
 *   call in this sense.
 * - All calls share the array.  Calls that overlap on the GPU (other streams,
 *   unordered host threads) race on it and give wrong results; calls ordered
 *   on one stream are safe (each call re-initialises what it uses).
 */
size_t pkv_noalloc_scratch_bytes(void);
int pkv_paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       int max_blocks, const int32_t* seq_lens,
                                       const int32_t* q_lens, int num_seqs, int total_q,
                                       int max_q_len, int max_seq_len, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, int num_blocks, float scale,
                                       int partition_tokens, int flags, int32_t* status,
                                       void* stream);

/*
 * a1 + a2 in one launch: the slot mapping of pkv_slot_mapping (the new tokens
 * of sequence b are its last append_lens[b] positions, [KVC] 05) fused with
 * the append of pkv_kv_append ([KVC] 02).  Same arguments and status bits as
 * the two calls; slots (int64 [num_tokens]) receives the slots as
 * pkv_slot_mapping writes them.  Bit-exact with the two calls.  Batches of
 * more than 2048 sequences run the two kernels.
 */
int pkv_kv_append_paged(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                        const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                        const int32_t* append_lens, int num_seqs, int num_tokens, int num_blocks,
                        int block_size, int num_kv_heads, int head_dim, int64_t* slots,
                        int32_t* status, void* stream);

/*
 * FP8 KV cache ([KVC] 03, "KV cache quantization": store K and V in FP8, one
 * byte per value instead of two, halving the cache and the bytes decode
 * attention rereads; the formats are e4m3 and e5m2 -- these entry points use
 * e4m3, the variant without infinities: bias 7, 3 mantissa bits, largest
 * finite 448, S.1111.111 = NaN).
 *
 * Pools are uint8 [num_blocks][num_kv_heads][block_size][head_dim] in the
 * bf16 pools' layout.  Scales (the pages fix none): one fp32 dequantisation
 * scale per kv head for K (k_scale[num_kv_heads]) and for V, device memory,
 * chosen by the caller (for instance the head's largest magnitude / 448).
 *
 * pkv_kv_append_fp8: as pkv_kv_append, each bf16 value x of head h stored as
 * e4m3(x * (1 / scale[h])) -- the reciprocal and the product rounded to fp32
 * (nearest even), the conversion rounding to nearest even and saturating to
 * +-448 (NaN stays NaN).  Bit-exact; pools need 8-byte alignment.
 */
int pkv_kv_append_fp8(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                      const int64_t* slot_mapping, const float* k_scale, const float* v_scale,
                      int num_tokens, int num_blocks, int block_size, int num_kv_heads, int head_dim,
                      int32_t* status, void* stream);

/* pkv_copy_blocks for e4m3 pools (head_dim a multiple of 16).  Bit-exact. */
int pkv_copy_blocks_fp8(void* k_cache, void* v_cache, const int32_t* src_dst, int num_pairs,
                        int num_blocks, int block_size, int num_kv_heads, int head_dim,
                        int32_t* status, void* stream);

/*
 * pkv_paged_attention_decode over e4m3 pools: the same softmax attention with
 * K_t = e4m3(code) * k_scale[h / g] and V_t = e4m3(code) * v_scale[h / g]
 * ([KVC] 03; the attention itself as in pkv_paged_attention_decode, [KVC]
 * 05, 07, 08).  head_dim 128 and g <= 16; the other arguments, the workspace
 * (pkv_attention_workspace_bytes), the outputs and the error behaviour are
 * those of pkv_paged_attention_decode (no flags).  The products run on f16
 * tensor cores: e4m3 -> f16 is exact, q is rounded from bf16 to f16 (exact
 * for |q| in [6.1e-5, 65504]), accumulation is fp32, out is bf16.
 */
int pkv_paged_attention_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                                   const float* k_scale, const float* v_scale, const int32_t* block_tables,
                                   int max_blocks, const int32_t* seq_lens, const int32_t* q_lens,
                                   int num_seqs, int total_q, int max_q_len, int max_seq_len,
                                   int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                   float scale, int partition_tokens, void* workspace,
                                   size_t workspace_bytes, int32_t* status, void* stream);

/*
 * FP8 pools of either format and scale granularity ([KVC] 03, "KV cache
 * quantization": FP8 as fp8_e4m3 or fp8_e5m2; the pages fix no scaling).
 *   kv_format   PKV_FP8_E4M3 (as above) or PKV_FP8_E5M2: sign, 5 exponent bits
 *               (bias 15), 2 mantissa bits, subnormals m * 2^-16, infinities
 *               and NaN in exponent field 31, largest finite 57344; encoding
 *               rounds to nearest even and saturates to +-57344 (infinities
 *               too), NaN is stored as 0x7f
 *   scale_mode  PKV_FP8_SCALE_PER_HEAD: k_scale, v_scale fp32 [num_kv_heads],
 *               read only (as the e4m3 entry points above);
 *               PKV_FP8_SCALE_PER_BLOCK: fp32 [num_blocks][num_kv_heads], one
 *               scale per (block, kv head) tile.  A block's scales are set when
 *               the block is opened -- by the append that writes its row 0 --
 *               from that row's values of each kv head: the smallest power of
 *               two s = 2^e, e in [-120, 120], with max|x| <= s * FMAX / 2
 *               (FMAX = 448 for e4m3, 57344 for e5m2; NaN values ignored;
 *               s = 1 for an all-zero or infinite row).  The opening row then
 *               uses at most half of the format's range; later rows of the
 *               block are stored with the same scale and saturate only beyond
 *               twice its magnitude.  Rows appended in the same call as their
 *               block's row 0 use the scale that row sets (the call runs a
 *               small scale kernel first).  The caller initialises the scales
 *               of blocks that hold data before their row 0 is appended here.
 *               With per-block V scales the kernel multiplies each token's
 *               probability (<= 2^8) by its V scale in f16: V scales up to 2^7
 *               are safe.
 * pkv_kv_append_fp8_ex: as pkv_kv_append_fp8, in the given format; with
 *   per-block scales it sets the opened blocks' scales (k_scale, v_scale are
 *   then written) and stores every row with its block's scales.
 * pkv_copy_blocks_fp8_ex: as pkv_copy_blocks_fp8; with per-block scales the
 *   copied blocks' scales are copied too.
 * pkv_paged_attention_decode_fp8_ex: the attention of
 *   pkv_paged_attention_decode_fp8 with K_t = fp8(code) * (scale of t's kv
 *   head, or of t's (block, kv head) tile), V likewise.  e5m2 -> f16 is exact
 *   (an e5m2 code is the upper byte of its f16).
 * Every other argument, the workspace and the error behaviour as in the e4m3
 * entry points; an unknown kv_format or scale_mode is PKV_ERR_UNSUPPORTED.
 */
#define PKV_FP8_E4M3 0
#define PKV_FP8_E5M2 1
#define PKV_FP8_SCALE_PER_HEAD 0
#define PKV_FP8_SCALE_PER_BLOCK 1
int pkv_kv_append_fp8_ex(void* k_cache, void* v_cache, float* k_scale, float* v_scale, const void* k_new,
                         const void* v_new, const int64_t* slots, int num_tokens, int num_blocks, int block_size,
                         int num_kv_heads, int head_dim, int kv_format, int scale_mode, int32_t* status,
                         void* stream);
int pkv_copy_blocks_fp8_ex(void* k_cache, void* v_cache, float* k_scale, float* v_scale, const int32_t* src_dst,
                           int num_pairs, int num_blocks, int block_size, int num_kv_heads, int head_dim,
                           int scale_mode, int32_t* status, void* stream);
int pkv_paged_attention_decode_fp8_ex(void* out, const void* q, const void* k_cache, const void* v_cache,
                                      const float* k_scale, const float* v_scale, int kv_format, int scale_mode,
                                      const int32_t* block_tables, int max_blocks, const int32_t* seq_lens,
                                      const int32_t* q_lens, int num_seqs, int total_q, int max_q_len,
                                      int max_seq_len, int num_q_heads, int num_kv_heads, int head_dim,
                                      int block_size, int num_blocks, float scale, int partition_tokens,
                                      void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Prefix-cache block lookup ([KVC] 05, "Prefix caching": every full block is
 * identified by a hash of itself plus the hash of its parent block -- of the
 * whole prefix up to it; a new request looks the hashes up and, on a match,
 * bumps the block's ref count and skips that part of prefill.  [SE] 31.3:
 * only a shared beginning counts, and the key must cover the computation
 * version as well as the tokens).  The results feed the block tables the
 * attention reads.
 *
 * Block hash (this library's definition; the pages fix none): 128 bits, two
 * 64-bit lanes L = 0, 1, seeds S0 = 0x243F6A8885A308D3, S1 = 0x13198A2E03707344,
 * multipliers X0 = 0x0C3A5F1D2B4E6978, X1 = 0x15D3B7E9A1C4F286, P = 2^61 - 1:
 *   mix(x):  x ^= x >> 32; x *= M; x ^= x >> 29; x *= M; x ^= x >> 32,
 *            M = 0xD6E8FEB86659FD93 (mod 2^64)
 *   digest of block j:  c = S_L ^ salt;
 *                       for i < block_size: c = mix(c + (uint32)tok[j*bs+i] + (i << 32));
 *                       d_j = mix(c + 0x9E3779B97F4A7C15) mod P
 *   chain:   a_-1 = S_L mod P;  a_j = (a_{j-1} * X_L + d_j) mod P
 *            (the parent's hash times X plus the block's own digest)
 *   key_j:   lane L = mix(a_j); a key with lane 1 == 0 and lane 0 < 2 takes
 *            lane 1 = 1 ((0, 0) and (1, 0) mark empty and removed entries).
 * salt is the caller's computation-version key (model, adapter, positional
 * settings).  Only full blocks are hashed.  The chain's affine steps compose
 * associatively, so the GPU evaluates it as a parallel prefix scan.
 *
 * Table: device memory of pkv_prefix_table_bytes(capacity) bytes (capacity a
 * power of two, 16-byte aligned), caller-owned; entries are 32 bytes
 * {uint64 key lane 0, uint64 key lane 1, int32 block id, int32 ref count},
 * open addressing with linear probing from lane 0 mod capacity.  Calls on one
 * table must be ordered (one stream).
 */
size_t pkv_prefix_table_bytes(int capacity);
int pkv_prefix_table_init(void* table, int capacity, void* stream);

/*
 * hashes uint64 [num_seqs][max_blocks][2] out: keys of the full blocks
 * j < lens[b] / block_size (entries past them untouched); tokens int32
 * [num_seqs][max_tokens], max_tokens >= max_blocks * block_size.
 */
int pkv_prefix_hash(uint64_t* hashes, const int32_t* tokens, int max_tokens, const int32_t* lens,
                    int num_seqs, int block_size, int max_blocks, uint64_t salt, void* stream);

/*
 * For each sequence, the longest run of leading full blocks whose keys are in
 * the table: cached_blocks[b] = its length n, block_tables[b][j] (int32
 * [num_seqs][max_blocks]) = the cached block of key j for j < n (other entries
 * untouched), and each of those entries gains a reference.
 */
int pkv_prefix_lookup(void* table, int capacity, const uint64_t* hashes, const int32_t* lens,
                      int num_seqs, int block_size, int max_blocks, int32_t* block_tables,
                      int32_t* cached_blocks, void* stream);

/*
 * Register block_tables[b][j] under hashes[b][j] for j in [first[b],
 * first[b] + count[b]), each registration taking a reference.  A key already
 * in the table keeps its block; several sequences inserting one new key in
 * the same call agree on one of their blocks.  resolved (int32
 * [num_seqs][max_blocks], entries in range only) = the block the table holds
 * for the key afterwards (the caller's own, or the one to share instead);
 * -1 and PKV_STATUS_TABLE_FULL when no free entry was left.  Removed entries
 * are not reused; re-initialise the table to reclaim them.
 */
int pkv_prefix_insert(void* table, int capacity, const uint64_t* hashes, const int32_t* block_tables,
                      const int32_t* first, const int32_t* count, int num_seqs, int max_blocks,
                      int32_t* resolved, int32_t* status, void* stream);

/*
 * Drop one reference of the blocks j < count[b] of each sequence (a finished
 * request); a key not in the table sets PKV_STATUS_NOT_FOUND.  Entries whose
 * count reaches 0 stay cached (evictable by the caller's policy).
 */
int pkv_prefix_release(void* table, int capacity, const uint64_t* hashes, const int32_t* count,
                       int num_seqs, int max_blocks, int32_t* status, void* stream);

/*
 * a9. Greedy speculative acceptance ([SI] 12.4; [KVC] 08: with greedy
 * decoding a draft token is accepted when it equals the target's argmax;
 * stop at the first mismatch; the round always adds one target token).
 *   logits      fp32 [num_seqs][k+1][vocab]: target scores at the k drafted
 *               positions and the one after them
 *   draft       int32 [num_seqs][k]
 *   argmax_out  int32 [num_seqs][k+1] out: first index of the row maximum
 *               (NaN counts as the maximum, the first NaN wins)
 *   accepted    int32 [num_seqs] out: leading j < k with draft == argmax
 *   next_token  int32 [num_seqs] out: argmax_out[b][accepted[b]] (the
 *               correction, or the bonus token when all k are accepted)
 * Exact integers.  vocab >= 1, 1 <= k <= 64.
 */
int pkv_spec_accept_greedy(const float* logits, const int32_t* draft, int num_seqs, int k,
                           int vocab, int32_t* argmax_out, int32_t* accepted, int32_t* next_token,
                           void* stream);

/*
 * Stochastic speculative acceptance: modified rejection sampling ([SE] 31.5
 * and Example 31.3; [SI] 12.4; [KVC] 08 "Why the output keeps the exact
 * distribution").  For each sequence the drafts are checked in order: draft
 * x_j (drawn by the caller from q_j) is accepted with probability
 * min(1, p_j(x_j) / q_j(x_j)); at the first rejection j the round ends and the
 * next token is drawn from the normalised positive part max(0, p_j - q_j);
 * when all k drafts pass it is drawn from p_k, the target's distribution after
 * them.  The emitted tokens are distributed exactly as the target's.
 *   p           fp32 [num_seqs][k+1][vocab]  target distributions (rows sum to 1)
 *   q           fp32 [num_seqs][k][vocab]    draft distributions
 *   draft       int32 [num_seqs][k]
 *   r           fp32 [num_seqs][k] uniforms in [0, 1): x_j is accepted iff
 *               r_j * q_j(x_j) < p_j(x_j), fp32 multiply (round to nearest)
 *   s           fp32 [num_seqs] uniform in [0, 1) for the one draw of the round
 *   accepted    int32 [num_seqs] out: number of leading drafts accepted (0..k)
 *   next_token  int32 [num_seqs] out: the drawn token
 *   status      PKV_STATUS_* bits, may be null
 * The draw: weights w_t = quant(value_t), value = the fp32 difference p - q
 * (or p), quant(x) = 0 for x <= 0 or NaN, 2^32 for x >= 1, else
 * floor(x * 2^32); T = floor(s * sum_t w_t) exactly; next_token = the smallest
 * t whose inclusive prefix sum of w exceeds T.  Integer sums make the token
 * independent of summation order, so it is reproducible and bit-exact against
 * a reference.  A residual with no positive weight falls back to p_j; if that
 * has none either, next_token = -1 and PKV_STATUS_BAD_DIST is set.  A draft
 * outside [0, vocab) is rejected at its position and sets
 * PKV_STATUS_BAD_TOKEN.  1 <= k <= 1024, vocab >= 1.  Reads the two rows of
 * the rejected position (one when all pass) plus 2k scalars per sequence.
 */
int pkv_spec_accept_sample(const float* p, const float* q, const int32_t* draft, const float* r,
                           const float* s, int num_seqs, int k, int vocab, int32_t* accepted,
                           int32_t* next_token, int32_t* status, void* stream);

/*
 * Self-test of the library's failure detection (no counterpart on the pages):
 * one warp waits, through the same bounded device wait every attention kernel
 * uses, on an mbarrier phase that nothing ever completes.  The wait gives up
 * after limit_ns nanoseconds of %globaltimer (1 ns .. 10 s), ORs
 * PKV_STATUS_TIMEOUT into *status (device int32, required) and the kernel
 * returns normally, so the context stays usable -- which is what a caller
 * relies on when a real wait inside an attention call runs out.
 * Returns PKV_ERR_SIZE for a limit outside the range, PKV_ERR_NULL for a null
 * status.
 */
int pkv_wait_selftest(long long limit_ns, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
