/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact-attention forward library.
 *
 * What it computes is defined on the explainer page "FlashAttention for
 * inference: tiled prefill and split-KV decoding" (pofe.ai):
 *   - attention itself: S = Q K^T * scale, P = softmax(S), O = P V
 *     (section "The bottleneck it attacks"), computed exactly up to rounding
 *     with the online softmax of section "The online softmax, with every
 *     symbol defined";
 *   - causal prefill in FlashAttention-2 loop order, one thread block per
 *     query tile, tiles above the diagonal skipped, each row's log-sum-exp
 *     written (section "Prefill: tiles, loop order and the tensor cores");
 *   - split-KV single-token decode over a grouped-query, optionally paged
 *     cache, with per-split partial outputs and LSEs (section "Decode: a
 *     different bottleneck");
 *   - the merge of partial results by their LSE weights (section "The online
 *     softmax ...", combining partial results, and the merge rule in section
 *     "Minimal implementation").
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer, allocated and owned by the
 *     caller.  The library never allocates, never frees and never
 *     synchronises (except attn_check_device_status), and launches all work
 *     on the caller's stream (`stream` is a cudaStream_t; NULL = the legacy
 *     default stream).
 *   - bf16 tensors are passed as `const attn_bf16*` (the raw 16-bit pattern).
 *   - All arrays are dense and row-major in the order their shape is written.
 *   - LSE values are natural logarithms of sums of exp(scaled score); an
 *     empty key set yields LSE = -inf and O = 0.
 *   - Arguments are validated before anything is launched; on any error the
 *     call returns a nonzero attn_status and launches nothing.
 *   - Kernel-side waits are bounded; a timeout, a block-table entry outside
 *     [0, num_blocks) or a kv_len above the cache capacity is recorded in a
 *     per-device error word that attn_check_device_status reports.
 *   - Grouped-query attention: g = n_q_heads / n_kv_heads query heads share a
 *     key/value head; query head h reads key/value head h / g.
 */
#ifndef ATTN_SM103_H
#define ATTN_SM103_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t attn_bf16; /* bfloat16 bit pattern */

typedef enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_NULL = 1,     /* a required pointer is NULL                          */
  ATTN_ERR_SHAPE = 2,    /* a size is out of range (batch, heads, seqlen, ...)   */
  ATTN_ERR_HEADDIM = 3,  /* head_dim not supported by the call (see its limits) */
  ATTN_ERR_GQA = 4,      /* n_q_heads not a multiple of n_kv_heads, or g > 64 in decode */
  ATTN_ERR_SPLITS = 5,   /* num_splits < 0 or above the supported maximum        */
  ATTN_ERR_ALIGN = 6,    /* a pointer is not aligned as documented               */
  ATTN_ERR_ARCH = 7,     /* the current device is not sm_103 (GB300)             */
  ATTN_ERR_LAUNCH = 8,   /* a CUDA runtime call or kernel launch failed          */
  ATTN_ERR_TIMEOUT = 9,  /* a kernel's bounded wait gave up (device error word)  */
  ATTN_ERR_DEVICE = 10,  /* bad block-table entry or kv_len seen by a kernel     */
  ATTN_ERR_SCRATCH = 11  /* attn_decode_noalloc: partials exceed its fixed buffer */
} attn_status;

/* Name of a status code; never NULL. */
const char* attn_status_string(int status);

/*
 * attn_prefill -- attention forward over whole sequences (causal prefill).
 *
 * Page: "FlashAttention for inference: tiled prefill and split-KV decoding",
 * section "Prefill: tiles, loop order and the tensor cores" (loop order,
 * causal skipping, the per-row log-sum-exp output) and the layout of
 * section "Minimal implementation" (batch, heads, seq, head_dim).
 *
 *   q   : (batch, n_q_heads,  seqlen, head_dim) bf16, 16-byte aligned
 *   k, v: (batch, n_kv_heads, seqlen, head_dim) bf16, 16-byte aligned
 *   o   : (batch, n_q_heads,  seqlen, head_dim) fp32 output, 16-byte aligned
 *   lse : (batch, n_q_heads,  seqlen) fp32 output (natural log), 4-byte aligned
 *   scale: multiplies q.k (pass 1/sqrt(head_dim) for standard attention)
 *   causal: nonzero -> row i attends to keys j <= i; zero -> to every key.
 * Limits: head_dim in {64, 128, 256} (256: 64-key tiles); 1 <= seqlen <= 2^24;
 *   batch*n_q_heads <= 2^20;
 *   batch*n_q_heads*ceil(seqlen/128) < 2^31; n_q_heads % n_kv_heads == 0.  bf16 inputs, fp32 accumulation, P rounded
 *   to bf16 before the P*V product.
 * Errors: ATTN_ERR_NULL, _SHAPE, _HEADDIM, _GQA, _ALIGN, _ARCH, _LAUNCH.
 */
int attn_prefill(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, float* o,
                 float* lse, int batch, int n_q_heads, int n_kv_heads, int seqlen,
                 int head_dim, float scale, int causal, void* stream);

/*
 * attn_prefill_ex -- attn_prefill with the attention variants of the page's
 * section "Interaction with post-trained models" (sliding windows, ALiBi and
 * logit soft-capping are among the variants current kernels support).
 *
 *   window_left: -1 for none; otherwise row i attends only to keys
 *                j >= i - window_left (with causal, i - window_left <= j <= i)
 *   softcap    : 0 for none; otherwise each scaled score s = scale * q.k is
 *                replaced by softcap * tanh(s / softcap) before the softmax
 *   alibi_slopes: NULL for none; otherwise (n_q_heads,) fp32 on the device,
 *                4-byte aligned: head h adds -alibi_slopes[h] * |i - j| to the
 *                score of query i and key j (after soft-capping)
 * ALiBi and soft-capping together are ATTN_ERR_SHAPE.  Everything else
 * (head_dim 64, 128 or 256), and the errors, as attn_prefill (a negative
 * window_left other than -1, or a negative or non-finite softcap, is
 * ATTN_ERR_SHAPE).
 */
int attn_prefill_ex(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, float* o,
                    float* lse, int batch, int n_q_heads, int n_kv_heads, int seqlen, int head_dim,
                    float scale, int causal, int window_left, float softcap,
                    const float* alibi_slopes, void* stream);

/*
 * attn_prefill_ex2 -- attn_prefill_ex with flags; ATTN_PREFILL_OUT_BF16 writes
 * O as bf16.
 *
 * Page: same, section "Prefill: tiles, loop order and the tensor cores" (the
 * output tile O_i = acc / l written once per query tile).
 *   o     : (batch, n_q_heads, seqlen, head_dim), fp32, or bf16 with
 *           ATTN_PREFILL_OUT_BF16: each value acc / l is computed in fp32 and
 *           rounded to the nearest bf16 (ties to even) once, so the bf16 O
 *           equals the fp32 O of the same call rounded; 16-byte aligned
 *   flags : 0 or ATTN_PREFILL_OUT_BF16; any other bit is ATTN_ERR_SHAPE
 * lse stays fp32.  Everything else, and the errors, as attn_prefill_ex.
 */
#define ATTN_PREFILL_OUT_BF16 1u
int attn_prefill_ex2(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, void* o,
                     float* lse, int batch, int n_q_heads, int n_kv_heads, int seqlen,
                     int head_dim, float scale, int causal, int window_left, float softcap,
                     const float* alibi_slopes, unsigned flags, void* stream);

/*
 * attn_prefill_varlen -- prefill of several sequences packed end to end
 * without padding (variable-length batch).
 *
 * Page: same, section "Interaction with post-trained models" (packed data and
 * variable-length batches: examples packed into one sequence do not attend to
 * each other; engines batch prompts of different lengths this way), with the
 * per-sequence computation of attn_prefill.
 *
 *   q   : (n_q_heads,  total_tokens, head_dim) bf16, 16-byte aligned
 *   k, v: (n_kv_heads, total_tokens, head_dim) bf16, 16-byte aligned
 *   o   : (n_q_heads,  total_tokens, head_dim) fp32 output, 16-byte aligned
 *   lse : (n_q_heads,  total_tokens) fp32 output (natural log), 4-byte aligned
 *   cu_seqlens: (num_seqs + 1,) int32 on the device, 0 = cu[0] <= cu[1] <= ...
 *         <= cu[num_seqs] <= total_tokens; sequence s is rows [cu[s], cu[s+1])
 *         (empty sequences allowed)
 *   causal: nonzero -> row i of a sequence attends to its keys j <= i; zero ->
 *         to every key of its own sequence.
 * Rows outside every sequence are not written.  A cu_seqlens that breaks the
 * rule above is clamped into it and flagged (ATTN_ERR_DEVICE from
 * attn_check_device_status).
 * Limits: 1 <= num_seqs <= 2^20 (more than 512 run as one launch per slice of
 *   512 sequences, in order on the stream); head_dim in {64, 128, 256};
 *   1 <= total_tokens <= 2^24; n_q_heads % n_kv_heads == 0;
 *   n_q_heads * (ceil(total_tokens/128) + num_seqs) < 2^31.
 * Errors: ATTN_ERR_NULL, _SHAPE, _HEADDIM, _GQA, _ALIGN, _ARCH, _LAUNCH.
 */
int attn_prefill_varlen(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, float* o,
                        float* lse, const int32_t* cu_seqlens, int num_seqs, int total_tokens,
                        int n_q_heads, int n_kv_heads, int head_dim, float scale, int causal,
                        void* stream);

/*
 * attn_prefill_varlen_ex -- attn_prefill_varlen with the variants of
 * attn_prefill_ex (sliding window, logit soft-capping, ALiBi).
 *
 * Page: same, section "Interaction with post-trained models" (packed batches
 * and the variants models are trained with).  Each sequence is attended on
 * its own rows with the variant applied as in attn_prefill_ex, positions i, j
 * counted from the sequence's first row: the window keeps keys j >= i -
 * window_left, ALiBi adds -alibi_slopes[h] * |i - j|.
 *   window_left, softcap, alibi_slopes: as attn_prefill_ex (ALiBi and
 *          soft-capping together are ATTN_ERR_SHAPE; alibi_slopes 4-byte aligned).
 * Other arguments, limits and errors as attn_prefill_varlen.
 */
int attn_prefill_varlen_ex(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, float* o,
                           float* lse, const int32_t* cu_seqlens, int num_seqs, int total_tokens,
                           int n_q_heads, int n_kv_heads, int head_dim, float scale, int causal,
                           int window_left, float softcap, const float* alibi_slopes,
                           void* stream);

/*
 * attn_prefill_varlen_ex2 -- attn_prefill_varlen_ex with the flags of
 * attn_prefill_ex2 (ATTN_PREFILL_OUT_BF16: o is (n_q_heads, total_tokens,
 * head_dim) bf16).  Rows outside every sequence are not written.  Everything
 * else as attn_prefill_varlen_ex.
 */
int attn_prefill_varlen_ex2(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, void* o,
                            float* lse, const int32_t* cu_seqlens, int num_seqs, int total_tokens,
                            int n_q_heads, int n_kv_heads, int head_dim, float scale, int causal,
                            int window_left, float softcap, const float* alibi_slopes,
                            unsigned flags, void* stream);

/*
 * attn_decode_num_splits -- the split-count policy for single-token decode.
 *
 * Page: same, section "Decode: a different bottleneck": splitting the key/value
 * sequence restores parallelism at small batch, adds only reduction overhead
 * at large batch, so the split count is chosen from batch, heads and length.
 * Returns a value in [1, ATTN_MAX_SPLITS] (1 for non-positive arguments).
 * num_sms <= 0 means "query the current device".  Pure host function.
 */
#define ATTN_MAX_SPLITS 1024
int attn_decode_num_splits(int batch, int n_kv_heads, int max_kv_len, int num_sms);

/*
 * attn_decode_splitkv -- split-KV single-token decode (partial results).
 *
 * Page: same, section "Decode: a different bottleneck" (split-KV, GQA-aware
 * key/value sharing, paged caches) and section "Minimal implementation" for
 * the cache, block-table and cache-length layouts.
 *
 *   q          : (batch, n_q_heads, head_dim) bf16, one query token per sequence,
 *                16-byte aligned
 *   k_cache,
 *   v_cache    : paged (block_table != NULL): (num_blocks, block_size, n_kv_heads, head_dim)
 *                contiguous (block_table == NULL): (batch, max_kv_len, n_kv_heads, head_dim)
 *                bf16, 16-byte aligned
 *   block_table: (batch, max_blocks_per_seq) int32 physical block ids, or NULL
 *   kv_lens    : (batch,) int32 tokens already cached per sequence (0 allowed);
 *                must not exceed max_blocks_per_seq*block_size (paged) or
 *                max_kv_len (contiguous) -- a larger value is clamped and flagged
 *   num_splits : number of splits S >= 1, or 0 for attn_decode_num_splits(batch,
 *                n_kv_heads, max_kv_len, 0) (the caller must size the partials for it)
 *   o_partial  : (S, batch, n_q_heads, head_dim) fp32 output, 16-byte aligned
 *   lse_partial: (S, batch, n_q_heads) fp32 output, 4-byte aligned
 *   block_size, max_blocks_per_seq, num_blocks: paged cache geometry (ignored
 *                when block_table is NULL); block_size must be >= 1
 *   max_kv_len : contiguous cache length; for a paged cache, the largest kv_len
 *                (used only by the num_splits = 0 policy)
 *   scale      : multiplies q.k
 * Split rule: with c = roundup(ceil(kv_len / S), 16), split s of a sequence
 * covers tokens [s*c, min((s+1)*c, kv_len)); an empty split writes o = 0 and
 * lse = -inf.  Each split's (o, lse) is attention restricted to its tokens.
 * Limits: head_dim in {64, 128, 256}; n_q_heads / n_kv_heads <= 64.
 * Errors: ATTN_ERR_NULL, _SHAPE, _HEADDIM, _GQA, _SPLITS, _ALIGN, _ARCH, _LAUNCH.
 */
int attn_decode_splitkv(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                        const int32_t* block_table, const int32_t* kv_lens, int num_splits,
                        float* o_partial, float* lse_partial, int batch, int n_q_heads,
                        int n_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                        int num_blocks, int max_kv_len, float scale, void* stream);

/*
 * attn_decode_splitkv_ex -- attn_decode_splitkv with the variants of
 * attn_prefill_ex.  The query is the sequence's last token (position
 * kv_len - 1), so a window keeps tokens lo = max(0, kv_len - 1 - window_left)
 * .. kv_len - 1.  With a window the split rule applies to tokens
 * [lo16, kv_len), lo16 = lo rounded down to a multiple of 16: c =
 * roundup(ceil((kv_len - lo16) / S), 16), split s covers [lo16 + s*c,
 * min(lo16 + (s+1)*c, kv_len)), and tokens below lo carry no weight.
 * ALiBi adds -alibi_slopes[h] * (kv_len - 1 - j) to the score of token j.
 */
int attn_decode_splitkv_ex(const attn_bf16* q, const attn_bf16* k_cache,
                           const attn_bf16* v_cache, const int32_t* block_table,
                           const int32_t* kv_lens, int num_splits, float* o_partial,
                           float* lse_partial, int batch, int n_q_heads, int n_kv_heads,
                           int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                           int max_kv_len, float scale, int window_left, float softcap,
                           const float* alibi_slopes, void* stream);

/*
 * attn_decode_splitkv_ex2 -- attn_decode_splitkv_ex with flags.
 *
 * Page: same, section "Decode: a different bottleneck" (the decode is bound
 * by streaming the cache, so the stream should start as early as possible).
 *
 *   flags: 0, or ATTN_DECODE_EARLY_CACHE.  With it, when the call follows
 *          another kernel on the same stream, the decode grid may begin
 *          while that kernel is still running (programmatic dependent
 *          launch): it reads kv_lens and the block table and copies cache
 *          rows into its shared-memory ring before that kernel has finished,
 *          and reads q and alibi_slopes and writes o_partial / lse_partial
 *          only after it.  The CALLER GUARANTEES that the kernel immediately
 *          before the call on the stream writes none of kv_lens, block_table,
 *          k_cache and v_cache (for example: a layer's decode right after the
 *          previous layer's attn_combine, each layer with its own cache).
 *          Results are the same as without the flag.
 * Other arguments, limits and errors as attn_decode_splitkv_ex; unknown flag
 * bits are ATTN_ERR_SHAPE.
 */
#define ATTN_DECODE_EARLY_CACHE 1u
int attn_decode_splitkv_ex2(const attn_bf16* q, const attn_bf16* k_cache,
                            const attn_bf16* v_cache, const int32_t* block_table,
                            const int32_t* kv_lens, int num_splits, float* o_partial,
                            float* lse_partial, int batch, int n_q_heads, int n_kv_heads,
                            int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                            int max_kv_len, float scale, int window_left, float softcap,
                            const float* alibi_slopes, unsigned flags, void* stream);

/*
 * attn_decode_append_splitkv -- split-KV single-token decode that first
 * appends each sequence's new key and value to its cache.
 *
 * Page: same, section "Minimal implementation": the decode call against a
 * paged cache takes the cache, the block table and the per-sequence count of
 * tokens already cached, appends the new keys and values in place, and the
 * caller increments the counts afterwards.
 *
 *   k_new, v_new: (batch, n_kv_heads, head_dim) bf16, the new token's key and
 *                value per sequence, 16-byte aligned
 *   k_cache,
 *   v_cache    : as for attn_decode_splitkv, but WRITTEN: the row of token
 *                kv_lens[b] (all kv heads) receives k_new[b] / v_new[b]; no
 *                other byte of either cache changes
 *   kv_lens    : (batch,) int32 tokens already cached (read, not modified); the
 *                query of sequence b attends over kv_lens[b] + 1 tokens, the
 *                new one last; kv_lens[b] + 1 must not exceed the capacity --
 *                a larger value is flagged, clamped and nothing is written
 *   other arguments, the split rule (applied to kv_lens[b] + 1 tokens), the
 *   partial outputs and the errors are those of attn_decode_splitkv.
 * A block-table entry outside [0, num_blocks) for the new position is flagged
 * and that row is not written.  The call must not overlap, on the device,
 * another call that reads or writes the same cache rows.
 */
int attn_decode_append_splitkv(const attn_bf16* q, const attn_bf16* k_new,
                               const attn_bf16* v_new, attn_bf16* k_cache, attn_bf16* v_cache,
                               const int32_t* block_table, const int32_t* kv_lens,
                               int num_splits, float* o_partial, float* lse_partial, int batch,
                               int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                               int max_blocks_per_seq, int num_blocks, int max_kv_len,
                               float scale, void* stream);

/*
 * attn_decode_append_splitkv_ex -- attn_decode_append_splitkv with the
 * attention variants of attn_decode_splitkv_ex (page: same, sections
 * "Minimal implementation" and "Interaction with post-trained models").
 *
 *   window_left, softcap, alibi_slopes: as attn_decode_splitkv_ex, applied to
 *                the kv_lens[b] + 1 tokens with the new token as the query's
 *                own position kv_lens[b]: a window keeps tokens
 *                kv_lens[b] - window_left .. kv_lens[b]; ALiBi adds
 *                -alibi_slopes[h] * (kv_lens[b] - j).
 * Everything else, the writes and the errors, as attn_decode_append_splitkv and
 * attn_decode_splitkv_ex (ALiBi with soft-capping is ATTN_ERR_SHAPE).
 */
int attn_decode_append_splitkv_ex(const attn_bf16* q, const attn_bf16* k_new,
                                  const attn_bf16* v_new, attn_bf16* k_cache, attn_bf16* v_cache,
                                  const int32_t* block_table, const int32_t* kv_lens,
                                  int num_splits, float* o_partial, float* lse_partial, int batch,
                                  int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int num_blocks, int max_kv_len,
                                  float scale, int window_left, float softcap,
                                  const float* alibi_slopes, void* stream);

/*
 * attn_prefill_fp8 -- causal (or full) prefill on FP8 inputs prepared by
 * attn_quantize_fp8.
 *
 * Page: same, section "Interaction with post-trained models" (FlashAttention-3's
 * FP8 path: block quantisation and incoherent processing) and section "Prefill:
 * tiles, loop order and the tensor cores" for everything else.
 *
 *   q        : (batch, n_q_heads,  seqlen, head_dim) e4m3, 16-byte aligned (rotated
 *              if k is: pass the same signs to attn_quantize_fp8 for both)
 *   k        : (batch, n_kv_heads, seqlen, head_dim) e4m3
 *   v_t      : (batch, n_kv_heads, head_dim, seqlen) e4m3 (transposed)
 *   q_scales : (batch, n_q_heads,  ceil(seqlen/128)) fp32 block scales
 *   k_scales : (batch, n_kv_heads, ceil(seqlen/128)) fp32 block scales
 *   v_scales : (batch, n_kv_heads) fp32 per-head scales
 *   o, lse, scale, causal: as attn_prefill (o is the attention of the
 *              dequantised inputs).  P is rounded to e4m3 for the P V product.
 * Limits: head_dim 64 or 128 (64 runs the 128-column kernel, its copies
 *   reading zeros past the 64 columns: the same time per score as 128);
 *   seqlen a multiple of 16 (the rows of v_t are seqlen bytes); the other
 *   limits of attn_prefill.
 * Errors: ATTN_ERR_NULL, _SHAPE, _HEADDIM, _GQA, _ALIGN, _ARCH, _LAUNCH.
 */
int attn_prefill_fp8(const uint8_t* q, const uint8_t* k, const uint8_t* v_t,
                     const float* q_scales, const float* k_scales, const float* v_scales,
                     float* o, float* lse, int batch, int n_q_heads, int n_kv_heads, int seqlen,
                     int head_dim, float scale, int causal, void* stream);

/*
 * attn_quantize_fp8 -- FP8 (e4m3) block quantisation with optional
 * incoherent processing, the input preparation of attn_prefill_fp8.
 *
 * Page: same, section "Interaction with post-trained models" (FlashAttention-3's
 * FP8 path lowers the error of naive FP8 attention by block quantisation and
 * incoherent processing) and section "The line of work".
 *
 *   x         : (planes, rows, head_dim) bf16, 16-byte aligned
 *   signs     : (head_dim,) fp32 +-1, or NULL.  When given, every row is first
 *               multiplied by diag(signs) H / sqrt(head_dim), H the Sylvester
 *               Hadamard matrix (pass the same signs for Q and K, none for V)
 *   block_rows: 128 -> one scale per block of 128 rows of a plane;
 *               0   -> one scale per plane
 *   codes     : e4m3 output, (planes, rows, head_dim), or with transpose = 1
 *               (planes, head_dim, rows); 16-byte aligned
 *   scales    : fp32 output, (planes, ceil(rows / 128)) or (planes,): each
 *               block's amax / 448; codes = e4m3(x * (448 / amax)), rounded to
 *               nearest, ties to even, saturating (amax 0 counts as 1)
 * Every step is float32 with round-to-nearest: the rotation's butterflies run
 * with stride 1, 2, 4, ..., head_dim/2 and end with one multiply by the
 * float32 value of 1/sqrt(head_dim).
 * Errors: ATTN_ERR_NULL, _SHAPE, _HEADDIM, _ALIGN, _ARCH, _LAUNCH.
 */
int attn_quantize_fp8(const attn_bf16* x, uint8_t* codes, float* scales, const float* signs,
                      int planes, int rows, int head_dim, int block_rows, int transpose,
                      void* stream);

/*
 * attn_quantize_fp8_qkv -- the FP8 inputs of attn_prefill_fp8 for Q, K and V
 * in one call, with fewer launches than three attn_quantize_fp8 calls (Q, K
 * and V's amax in one kernel, then V's codes and scales).
 *
 * Page: same, section "Interaction with post-trained models" (FlashAttention-3's
 * FP8 path: block quantisation and incoherent processing).
 *
 *   q        : (planes_q, rows, head_dim) bf16; k, v: (planes_kv, rows, head_dim) bf16;
 *              16-byte aligned
 *   signs    : (head_dim,) fp32 +-1 for the rotation of q and k, or NULL
 *   q_codes  : (planes_q, rows, head_dim) e4m3;  q_scales: (planes_q, ceil(rows/128)) fp32
 *   k_codes  : (planes_kv, rows, head_dim) e4m3; k_scales: (planes_kv, ceil(rows/128)) fp32
 *   v_codes_t: (planes_kv, head_dim, rows) e4m3; v_scales: (planes_kv,) fp32
 *   codes 16-byte aligned, scales 4-byte aligned
 * The results are bit for bit those of attn_quantize_fp8 on q and on k with
 * block_rows = 128 and these signs, and on v with no rotation, block_rows = 0
 * and transpose = 1.  Limits: planes_q, planes_kv <= 65535; 1 <= rows <= 2^24;
 * head_dim 64 or 128.
 * Errors: ATTN_ERR_NULL, _SHAPE, _HEADDIM, _ALIGN, _ARCH, _LAUNCH.
 */
int attn_quantize_fp8_qkv(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v,
                          uint8_t* q_codes, uint8_t* k_codes, uint8_t* v_codes_t,
                          float* q_scales, float* k_scales, float* v_scales, const float* signs,
                          int planes_q, int planes_kv, int rows, int head_dim, void* stream);

/*
 * attn_quantize_fp8_varlen -- attn_quantize_fp8 with block scales for
 * sequences packed end to end (the Q and K of attn_prefill_fp8_varlen).
 *
 * Page: same, section "Interaction with post-trained models" (packed batches;
 * FP8 block quantisation).  Each sequence is cut into tiles of 128 rows
 * starting at its first row, so that no attention tile straddles two scales;
 * tile t of sequence s gets the scale in column prefix(s) + t, prefix(s) the
 * number of tiles of the sequences before it.
 *   x      : (planes, total_tokens, head_dim) bf16, 16-byte aligned
 *   codes  : (planes, total_tokens, head_dim) e4m3 output, 16-byte aligned; rows
 *            outside every sequence are not written
 *   scales : (planes, ceil(total_tokens / 128) + num_seqs) fp32 output, the
 *            columns past the last tile not written
 *   signs  : as attn_quantize_fp8 (NULL: no rotation)
 *   cu_seqlens, num_seqs: as attn_prefill_varlen (clamped the same way)
 * V takes one scale per head: attn_quantize_fp8 with block_rows 0 and
 * transpose 1 over the packed rows.
 * Limits: head_dim in {64, 128}; 1 <= num_seqs <= 512; 1 <= total_tokens <= 2^24.
 * Errors: ATTN_ERR_NULL, _SHAPE, _HEADDIM, _ALIGN, _ARCH, _LAUNCH.
 */
int attn_quantize_fp8_varlen(const attn_bf16* x, uint8_t* codes, float* scales,
                             const float* signs, const int32_t* cu_seqlens, int num_seqs,
                             int total_tokens, int planes, int head_dim, void* stream);

/*
 * attn_prefill_fp8_varlen -- attn_prefill_fp8 over sequences packed end to
 * end (attn_prefill_varlen's layout and rules).
 *
 * Page: same, sections "Interaction with post-trained models" (packed batches,
 * FP8) and "Prefill: tiles, loop order and the tensor cores".
 *   q, k     : (n_q_heads / n_kv_heads, total_tokens, head_dim) e4m3 from
 *              attn_quantize_fp8_varlen (the same signs for both)
 *   v_t      : (n_kv_heads, head_dim, total_tokens) e4m3 from attn_quantize_fp8
 *              (block_rows 0, transpose 1)
 *   q_scales, k_scales: (planes, ceil(total_tokens / 128) + num_seqs) fp32
 *   v_scales : (n_kv_heads,) fp32
 *   o, lse, cu_seqlens, num_seqs, scale, causal: as attn_prefill_varlen
 * V^T is copied with the tokens along the innermost coordinate, so EVERY
 * NON-EMPTY SEQUENCE MUST START AT A MULTIPLE OF 16 ROWS: otherwise nothing
 * is computed and the launch is flagged (ATTN_ERR_DEVICE from
 * attn_check_device_status), as for a cu_seqlens that breaks its rule.
 * Limits: head_dim 64 or 128 (as attn_prefill_fp8); 1 <= num_seqs <= 512 (one
 * launch: the scale columns are numbered across the whole list); total_tokens
 * a multiple of 16 (16 .. 2^24); the other limits of attn_prefill_varlen.
 * Errors: ATTN_ERR_NULL, _SHAPE, _HEADDIM, _GQA, _ALIGN, _ARCH, _LAUNCH.
 */
int attn_prefill_fp8_varlen(const uint8_t* q, const uint8_t* k, const uint8_t* v_t,
                            const float* q_scales, const float* k_scales, const float* v_scales,
                            float* o, float* lse, const int32_t* cu_seqlens, int num_seqs,
                            int total_tokens, int n_q_heads, int n_kv_heads, int head_dim,
                            float scale, int causal, void* stream);

/*
 * attn_combine -- merge per-split partial results by their LSE weights.
 *
 * Page: same, section "The online softmax, with every symbol defined" (the
 * rule for combining independent partial results: lambda = log sum_k
 * exp(lambda_k), o = sum_k exp(lambda_k - lambda) o_k) and the merge rule in
 * section "Minimal implementation" (a softmax over the split axis).
 *
 *   o_partial  : (num_splits, batch, n_q_heads, head_dim) fp32, 16-byte aligned
 *   lse_partial: (num_splits, batch, n_q_heads) fp32, 4-byte aligned
 *   o          : (batch, n_q_heads, head_dim) fp32 output, 16-byte aligned
 *   lse        : (batch, n_q_heads) fp32 output, 4-byte aligned
 * Splits with lse = -inf carry zero weight; if all are -inf, o = 0, lse = -inf.
 * Limits: 1 <= num_splits <= ATTN_MAX_SPLITS; head_dim in {64, 128, 256}.
 * Errors: ATTN_ERR_NULL, _SHAPE, _HEADDIM, _SPLITS, _ALIGN, _ARCH, _LAUNCH.
 */
int attn_combine(const float* o_partial, const float* lse_partial, int num_splits, int batch,
                 int n_q_heads, int head_dim, float* o, float* lse, void* stream);

/*
 * attn_check_device_status -- synchronises `stream`, then reads and clears the
 * current device's error word.  Returns ATTN_OK, ATTN_ERR_TIMEOUT (a bounded
 * wait gave up), ATTN_ERR_DEVICE (bad block-table entry or kv_len), or
 * ATTN_ERR_LAUNCH (a CUDA error, e.g. from an earlier launch).  Meant for
 * tests and debugging: it blocks the host.
 */
int attn_check_device_status(void* stream);

/*
 * attn_set_wait_timeout_ns -- upper bound, in nanoseconds, on any single
 * kernel-side wait (default 2e9).  Values below 1000 are raised to 1000.
 * One process-wide value, read and written atomically: each launch takes the
 * value current when it is issued, so a change made from another thread
 * applies to the launches issued after it.  Returns the previous value.
 */
uint64_t attn_set_wait_timeout_ns(uint64_t timeout_ns);

/*
 * attn_selftest_bounded_wait -- launches one CTA that waits on a barrier no
 * one arrives at, with the current timeout, then returns the resulting
 * device status (ATTN_ERR_TIMEOUT when the bounded wait works).  Synchronises
 * `stream`.  Exercises the give-up path without faulting or hanging the GPU.
 */
int attn_selftest_bounded_wait(void* stream);

/*
 * attn_decode_noalloc -- split-KV decode and combine in one call, for callers
 * that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point: it is a convenience of
 * this library.  Some callers may not call cudaMalloc on their decode path:
 * a serving loop that reserved all device memory at start-up and forbids
 * later allocations, a plugin inside a host framework that owns the device
 * allocator and only hands it the tensors it needs, or a latency-critical step
 * where cudaMalloc's implicit synchronisation is unacceptable.  Such a caller
 * cannot provide the per-split partial buffers that attn_decode_splitkv
 * writes and attn_combine reads.  This entry point keeps those partials in a
 * fixed buffer of ATTN_NOALLOC_SCRATCH_BYTES compiled into the library (a
 * file-scope device array): every GPU that loads the library holds it until
 * the process exits.  It calls no allocating routine.
 *
 * Arguments are those of attn_decode_splitkv, except that the final results
 * are written directly:
 *   o   : (batch, n_q_heads, head_dim) fp32 output, 16-byte aligned
 *   lse : (batch, n_q_heads) fp32 output (natural log), 4-byte aligned
 * The results equal attn_decode_splitkv followed by attn_combine with the same
 * num_splits (0 = the same policy).
 * Limit: num_splits * batch * n_q_heads * (head_dim + 1) * 4 bytes, with the
 *   output part rounded up to 256 bytes, must fit in ATTN_NOALLOC_SCRATCH_BYTES;
 *   larger requests return ATTN_ERR_SCRATCH and launch nothing.
 * Set-up: the first call on each device looks up the buffer's device address
 *   (cudaGetSymbolAddress, with that device current) and keeps it for the
 *   process; make that first call before any stream capture begins.  A
 *   lookup that fails returns ATTN_ERR_LAUNCH and is tried again by the next
 *   call on that device.
 * Sharing: every call reuses the same buffer, which keeps the previous call's
 *   contents.  Each call overwrites every partial value it later reads, so
 *   nothing needs clearing; but two calls whose kernels overlap on the GPU
 *   (unordered streams, or concurrent host threads) race on the buffer and
 *   give wrong results -- order them on one stream or with events.
 * Errors: those of attn_decode_splitkv, plus ATTN_ERR_SCRATCH.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (8u << 20)
int attn_decode_noalloc(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                        const int32_t* block_table, const int32_t* kv_lens, int num_splits,
                        float* o, float* lse, int batch, int n_q_heads, int n_kv_heads,
                        int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                        int max_kv_len, float scale, void* stream);

/* Library version string, e.g. "0.1.0 sm_103a". */
const char* attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_SM103_H */
