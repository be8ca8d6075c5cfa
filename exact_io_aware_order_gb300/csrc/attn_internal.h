// Internal launch interface shared by the C-ABI layer and the kernel files.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace attn {

// Device error word bits (read back and cleared by attn_check_device_status).
constexpr uint32_t kErrTimeout = 1u;     // a bounded wait gave up
constexpr uint32_t kErrBlockIndex = 2u;  // a block-table entry outside [0, num_blocks)
constexpr uint32_t kErrKvLen = 4u;       // a kv_len outside [0, capacity]
constexpr uint32_t kErrSeqLens = 8u;     // cu_seqlens not increasing within [0, total]

struct LaunchCtx {
  cudaStream_t stream;
  uint32_t* err_word;   // device address of this device's error word
  uint64_t timeout_ns;  // bound on any single kernel-side wait
  int num_sms;
};

struct PrefillArgs {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  void* o;     // fp32, or bf16 with o_bf16
  float* lse;
  int batch, n_q_heads, n_kv_heads, seqlen, head_dim;
  float scale;
  int causal;
  // Packed variable-length mode: when set, batch is 1, seqlen is the total
  // of packed rows and sequence s occupies rows [cu_seqlens[s], cu_seqlens[s+1]).
  const int32_t* cu_seqlens = nullptr;
  int num_seqs = 0;
  int seq_base = 0;  // index of cu_seqlens[0] in the caller's list (0: its start)
  int o_bf16 = 0;    // O written as bf16 (O / l in fp32, rounded once) instead of fp32
  // Variants: a sliding window (row i sees keys j >= i - window_left; -1 =
  // none) and logit soft-capping (s -> softcap * tanh(s / softcap); 0 = off).
  int window_left = -1;
  float softcap = 0.f;
  const float* alibi_slopes = nullptr;  // (n_q_heads,): adds -slope_h * |i - j|
  // FP8 inputs: q, k are e4m3 (planes, seqlen, head_dim), v e4m3 transposed
  // (planes, head_dim, seqlen); their dequantisation scales per 128-row block
  // (q, k) and per head (v).
  int fp8 = 0;
  const float* q_scales = nullptr;
  const float* k_scales = nullptr;
  const float* v_scales = nullptr;
};

// Packed sequences per prefill launch (the kernel keeps a table per sequence
// in shared memory); a bf16 packed prefill runs longer lists as one launch per
// slice of at most this many, up to kMaxVarlenSeqsPerCall.  The FP8 packed
// prefill and its quantiser number their scale columns across the whole list
// and take one launch, so at most kMaxVarlenSeqs.
constexpr int kMaxVarlenSeqs = 512;
constexpr int kMaxVarlenSeqsPerCall = 1 << 20;

struct DecodeArgs {
  const uint16_t* q;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  const int32_t* block_table;
  const int32_t* kv_lens;
  int num_splits;
  float* o_partial;
  float* lse_partial;
  int batch, n_q_heads, n_kv_heads, head_dim;
  int block_size, max_blocks_per_seq, num_blocks, max_kv_len;
  float scale;
  // Decode with append: when set, each sequence's new key / value row
  // ((batch, n_kv_heads, head_dim) bf16) is written into the cache at
  // position kv_lens[b] and attended together with the cached tokens.  The
  // caches are then written, so the entry point that sets these takes
  // writable cache pointers.
  const uint16_t* k_new = nullptr;
  const uint16_t* v_new = nullptr;
  // Variants, as for prefill; the query is the sequence's last token, so the
  // window keeps tokens kv_len - 1 - window_left .. kv_len - 1.
  int window_left = -1;
  float softcap = 0.f;
  const float* alibi_slopes = nullptr;  // (n_q_heads,): adds -slope_h * (kv_len - 1 - j)
  // Early cache streaming (never with append): kv_lens, the block table and
  // the cache are read, and the ring filled, before the wait for the previous
  // grid on the stream; q and the slopes are read and the partials written
  // after it.
  int early_cache = 0;
};

struct CombineArgs {
  const float* o_partial;
  const float* lse_partial;
  int num_splits, batch, n_q_heads, head_dim;
  float* o;
  float* lse;
};

struct QuantArgs {
  const uint16_t* x;    // (planes, rows, head_dim) bf16
  uint8_t* codes;       // (planes, rows, head_dim) or, transposed, (planes, head_dim, rows) e4m3
  float* scales;        // (planes, ceil(rows / 128)) or (planes,) when block_rows == 0
  const float* signs;   // (head_dim,) +-1 for the rotation, or null
  int planes, rows, head_dim;
  int block_rows;       // 128: one scale per 128 rows; 0: one scale per plane
  int transpose;
  float inv_sqrt_d;     // float32 value of 1 / sqrt(head_dim)
  // Packed sequences (block scales only): sequence s is rows [cu[s], cu[s+1]);
  // its tiles of 128 rows start at its first row and tile t's scale is column
  // prefix[s] + t of a (planes, tiles) array (prefix: tiles of the earlier
  // sequences).
  const int32_t* cu_seqlens = nullptr;
  int num_seqs = 0;
  int tiles = 0;        // columns of the scale array: ceil(rows / 128) + num_seqs
};

// Each returns cudaSuccess or the launch error.  Arguments are already
// validated by the caller.
cudaError_t launch_prefill(const PrefillArgs& a, const LaunchCtx& ctx);
cudaError_t launch_decode(const DecodeArgs& a, const LaunchCtx& ctx);
cudaError_t launch_combine(const CombineArgs& a, const LaunchCtx& ctx);
cudaError_t launch_wait_selftest(const LaunchCtx& ctx);
cudaError_t launch_quantize(const QuantArgs& a, const LaunchCtx& ctx);
// Q and K with block scales (128 rows), V with one scale per plane and
// transposed; the three share rows and head_dim.
cudaError_t launch_quantize_qkv(const QuantArgs& q, const QuantArgs& k, const QuantArgs& v,
                                const LaunchCtx& ctx);

// Resolves the current device's launch context (architecture check, error
// word, SM count) for a call on `stream`; returns an attn_status code.
int resolve_launch_ctx(void* stream, LaunchCtx* out);

// Validation of a split-KV decode request, shared by every decode entry
// point: pointers (o_partial / lse_partial stand for whatever the entry
// point writes its per-split or final results to), shapes, GQA ratio, split
// count, variants and alignment.  Returns an attn_status code; launches
// nothing and touches no device state.
int validate_decode(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                    const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* block_table,
                    const int32_t* kv_lens, int num_splits, const float* o_partial,
                    const float* lse_partial, int batch, int n_q_heads, int n_kv_heads,
                    int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                    int max_kv_len, float scale, bool append, int window_left, float softcap,
                    const float* alibi_slopes);

// Split rule shared by the decode kernel's documentation and the host:
// c = roundup(ceil(len / S), 16); split s covers [s*c, min((s+1)*c, len)).
constexpr int kSplitGranule = 16;

}  // namespace attn
