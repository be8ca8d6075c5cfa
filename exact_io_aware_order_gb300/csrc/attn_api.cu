// C ABI of the attention library: argument validation, per-device state
// (error word, architecture check) and kernel launches on the caller's stream.
// The operations themselves are defined in include/attn.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "attn.h"
#include "attn_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// One 32-bit error word per device; kernels atomically OR error bits into it.
__device__ uint32_t g_attn_error_word;

struct DeviceState {
  std::once_flag once;
  bool ok = false;         // sm_103 and the symbol address resolved
  bool arch_ok = false;
  uint32_t* err_word = nullptr;
  int num_sms = 0;
};

DeviceState g_dev[kMaxDevices];
std::atomic<uint64_t> g_timeout_ns{2000000000ull};

// Resolves per-device state once per device, with that device current.
DeviceState* device_state(int* status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = ATTN_ERR_LAUNCH;
    return nullptr;
  }
  DeviceState* s = &g_dev[dev];
  std::call_once(s->once, [s, dev] {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return;
    s->num_sms = sms;
    s->arch_ok = (major == 10 && minor == 3);
    if (!s->arch_ok) return;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_error_word) != cudaSuccess) return;
    s->err_word = static_cast<uint32_t*>(p);
    s->ok = true;
  });
  if (!s->arch_ok) {
    *status = ATTN_ERR_ARCH;
    return nullptr;
  }
  if (!s->ok) {
    *status = ATTN_ERR_LAUNCH;
    return nullptr;
  }
  *status = ATTN_OK;
  return s;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

attn::LaunchCtx make_ctx(void* stream, const DeviceState* s) {
  attn::LaunchCtx c;
  c.stream = static_cast<cudaStream_t>(stream);
  c.err_word = s->err_word;
  c.timeout_ns = g_timeout_ns.load();
  c.num_sms = s->num_sms;
  return c;
}

bool valid_scale(float scale) { return std::isfinite(scale) && scale > 0.f; }

bool valid_variant(int window_left, float softcap) {
  return window_left >= -1 && softcap >= 0.f && softcap < 3.0e38f;
}

int split_policy(int batch, int n_kv_heads, int max_kv_len, int num_sms) {
  if (batch <= 0 || n_kv_heads <= 0 || max_kv_len <= 0 || num_sms <= 0) return 1;
  // Two decode CTAs are resident per SM.  One sequence: exactly one full wave
  // of equal chunks.  Several sequences (lengths may differ): about four waves
  // of smaller chunks so the block scheduler can balance long and short ones.
  // Never cut chunks much below 256 tokens (a CTA must stream long enough to
  // hide its start-up), and use one split once (sequence, kv head) pairs
  // already fill the GPU.
  const long long slots = 2LL * num_sms;
  const long long pairs = (long long)batch * n_kv_heads;
  if (pairs >= slots) return 1;
  const long long waves = batch == 1 ? 1 : 4;
  long long splits = (waves * slots + pairs - 1) / pairs;
  const long long max_useful = (max_kv_len + 255) / 256;
  if (splits > max_useful) splits = max_useful;
  if (splits < 1) splits = 1;
  if (splits > ATTN_MAX_SPLITS) splits = ATTN_MAX_SPLITS;
  return static_cast<int>(splits);
}

}  // namespace

namespace attn {
int resolve_launch_ctx(void* stream, LaunchCtx* out) {
  int st = ATTN_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  *out = make_ctx(stream, ds);
  return ATTN_OK;
}

int validate_decode(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                    const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* block_table,
                    const int32_t* kv_lens, int num_splits, const float* o_partial,
                    const float* lse_partial, int batch, int n_q_heads, int n_kv_heads,
                    int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                    int max_kv_len, float scale, bool append, int window_left, float softcap,
                    const float* alibi_slopes) {
  if (!q || !k_cache || !v_cache || !kv_lens || !o_partial || !lse_partial) return ATTN_ERR_NULL;
  if (append && (!k_new || !v_new)) return ATTN_ERR_NULL;
  if (!valid_variant(window_left, softcap)) return ATTN_ERR_SHAPE;
  if (alibi_slopes && softcap > 0.f) return ATTN_ERR_SHAPE;  // not combined
  if (!aligned(alibi_slopes, 4)) return ATTN_ERR_ALIGN;
  if (append && (!aligned(k_new, 16) || !aligned(v_new, 16))) return ATTN_ERR_ALIGN;
  const bool paged = block_table != nullptr;
  if (batch < 1 || batch > 65535 || n_q_heads < 1 || n_kv_heads < 1 || n_kv_heads > 65535 ||
      max_kv_len < 0 || !valid_scale(scale))
    return ATTN_ERR_SHAPE;
  if (paged && (block_size < 1 || max_blocks_per_seq < 1 || num_blocks < 1 ||
                (long long)block_size * max_blocks_per_seq > (1LL << 30)))
    return ATTN_ERR_SHAPE;
  if (!paged && max_kv_len < 1) return ATTN_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return ATTN_ERR_HEADDIM;
  if (n_q_heads % n_kv_heads != 0 || n_q_heads / n_kv_heads > 64) return ATTN_ERR_GQA;
  if (num_splits < 0 || num_splits > ATTN_MAX_SPLITS) return ATTN_ERR_SPLITS;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(o_partial, 16) || !aligned(lse_partial, 4) || !aligned(kv_lens, 4) ||
      (paged && !aligned(block_table, 4)))
    return ATTN_ERR_ALIGN;
  return ATTN_OK;
}
}  // namespace attn

extern "C" {

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_NULL: return "ATTN_ERR_NULL: a required pointer is NULL";
    case ATTN_ERR_SHAPE: return "ATTN_ERR_SHAPE: a size or the scale is out of range";
    case ATTN_ERR_HEADDIM: return "ATTN_ERR_HEADDIM: head_dim not supported by this call (see its limits)";
    case ATTN_ERR_GQA: return "ATTN_ERR_GQA: n_q_heads must be a multiple of n_kv_heads (decode: ratio <= 64)";
    case ATTN_ERR_SPLITS: return "ATTN_ERR_SPLITS: num_splits out of range";
    case ATTN_ERR_ALIGN: return "ATTN_ERR_ALIGN: a pointer is misaligned";
    case ATTN_ERR_ARCH: return "ATTN_ERR_ARCH: the current device is not sm_103 (GB300)";
    case ATTN_ERR_LAUNCH: return "ATTN_ERR_LAUNCH: a CUDA call or kernel launch failed";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: a kernel-side bounded wait gave up";
    case ATTN_ERR_DEVICE: return "ATTN_ERR_DEVICE: a kernel saw a bad block-table entry or kv_len";
    case ATTN_ERR_SCRATCH: return "ATTN_ERR_SCRATCH: the split partials exceed the fixed scratch buffer";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

const char* attn_version(void) { return "0.1.0 sm_103a"; }

uint64_t attn_set_wait_timeout_ns(uint64_t timeout_ns) {
  if (timeout_ns < 1000) timeout_ns = 1000;
  return g_timeout_ns.exchange(timeout_ns);
}

int attn_decode_num_splits(int batch, int n_kv_heads, int max_kv_len, int num_sms) {
  if (num_sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 1;
    }
  }
  return split_policy(batch, n_kv_heads, max_kv_len, num_sms);
}

namespace {

int prefill_impl(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, void* o, float* lse,
                 int batch, int n_q_heads, int n_kv_heads, int seqlen, int head_dim, float scale,
                 int causal, int window_left, float softcap, const float* alibi_slopes,
                 unsigned flags, void* stream) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  if (flags & ~ATTN_PREFILL_OUT_BF16) return ATTN_ERR_SHAPE;
  if (batch < 1 || n_q_heads < 1 || n_kv_heads < 1 || seqlen < 1 || seqlen > (1 << 24) ||
      (long long)batch * n_q_heads > (1LL << 20) || !valid_scale(scale) ||
      !valid_variant(window_left, softcap))
    return ATTN_ERR_SHAPE;
  // work items (query tiles x heads x sequences) are counted in 32 bits
  if ((long long)batch * n_q_heads * ((seqlen + 127) / 128) > 0x7fffffffLL) return ATTN_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return ATTN_ERR_HEADDIM;
  if (n_q_heads % n_kv_heads != 0) return ATTN_ERR_GQA;
  if (alibi_slopes && softcap > 0.f) return ATTN_ERR_SHAPE;  // not combined
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(alibi_slopes, 4))
    return ATTN_ERR_ALIGN;
  int st = ATTN_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  attn::PrefillArgs a{q, k, v, o, lse, batch, n_q_heads, n_kv_heads, seqlen, head_dim, scale,
                      causal ? 1 : 0};
  a.window_left = window_left;
  a.softcap = softcap;
  a.alibi_slopes = alibi_slopes;
  a.o_bf16 = (flags & ATTN_PREFILL_OUT_BF16) ? 1 : 0;
  if (attn::launch_prefill(a, make_ctx(stream, ds)) != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

}  // namespace

int attn_prefill(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, float* o, float* lse,
                 int batch, int n_q_heads, int n_kv_heads, int seqlen, int head_dim, float scale,
                 int causal, void* stream) {
  return prefill_impl(q, k, v, o, lse, batch, n_q_heads, n_kv_heads, seqlen, head_dim, scale,
                      causal, -1, 0.f, nullptr, 0u, stream);
}

int attn_prefill_ex(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, float* o,
                    float* lse, int batch, int n_q_heads, int n_kv_heads, int seqlen, int head_dim,
                    float scale, int causal, int window_left, float softcap,
                    const float* alibi_slopes, void* stream) {
  return prefill_impl(q, k, v, o, lse, batch, n_q_heads, n_kv_heads, seqlen, head_dim, scale,
                      causal, window_left, softcap, alibi_slopes, 0u, stream);
}

int attn_prefill_ex2(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, void* o,
                     float* lse, int batch, int n_q_heads, int n_kv_heads, int seqlen,
                     int head_dim, float scale, int causal, int window_left, float softcap,
                     const float* alibi_slopes, unsigned flags, void* stream) {
  return prefill_impl(q, k, v, o, lse, batch, n_q_heads, n_kv_heads, seqlen, head_dim, scale,
                      causal, window_left, softcap, alibi_slopes, flags, stream);
}

namespace {

int prefill_varlen_impl(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, void* o,
                        float* lse, const int32_t* cu_seqlens, int num_seqs, int total_tokens,
                        int n_q_heads, int n_kv_heads, int head_dim, float scale, int causal,
                        int window_left, float softcap, const float* alibi_slopes, unsigned flags,
                        void* stream) {
  if (!q || !k || !v || !o || !lse || !cu_seqlens) return ATTN_ERR_NULL;
  if (flags & ~ATTN_PREFILL_OUT_BF16) return ATTN_ERR_SHAPE;
  if (num_seqs < 1 || num_seqs > attn::kMaxVarlenSeqsPerCall || n_q_heads < 1 ||
      n_kv_heads < 1 || n_q_heads > (1 << 20) || total_tokens < 1 || total_tokens > (1 << 24) ||
      !valid_scale(scale) || !valid_variant(window_left, softcap))
    return ATTN_ERR_SHAPE;
  if (alibi_slopes && softcap > 0.f) return ATTN_ERR_SHAPE;  // not combined
  // work items (at most total/128 + num_seqs query tiles per head) are counted in 32 bits
  if ((long long)n_q_heads * ((total_tokens + 127) / 128 + num_seqs) > 0x7fffffffLL)
    return ATTN_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return ATTN_ERR_HEADDIM;
  if (n_q_heads % n_kv_heads != 0) return ATTN_ERR_GQA;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(cu_seqlens, 4) || !aligned(alibi_slopes, 4))
    return ATTN_ERR_ALIGN;
  int st = ATTN_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  attn::PrefillArgs a{q, k, v, o, lse, 1, n_q_heads, n_kv_heads, total_tokens, head_dim, scale,
                      causal ? 1 : 0};
  a.window_left = window_left;
  a.softcap = softcap;
  a.alibi_slopes = alibi_slopes;
  a.o_bf16 = (flags & ATTN_PREFILL_OUT_BF16) ? 1 : 0;
  // One launch per slice of at most kMaxVarlenSeqs sequences, in order on the
  // stream: the entries of cu_seqlens are absolute row offsets, so a slice is
  // the same array from its first sequence on.
  const attn::LaunchCtx ctx = make_ctx(stream, ds);
  for (int g = 0; g < num_seqs; g += attn::kMaxVarlenSeqs) {
    a.cu_seqlens = cu_seqlens + g;
    a.num_seqs = std::min(attn::kMaxVarlenSeqs, num_seqs - g);
    a.seq_base = g;
    if (attn::launch_prefill(a, ctx) != cudaSuccess) return ATTN_ERR_LAUNCH;
  }
  return ATTN_OK;
}

}  // namespace

int attn_prefill_varlen(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, float* o,
                        float* lse, const int32_t* cu_seqlens, int num_seqs, int total_tokens,
                        int n_q_heads, int n_kv_heads, int head_dim, float scale, int causal,
                        void* stream) {
  return prefill_varlen_impl(q, k, v, o, lse, cu_seqlens, num_seqs, total_tokens, n_q_heads,
                             n_kv_heads, head_dim, scale, causal, -1, 0.f, nullptr, 0u, stream);
}

int attn_prefill_varlen_ex(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, float* o,
                           float* lse, const int32_t* cu_seqlens, int num_seqs, int total_tokens,
                           int n_q_heads, int n_kv_heads, int head_dim, float scale, int causal,
                           int window_left, float softcap, const float* alibi_slopes,
                           void* stream) {
  return prefill_varlen_impl(q, k, v, o, lse, cu_seqlens, num_seqs, total_tokens, n_q_heads,
                             n_kv_heads, head_dim, scale, causal, window_left, softcap,
                             alibi_slopes, 0u, stream);
}

int attn_prefill_varlen_ex2(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, void* o,
                            float* lse, const int32_t* cu_seqlens, int num_seqs, int total_tokens,
                            int n_q_heads, int n_kv_heads, int head_dim, float scale, int causal,
                            int window_left, float softcap, const float* alibi_slopes,
                            unsigned flags, void* stream) {
  return prefill_varlen_impl(q, k, v, o, lse, cu_seqlens, num_seqs, total_tokens, n_q_heads,
                             n_kv_heads, head_dim, scale, causal, window_left, softcap,
                             alibi_slopes, flags, stream);
}

namespace {

// Launch shared by the plain and the appending decode (validation in
// attn::validate_decode, which attn_decode_noalloc calls too).
int decode_impl(const attn_bf16* q, const attn_bf16* k_new, const attn_bf16* v_new,
                const attn_bf16* k_cache, const attn_bf16* v_cache, const int32_t* block_table,
                const int32_t* kv_lens, int num_splits, float* o_partial, float* lse_partial,
                int batch, int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                int max_blocks_per_seq, int num_blocks, int max_kv_len, float scale,
                void* stream, bool append, int window_left = -1, float softcap = 0.f,
                const float* alibi_slopes = nullptr, unsigned flags = 0u) {
  if ((flags & ~ATTN_DECODE_EARLY_CACHE) != 0u || (append && flags != 0u)) return ATTN_ERR_SHAPE;
  const int vst = attn::validate_decode(q, k_new, v_new, k_cache, v_cache, block_table, kv_lens,
                                        num_splits, o_partial, lse_partial, batch, n_q_heads,
                                        n_kv_heads, head_dim, block_size, max_blocks_per_seq,
                                        num_blocks, max_kv_len, scale, append, window_left,
                                        softcap, alibi_slopes);
  if (vst != ATTN_OK) return vst;
  const bool paged = block_table != nullptr;
  int st = ATTN_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  if (num_splits == 0) num_splits = split_policy(batch, n_kv_heads, max_kv_len, ds->num_sms);
  attn::DecodeArgs a{q, k_cache, v_cache, block_table, kv_lens, num_splits, o_partial, lse_partial,
                     batch, n_q_heads, n_kv_heads, head_dim, paged ? block_size : 0,
                     paged ? max_blocks_per_seq : 0, paged ? num_blocks : 0, max_kv_len, scale};
  if (append) {
    a.k_new = k_new;
    a.v_new = v_new;
  }
  a.window_left = window_left;
  a.softcap = softcap;
  a.alibi_slopes = alibi_slopes;
  a.early_cache = (flags & ATTN_DECODE_EARLY_CACHE) ? 1 : 0;
  if (attn::launch_decode(a, make_ctx(stream, ds)) != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

}  // namespace

int attn_decode_splitkv(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                        const int32_t* block_table, const int32_t* kv_lens, int num_splits,
                        float* o_partial, float* lse_partial, int batch, int n_q_heads,
                        int n_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                        int num_blocks, int max_kv_len, float scale, void* stream) {
  return decode_impl(q, nullptr, nullptr, k_cache, v_cache, block_table, kv_lens, num_splits,
                     o_partial, lse_partial, batch, n_q_heads, n_kv_heads, head_dim, block_size,
                     max_blocks_per_seq, num_blocks, max_kv_len, scale, stream, false);
}

int attn_decode_splitkv_ex(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                           const int32_t* block_table, const int32_t* kv_lens, int num_splits,
                           float* o_partial, float* lse_partial, int batch, int n_q_heads,
                           int n_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                           int num_blocks, int max_kv_len, float scale, int window_left,
                           float softcap, const float* alibi_slopes, void* stream) {
  return decode_impl(q, nullptr, nullptr, k_cache, v_cache, block_table, kv_lens, num_splits,
                     o_partial, lse_partial, batch, n_q_heads, n_kv_heads, head_dim, block_size,
                     max_blocks_per_seq, num_blocks, max_kv_len, scale, stream, false, window_left,
                     softcap, alibi_slopes);
}

int attn_decode_splitkv_ex2(const attn_bf16* q, const attn_bf16* k_cache,
                            const attn_bf16* v_cache, const int32_t* block_table,
                            const int32_t* kv_lens, int num_splits, float* o_partial,
                            float* lse_partial, int batch, int n_q_heads, int n_kv_heads,
                            int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                            int max_kv_len, float scale, int window_left, float softcap,
                            const float* alibi_slopes, unsigned flags, void* stream) {
  return decode_impl(q, nullptr, nullptr, k_cache, v_cache, block_table, kv_lens, num_splits,
                     o_partial, lse_partial, batch, n_q_heads, n_kv_heads, head_dim, block_size,
                     max_blocks_per_seq, num_blocks, max_kv_len, scale, stream, false, window_left,
                     softcap, alibi_slopes, flags);
}

int attn_decode_append_splitkv(const attn_bf16* q, const attn_bf16* k_new, const attn_bf16* v_new,
                               attn_bf16* k_cache, attn_bf16* v_cache, const int32_t* block_table,
                               const int32_t* kv_lens, int num_splits, float* o_partial,
                               float* lse_partial, int batch, int n_q_heads, int n_kv_heads,
                               int head_dim, int block_size, int max_blocks_per_seq,
                               int num_blocks, int max_kv_len, float scale, void* stream) {
  return decode_impl(q, k_new, v_new, k_cache, v_cache, block_table, kv_lens, num_splits,
                     o_partial, lse_partial, batch, n_q_heads, n_kv_heads, head_dim, block_size,
                     max_blocks_per_seq, num_blocks, max_kv_len, scale, stream, true);
}

int attn_decode_append_splitkv_ex(const attn_bf16* q, const attn_bf16* k_new,
                                  const attn_bf16* v_new, attn_bf16* k_cache, attn_bf16* v_cache,
                                  const int32_t* block_table, const int32_t* kv_lens,
                                  int num_splits, float* o_partial, float* lse_partial, int batch,
                                  int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int num_blocks, int max_kv_len,
                                  float scale, int window_left, float softcap,
                                  const float* alibi_slopes, void* stream) {
  return decode_impl(q, k_new, v_new, k_cache, v_cache, block_table, kv_lens, num_splits,
                     o_partial, lse_partial, batch, n_q_heads, n_kv_heads, head_dim, block_size,
                     max_blocks_per_seq, num_blocks, max_kv_len, scale, stream, true, window_left,
                     softcap, alibi_slopes);
}

int attn_combine(const float* o_partial, const float* lse_partial, int num_splits, int batch,
                 int n_q_heads, int head_dim, float* o, float* lse, void* stream) {
  if (!o_partial || !lse_partial || !o || !lse) return ATTN_ERR_NULL;
  if (batch < 1 || n_q_heads < 1 || (long long)batch * n_q_heads > (1LL << 31) - 1)
    return ATTN_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return ATTN_ERR_HEADDIM;
  if (num_splits < 1 || num_splits > ATTN_MAX_SPLITS) return ATTN_ERR_SPLITS;
  if (!aligned(o_partial, 16) || !aligned(lse_partial, 4) || !aligned(o, 16) || !aligned(lse, 4))
    return ATTN_ERR_ALIGN;
  int st = ATTN_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  attn::CombineArgs a{o_partial, lse_partial, num_splits, batch, n_q_heads, head_dim, o, lse};
  if (attn::launch_combine(a, make_ctx(stream, ds)) != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

int attn_prefill_fp8(const uint8_t* q, const uint8_t* k, const uint8_t* v_t,
                     const float* q_scales, const float* k_scales, const float* v_scales,
                     float* o, float* lse, int batch, int n_q_heads, int n_kv_heads, int seqlen,
                     int head_dim, float scale, int causal, void* stream) {
  if (!q || !k || !v_t || !q_scales || !k_scales || !v_scales || !o || !lse) return ATTN_ERR_NULL;
  if (batch < 1 || n_q_heads < 1 || n_kv_heads < 1 || seqlen < 16 || seqlen > (1 << 24) ||
      seqlen % 16 != 0 || (long long)batch * n_q_heads > (1LL << 20) || !valid_scale(scale))
    return ATTN_ERR_SHAPE;  // v_t rows are seqlen bytes: a multiple of 16 for the copies
  if ((long long)batch * n_q_heads * ((seqlen + 127) / 128) > 0x7fffffffLL) return ATTN_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return ATTN_ERR_HEADDIM;
  if (n_q_heads % n_kv_heads != 0) return ATTN_ERR_GQA;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v_t, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(q_scales, 4) || !aligned(k_scales, 4) || !aligned(v_scales, 4))
    return ATTN_ERR_ALIGN;
  int st = ATTN_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  attn::PrefillArgs a{reinterpret_cast<const uint16_t*>(q), reinterpret_cast<const uint16_t*>(k),
                      reinterpret_cast<const uint16_t*>(v_t), o, lse, batch, n_q_heads,
                      n_kv_heads, seqlen, head_dim, scale, causal ? 1 : 0};
  a.fp8 = 1;
  a.q_scales = q_scales;
  a.k_scales = k_scales;
  a.v_scales = v_scales;
  if (attn::launch_prefill(a, make_ctx(stream, ds)) != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

int attn_quantize_fp8(const attn_bf16* x, uint8_t* codes, float* scales, const float* signs,
                      int planes, int rows, int head_dim, int block_rows, int transpose,
                      void* stream) {
  if (!x || !codes || !scales) return ATTN_ERR_NULL;
  if (planes < 1 || planes > 65535 || rows < 1 || rows > (1 << 24) ||
      (block_rows != 0 && block_rows != 128) || (transpose != 0 && transpose != 1))
    return ATTN_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return ATTN_ERR_HEADDIM;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 4) || !aligned(signs, 4))
    return ATTN_ERR_ALIGN;
  int st = ATTN_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  attn::QuantArgs a{x, codes, scales, signs, planes, rows, head_dim, block_rows, transpose,
                    static_cast<float>(1.0 / std::sqrt(static_cast<double>(head_dim)))};
  if (attn::launch_quantize(a, make_ctx(stream, ds)) != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

int attn_prefill_fp8_varlen(const uint8_t* q, const uint8_t* k, const uint8_t* v_t,
                            const float* q_scales, const float* k_scales, const float* v_scales,
                            float* o, float* lse, const int32_t* cu_seqlens, int num_seqs,
                            int total_tokens, int n_q_heads, int n_kv_heads, int head_dim,
                            float scale, int causal, void* stream) {
  if (!q || !k || !v_t || !q_scales || !k_scales || !v_scales || !o || !lse || !cu_seqlens)
    return ATTN_ERR_NULL;
  if (num_seqs < 1 || num_seqs > attn::kMaxVarlenSeqs || n_q_heads < 1 || n_kv_heads < 1 ||
      n_q_heads > (1 << 20) || total_tokens < 16 || total_tokens > (1 << 24) ||
      total_tokens % 16 != 0 || !valid_scale(scale))
    return ATTN_ERR_SHAPE;  // v_t rows are total_tokens bytes: a multiple of 16 for the copies
  if ((long long)n_q_heads * ((total_tokens + 127) / 128 + num_seqs) > 0x7fffffffLL)
    return ATTN_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return ATTN_ERR_HEADDIM;
  if (n_q_heads % n_kv_heads != 0) return ATTN_ERR_GQA;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v_t, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(q_scales, 4) || !aligned(k_scales, 4) ||
      !aligned(v_scales, 4) || !aligned(cu_seqlens, 4))
    return ATTN_ERR_ALIGN;
  int st = ATTN_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  attn::PrefillArgs a{reinterpret_cast<const uint16_t*>(q), reinterpret_cast<const uint16_t*>(k),
                      reinterpret_cast<const uint16_t*>(v_t), o, lse, 1, n_q_heads, n_kv_heads,
                      total_tokens, head_dim, scale, causal ? 1 : 0};
  a.cu_seqlens = cu_seqlens;
  a.num_seqs = num_seqs;
  a.fp8 = 1;
  a.q_scales = q_scales;
  a.k_scales = k_scales;
  a.v_scales = v_scales;
  if (attn::launch_prefill(a, make_ctx(stream, ds)) != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

int attn_quantize_fp8_varlen(const attn_bf16* x, uint8_t* codes, float* scales,
                             const float* signs, const int32_t* cu_seqlens, int num_seqs,
                             int total_tokens, int planes, int head_dim, void* stream) {
  if (!x || !codes || !scales || !cu_seqlens) return ATTN_ERR_NULL;
  if (planes < 1 || planes > 65535 || num_seqs < 1 || num_seqs > attn::kMaxVarlenSeqs ||
      total_tokens < 1 || total_tokens > (1 << 24))
    return ATTN_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return ATTN_ERR_HEADDIM;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 4) || !aligned(signs, 4) ||
      !aligned(cu_seqlens, 4))
    return ATTN_ERR_ALIGN;
  int st = ATTN_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  attn::QuantArgs a{x, codes, scales, signs, planes, total_tokens, head_dim, 128, 0,
                    static_cast<float>(1.0 / std::sqrt(static_cast<double>(head_dim)))};
  a.cu_seqlens = cu_seqlens;
  a.num_seqs = num_seqs;
  a.tiles = (total_tokens + 127) / 128 + num_seqs;
  if (attn::launch_quantize(a, make_ctx(stream, ds)) != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

int attn_quantize_fp8_qkv(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v,
                          uint8_t* q_codes, uint8_t* k_codes, uint8_t* v_codes_t,
                          float* q_scales, float* k_scales, float* v_scales, const float* signs,
                          int planes_q, int planes_kv, int rows, int head_dim, void* stream) {
  if (!q || !k || !v || !q_codes || !k_codes || !v_codes_t || !q_scales || !k_scales ||
      !v_scales)
    return ATTN_ERR_NULL;
  if (planes_q < 1 || planes_q > 65535 || planes_kv < 1 || planes_kv > 65535 || rows < 1 ||
      rows > (1 << 24) ||
      (long long)(planes_q + 2LL * planes_kv) * ((rows + 127) / 128) > 0x7fffffffLL)
    return ATTN_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128) return ATTN_ERR_HEADDIM;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q_codes, 16) ||
      !aligned(k_codes, 16) || !aligned(v_codes_t, 16) || !aligned(q_scales, 4) ||
      !aligned(k_scales, 4) || !aligned(v_scales, 4) || !aligned(signs, 4))
    return ATTN_ERR_ALIGN;
  int st = ATTN_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  const float inv = static_cast<float>(1.0 / std::sqrt(static_cast<double>(head_dim)));
  attn::QuantArgs aq{q, q_codes, q_scales, signs, planes_q, rows, head_dim, 128, 0, inv};
  attn::QuantArgs ak{k, k_codes, k_scales, signs, planes_kv, rows, head_dim, 128, 0, inv};
  attn::QuantArgs av{v, v_codes_t, v_scales, nullptr, planes_kv, rows, head_dim, 0, 1, inv};
  if (attn::launch_quantize_qkv(aq, ak, av, make_ctx(stream, ds)) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

int attn_check_device_status(void* stream) {
  int st = ATTN_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_LAUNCH;
  uint32_t word = 0;
  if (cudaMemcpy(&word, ds->err_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  if (word != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(ds->err_word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
  }
  if (word & attn::kErrTimeout) return ATTN_ERR_TIMEOUT;
  if (word) return ATTN_ERR_DEVICE;
  return ATTN_OK;
}

int attn_selftest_bounded_wait(void* stream) {
  int st = ATTN_OK;
  DeviceState* ds = device_state(&st);
  if (!ds) return st;
  if (attn::launch_wait_selftest(make_ctx(stream, ds)) != cudaSuccess) return ATTN_ERR_LAUNCH;
  return attn_check_device_status(stream);
}

}  // extern "C"
