// attn_decode_noalloc: split-KV decode + combine with the split partials kept
// in a fixed device buffer, for callers that cannot allocate device memory
// (see include/attn.h).  It reuses the decode and combine kernels unchanged.
#include <cmath>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "attn.h"
#include "attn_internal.h"

namespace {

constexpr size_t kScratchBytes = ATTN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The partials live here: one copy per device that loads the library, held
// until the process exits.  Host code must not pass this name to a kernel (on
// the host it is only a stand-in); it uses the address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct ScratchAddr {
  std::once_flag once;
  cudaError_t err = cudaErrorUnknown;
  void* ptr = nullptr;
};
ScratchAddr g_addr[kMaxDevices];

// Once per device, with that device current: the buffer's device address.
void* scratch_address(int* status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = ATTN_ERR_LAUNCH;
    return nullptr;
  }
  ScratchAddr& a = g_addr[dev];
  std::call_once(a.once, [&a] {
    a.err = cudaGetSymbolAddress(&a.ptr, g_noalloc_scratch);
  });
  if (a.err != cudaSuccess || a.ptr == nullptr) {
    *status = ATTN_ERR_LAUNCH;
    return nullptr;
  }
  *status = ATTN_OK;
  return a.ptr;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int attn_decode_noalloc(const attn_bf16* q, const attn_bf16* k_cache,
                                   const attn_bf16* v_cache, const int32_t* block_table,
                                   const int32_t* kv_lens, int num_splits, float* o, float* lse,
                                   int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                   int block_size, int max_blocks_per_seq, int num_blocks,
                                   int max_kv_len, float scale, void* stream) {
  if (!q || !k_cache || !v_cache || !kv_lens || !o || !lse) return ATTN_ERR_NULL;
  const bool paged = block_table != nullptr;
  if (batch < 1 || batch > 65535 || n_q_heads < 1 || n_kv_heads < 1 || n_kv_heads > 65535 ||
      max_kv_len < 0 || !std::isfinite(scale) || !(scale > 0.f))
    return ATTN_ERR_SHAPE;
  if (paged && (block_size < 1 || max_blocks_per_seq < 1 || num_blocks < 1 ||
                (long long)block_size * max_blocks_per_seq > (1LL << 30)))
    return ATTN_ERR_SHAPE;
  if (!paged && max_kv_len < 1) return ATTN_ERR_SHAPE;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return ATTN_ERR_HEADDIM;
  if (n_q_heads % n_kv_heads != 0 || n_q_heads / n_kv_heads > 16) return ATTN_ERR_GQA;
  if (num_splits < 0 || num_splits > ATTN_MAX_SPLITS) return ATTN_ERR_SPLITS;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(kv_lens, 4) || (paged && !aligned(block_table, 4)))
    return ATTN_ERR_ALIGN;

  attn::LaunchCtx ctx;
  if (num_splits == 0) {
    const int st = attn::resolve_launch_ctx(stream, &ctx);
    if (st != ATTN_OK) return st;
    num_splits = attn_decode_num_splits(batch, n_kv_heads, max_kv_len, ctx.num_sms);
  }
  // Partial outputs first, then the partial LSEs from the next 256-byte boundary.
  const size_t rows = (size_t)num_splits * (size_t)batch * (size_t)n_q_heads;
  const size_t o_bytes = (rows * (size_t)head_dim * sizeof(float) + 255) / 256 * 256;
  const size_t need = o_bytes + rows * sizeof(float);
  if (need > kScratchBytes) return ATTN_ERR_SCRATCH;

  const int st = attn::resolve_launch_ctx(stream, &ctx);
  if (st != ATTN_OK) return st;
  int sst = ATTN_OK;
  unsigned char* scratch = static_cast<unsigned char*>(scratch_address(&sst));
  if (!scratch) return sst;
  float* o_partial = reinterpret_cast<float*>(scratch);
  float* lse_partial = reinterpret_cast<float*>(scratch + o_bytes);

  attn::DecodeArgs d{q, k_cache, v_cache, block_table, kv_lens, num_splits, o_partial, lse_partial,
                     batch, n_q_heads, n_kv_heads, head_dim, paged ? block_size : 0,
                     paged ? max_blocks_per_seq : 0, paged ? num_blocks : 0, max_kv_len, scale};
  if (attn::launch_decode(d, ctx) != cudaSuccess) return ATTN_ERR_LAUNCH;
  attn::CombineArgs c{o_partial, lse_partial, num_splits, batch, n_q_heads, head_dim, o, lse};
  if (attn::launch_combine(c, ctx) != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}
