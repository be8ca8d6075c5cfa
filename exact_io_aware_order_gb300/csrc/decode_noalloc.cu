// attn_decode_noalloc: split-KV decode + combine with the split partials kept
// in a fixed device buffer, for callers that cannot allocate device memory
// (see include/attn.h).  It reuses the decode and combine kernels unchanged.
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

// Per device: the buffer's device address once a lookup has succeeded.  A
// failed lookup (for example one made while a stream capture forbids it) is
// not remembered: the next call on that device tries again.
struct ScratchAddr {
  std::mutex mu;
  void* ptr = nullptr;
};
ScratchAddr g_addr[kMaxDevices];

// The buffer's device address on the current device, looked up with that
// device current.
void* scratch_address(int* status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = ATTN_ERR_LAUNCH;
    return nullptr;
  }
  ScratchAddr& a = g_addr[dev];
  std::lock_guard<std::mutex> lock(a.mu);
  if (a.ptr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // clear the recorded error: it must not surface at a later CUDA call
      *status = ATTN_ERR_LAUNCH;
      return nullptr;
    }
    a.ptr = p;
  }
  *status = ATTN_OK;
  return a.ptr;
}

}  // namespace

extern "C" int attn_decode_noalloc(const attn_bf16* q, const attn_bf16* k_cache,
                                   const attn_bf16* v_cache, const int32_t* block_table,
                                   const int32_t* kv_lens, int num_splits, float* o, float* lse,
                                   int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                   int block_size, int max_blocks_per_seq, int num_blocks,
                                   int max_kv_len, float scale, void* stream) {
  // The same checks as every other decode entry point (o and lse stand in
  // for the partial outputs they replace).
  const int vst = attn::validate_decode(q, nullptr, nullptr, k_cache, v_cache, block_table,
                                        kv_lens, num_splits, o, lse, batch, n_q_heads, n_kv_heads,
                                        head_dim, block_size, max_blocks_per_seq, num_blocks,
                                        max_kv_len, scale, false, -1, 0.f, nullptr);
  if (vst != ATTN_OK) return vst;
  const bool paged = block_table != nullptr;

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
