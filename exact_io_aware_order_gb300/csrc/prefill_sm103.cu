// Causal (or full) prefill attention forward, sm_103a: TMA + tcgen05 + TMEM.
//
// Page "FlashAttention for inference: tiled prefill and split-KV decoding",
// section "Prefill: tiles, loop order and the tensor cores": the outer,
// parallel loop runs over (sequence, head, query tile); each block loads its
// query tile once, streams key/value tiles up to the causal limit through
// on-chip memory, computes S = Q_i K_j^T * scale on the tensor cores (masking
// only the diagonal tile), updates the running max m and sum l with the
// correction c = exp(m_old - m_new) (section "The online softmax, with every
// symbol defined"), accumulates acc = c*acc + P V_j on the tensor cores, and
// finally writes O_i = acc / l and the row log-sum-exp m + log l.  Tiles
// strictly above the diagonal are never visited.
//
// GB300 design (the pages' A100/H100 kernels are prior art only):
//   * one CTA owns two 128-row query tiles (Q0, Q1) of one head; K/V tiles are
//     128 keys; K and V each have a 2-stage shared-memory ring fed by TMA
//     (128-byte swizzle, 3-D tensor maps so rows past the end read as zero);
//   * warp 8 is the TMA producer, warp 9 issues tcgen05.mma from one thread;
//     warps 0-3 / 4-7 run the softmax of Q0 / Q1, one query row per thread
//     (TMEM lane = row), so row max and row sum need no shuffles;
//   * TMEM (512 columns): S0 | S1 | O0 | O1.  P is written as bf16 over the
//     first half of its S columns and fed to the P V product straight from
//     TMEM (A operand in tensor memory), V from shared memory (MN-major);
//   * issue order S0(0), S1(0), then per key tile PV0(j), S0(j+1), PV1(j),
//     S1(j+1): the tensor core computes one tile's products while the other
//     tile's softmax runs (the overlap idea of FlashAttention-3, rebuilt
//     around tcgen05's single-thread issue and commit-to-mbarrier);
//   * base-2 exponentials with scale*log2(e) folded in; O is rescaled only
//     when a row max grows by more than 2^8 (the same stale max is used for
//     l and O, so the result is exact); the LSE is converted back to natural
//     log at the end.
//   * every wait is bounded; on a timeout all roles leave their loops, the
//     CTA waits for in-flight copies and MMAs, frees TMEM and exits.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;                 // rows per query tile
constexpr int kBN = 128;                 // keys per key/value tile
constexpr int kThreads = 320;            // 10 warps
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when max grows > 2^8

template <int D>
struct PrefillSmem {
  static constexpr int kTileBytes = 128 * D * 2;       // one Q, K or V tile
  static constexpr int kChunkBytes = 128 * 128;        // 128 rows x 64 bf16 (one swizzle span)
  static constexpr int kQ0 = 0;
  static constexpr int kQ1 = kTileBytes;
  static constexpr int kK = 2 * kTileBytes;            // 2 stages
  static constexpr int kV = 4 * kTileBytes;            // 2 stages
  static constexpr int kBar = 6 * kTileBytes;
  // barriers: q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2],
  // o_full[2], drain
  static constexpr int kNumBars = 16;
  static constexpr int kMisc = kBar + kNumBars * 8;    // tmem base, abort flag
  static constexpr int kUsed = kMisc + 16;
  // Ask for enough shared memory that two CTAs never share an SM (each
  // allocates all 512 TMEM columns).
  static constexpr int kAlloc = (kUsed + 1024) > 120 * 1024 ? (kUsed + 1024) : 120 * 1024;
};

enum BarId {
  kQFull = 0, kKFull = 1, kKEmpty = 3, kVFull = 5, kVEmpty = 7, kSFull = 9, kPFull = 11, kOFull = 13,
  kDrain = 15
};

struct PrefillParams {
  float* o;
  float* lse;
  int batch, n_q_heads, n_kv_heads, seqlen;
  float sl2;  // scale * log2(e)
  int causal;
  int n_row_blocks;  // ceil(seqlen / 256)
  uint32_t* err_word;
  uint64_t timeout_ns;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using L = PrefillSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item: longest causal rows first; adjacent CTAs share kv heads ----
  const int BH = p.batch * p.n_q_heads;
  const int rb = p.n_row_blocks - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int bidx = bh / p.n_q_heads, h = bh % p.n_q_heads;
  const int kvh = h / (p.n_q_heads / p.n_kv_heads);
  const int N = p.seqlen;
  const int n_kv_tiles_all = (N + kBN - 1) / kBN;
  // Query tile t covers rows [qa + t*128, +128) and visits nt_t key tiles.
  const int qa = rb * 2 * kBM, qb = qa + kBM;
  const int nt0 = p.causal ? (qa / kBN + 1) : n_kv_tiles_all;
  const int nt1 = qb >= N ? 0 : (p.causal ? (qb / kBN + 1) : n_kv_tiles_all);
  const int J = max(nt0, nt1);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kMisc + 4);

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bar(kQFull), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kKFull + i), 1);
      mbar_init(bar(kKEmpty + i), 1);
      mbar_init(bar(kVFull + i), 1);
      mbar_init(bar(kVEmpty + i), 1);
      mbar_init(bar(kSFull + i), 1);
      mbar_init(bar(kPFull + i), 4 * 32);
      mbar_init(bar(kOFull + i), 1);
    }
    mbar_init(bar(kDrain), 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S0 [0,128) | S1 [128,256) | O0 [256,256+D) | O1 [256+D, 256+2D)
  auto tS = [tmem](int t) { return tmem + (t ? 128u : 0u); };
  auto tO = [tmem](int t) { return tmem + 256u + (t ? (uint32_t)D : 0u); };
  const WaitCtl ctl{abort_flag, p.err_word, p.timeout_ns};
  const int zq = bidx * p.n_q_heads + h;      // Q / O tensor-map "plane"
  const int zk = bidx * p.n_kv_heads + kvh;   // K / V tensor-map plane

  if (warp == kProducerWarp) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      const uint32_t qbytes = (nt1 > 0 ? 2u : 1u) * (uint32_t)L::kTileBytes;
      mbar_arrive_expect_tx(bar(kQFull), qbytes);
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem_u32(smem + L::kQ0 + c * L::kChunkBytes), &tm_q, bar(kQFull), c * 64, qa, zq);
      if (nt1 > 0)
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem_u32(smem + L::kQ1 + c * L::kChunkBytes), &tm_q, bar(kQFull), c * 64, qb, zq);
      int nk = 0, nv = 0;  // K / V tiles issued
      for (int j = 0; j < J; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(bar(kKEmpty + st), ((j >> 1) - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(bar(kKFull + st), L::kTileBytes);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem_u32(smem + L::kK + st * L::kTileBytes + c * L::kChunkBytes), &tm_k,
                      bar(kKFull + st), c * 64, j * kBN, zk);
        ++nk;
        if (j >= 2 && !mbar_wait(bar(kVEmpty + st), ((j >> 1) - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(bar(kVFull + st), L::kTileBytes);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem_u32(smem + L::kV + st * L::kTileBytes + c * L::kChunkBytes), &tm_v,
                      bar(kVFull + st), c * 64, j * kBN, zk);
        ++nv;
      }
      if (*abort_flag) {
        // Let copies already in flight land before the CTA's memory is released.
        volatile uint32_t no_abort = 0u;
        WaitCtl drain{&no_abort, p.err_word, p.timeout_ns};
        mbar_wait(bar(kQFull), 0, drain);
        for (int j = max(0, nk - 2); j < nk; ++j) mbar_wait(bar(kKFull + (j & 1)), (j >> 1) & 1, drain);
        for (int j = max(0, nv - 2); j < nv; ++j) mbar_wait(bar(kVFull + (j & 1)), (j >> 1) & 1, drain);
      }
    }
  } else if (warp == kMmaWarp) {
    // ============================ MMA issuer ============================
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(kBM, kBN, false, false);  // Q, K both K-major
      const uint32_t id_pv = idesc_bf16_f32(kBM, D, false, true);    // V is MN-major
      const uint32_t sQ0 = smem_u32(smem + L::kQ0), sQ1 = smem_u32(smem + L::kQ1);
      const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);
      bool ok = mbar_wait(bar(kQFull), 0, ctl);
      tc_fence_after();
      auto first_user = [&](int j) { return j < nt0 ? 0 : 1; };
      auto last_user = [&](int j) { return j < nt1 ? 1 : 0; };
      auto issue_s = [&](int t, int j) -> bool {
        const int st = j & 1;
        if (first_user(j) == t) {
          if (!mbar_wait(bar(kKFull + st), (j >> 1) & 1, ctl)) return false;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
          mma_ss(tS(t), smem_desc_sw128((t ? sQ1 : sQ0) + off, 16, 1024),
                 smem_desc_sw128(sK + st * L::kTileBytes + off, 16, 1024), id_s, kk > 0);
        }
        mma_commit(bar(kSFull + t));
        if (last_user(j) == t) mma_commit(bar(kKEmpty + st));
        return true;
      };
      auto issue_pv = [&](int t, int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait(bar(kPFull + t), j & 1, ctl)) return false;
        tc_fence_after();
        if (first_user(j) == t) {
          if (!mbar_wait(bar(kVFull + st), (j >> 1) & 1, ctl)) return false;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // B = V tile rows [16kk, 16kk+16): 16 rows x 128 B per k step; the
          // 64-column halves of the head dimension are one chunk apart.
          const uint64_t bdesc =
              smem_desc_sw128(sV + st * L::kTileBytes + kk * 16 * 128, L::kChunkBytes, 1024);
          mma_ts(tO(t), tS(t) + kk * 8, bdesc, id_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        if (last_user(j) == t) mma_commit(bar(kVEmpty + st));
        if (j == (t ? nt1 : nt0) - 1) mma_commit(bar(kOFull + t));
        return true;
      };
      if (ok) ok = issue_s(0, 0);
      if (ok && nt1 > 0) ok = issue_s(1, 0);
      for (int j = 0; ok && j < J; ++j) {
        if (j < nt0) {
          ok = issue_pv(0, j);
          if (ok && j + 1 < nt0) ok = issue_s(0, j + 1);
        }
        if (ok && j < nt1) {
          ok = issue_pv(1, j);
          if (ok && j + 1 < nt1) ok = issue_s(1, j + 1);
        }
      }
      // Before TMEM can be freed every issued MMA must have finished (also on
      // the abort path): one more commit on a barrier of its own, then wait.
      mma_commit(bar(kDrain));
      volatile uint32_t no_abort = 0u;
      WaitCtl drain{&no_abort, p.err_word, p.timeout_ns};
      mbar_wait(bar(kDrain), 0, drain);
    }
    __syncwarp();
  } else {
    // ============================ softmax warps ============================
    const int t = warp >> 2;                        // query tile of this warpgroup
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int row = (warp & 3) * 32 + lane;         // row within the tile (= TMEM lane)
    const int q0 = t ? qb : qa;
    const int n_my = t ? nt1 : nt0;
    const uint32_t tSm = tS(t) + lane_base, tOm = tO(t) + lane_base;
    const int q_row = q0 + row;
    const float sl2 = p.sl2;
    float m = -INFINITY, l = 0.f;
    bool ok = n_my > 0;
    for (int j = 0; ok && j < n_my; ++j) {
      if (!mbar_wait_warp(bar(kSFull + t), j & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      float s[kBN];
      {
        uint32_t r[32];
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) {
          tmem_ld32(tSm + c * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[i]);
        }
      }
      const int kv0 = j * kBN;
      if (p.causal ? (kv0 + kBN - 1 > q0) : (kv0 + kBN > N)) {
        const int lim = p.causal ? (q_row - kv0) : (N - 1 - kv0);  // last allowed column
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c > lim) s[c] = -INFINITY;
      }
      // Row max: eight independent chains of 3-input max, then a small tree.
      float mxa[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mxa[k] = fmaxf(s[k], s[k + 8]);
#pragma unroll
      for (int c = 16; c < kBN; c += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k) mxa[k] = fmax3(mxa[k], s[c + k], s[c + 8 + k]);
      const float mx = fmax3(fmax3(mxa[0], mxa[1], mxa[2]), fmax3(mxa[3], mxa[4], mxa[5]),
                             fmaxf(mxa[6], mxa[7]));
      const float m_new = fmaxf(m, mx * sl2);
      // Rescale only when some row of the warp gained more than 2^8; otherwise
      // keep the stale max for both l and O (exact either way).
      float corr = 1.f;
      bool rescale_o = false;
      if (j == 0) {
        m = m_new;  // O is written fresh by the first P V product
      } else if (__any_sync(0xffffffffu, m_new - m > kRescaleThreshold)) {
        corr = ex2_approx(m - m_new);
        m = m_new;
        l *= corr;
        rescale_o = true;
      }
      // P = exp2(s * scale * log2e - m): packed FMA for the argument, MUFU ex2,
      // packed into bf16 pairs for TMEM; the row sum uses four packed chains.
      const float2 sl2v = make_float2(sl2, sl2), nmv = make_float2(-m, -m);
      float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 x = fma2(make_float2(s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1]), sl2v, nmv);
          const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          rs[i & 3] = add2(rs[i & 3], pp);
          pk[i] = pack_bf16x2(pp.x, pp.y);
        }
        tmem_st16(tSm + c * 16, pk);
      }
      const float2 rsum = add2(add2(rs[0], rs[1]), add2(rs[2], rs[3]));
      l += rsum.x + rsum.y;
      if (rescale_o) {  // O holds every P V product up to tile j-1 (in-order tensor core)
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tOm + c * 32, r);
          tmem_wait_ld();
          const float2 cv = make_float2(corr, corr);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 v = mul2(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), cv);
            r[2 * i] = __float_as_uint(v.x);
            r[2 * i + 1] = __float_as_uint(v.y);
          }
          tmem_st32(tOm + c * 32, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kPFull + t));
    }
    // ---- epilogue: O = acc / l, LSE = (m + log2 l) ln 2 ----
    if (ok) ok = mbar_wait_warp(bar(kOFull + t), 0, ctl);
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const bool row_ok = q_row < N;
      float* orow = p.o + ((size_t)zq * N + (size_t)(row_ok ? q_row : 0)) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tOm + c * 32, r);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float4 v = make_float4(__uint_as_float(r[4 * i]) * inv_l, __uint_as_float(r[4 * i + 1]) * inv_l,
                                   __uint_as_float(r[4 * i + 2]) * inv_l, __uint_as_float(r[4 * i + 3]) * inv_l);
            reinterpret_cast<float4*>(orow + c * 32)[i] = v;
          }
        }
      }
      if (row_ok) p.lse[(size_t)zq * N + q_row] = (m + __log2f(l)) * kLn2;
    }
  }

  // ---- teardown: every TMEM reader and the MMA drain are done ----
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch.
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// (rows, planes) bf16 tensor of shape (planes, rows, D): box = 64 x 128 x 1, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int D, int rows, int planes) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * (cuuint64_t)rows};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_prefill_t(const PrefillArgs& a, const LaunchCtx& ctx) {
  using L = PrefillSmem<D>;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kAlloc);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, D, a.seqlen, a.batch * a.n_q_heads) ||
      !make_map(&mk, a.k, D, a.seqlen, a.batch * a.n_kv_heads) ||
      !make_map(&mv, a.v, D, a.seqlen, a.batch * a.n_kv_heads))
    return cudaErrorInvalidValue;
  PrefillParams pp;
  pp.o = a.o;
  pp.lse = a.lse;
  pp.batch = a.batch;
  pp.n_q_heads = a.n_q_heads;
  pp.n_kv_heads = a.n_kv_heads;
  pp.seqlen = a.seqlen;
  pp.sl2 = a.scale * kLog2e;
  pp.causal = a.causal;
  pp.n_row_blocks = (a.seqlen + 2 * kBM - 1) / (2 * kBM);
  pp.err_word = ctx.err_word;
  pp.timeout_ns = ctx.timeout_ns;
  const unsigned grid = (unsigned)pp.n_row_blocks * (unsigned)(a.batch * a.n_q_heads);
  prefill_kernel<D><<<grid, kThreads, L::kAlloc, ctx.stream>>>(mq, mk, mv, pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const LaunchCtx& ctx) {
  return a.head_dim == 128 ? launch_prefill_t<128>(a, ctx) : launch_prefill_t<64>(a, ctx);
}

}  // namespace attn
