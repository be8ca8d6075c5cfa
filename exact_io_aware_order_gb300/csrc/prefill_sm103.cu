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
//   * one CTA owns one 128-row query tile of one head; key/value tiles are 128
//     keys, streamed by TMA (128-byte swizzle, 3-D tensor maps so rows past the
//     end read as zero) into a K ring and a V ring in shared memory;
//   * TMEM (512 columns): three S buffers (128 columns each) and O.  S is
//     triple-buffered, so the tensor core computes S(j+1), S(j+2) while the
//     softmax works on S(j).  P(j) is written as bf16 over the first half of
//     S(j)'s buffer and feeds O += P V straight from TMEM (A operand in tensor
//     memory), V from shared memory (MN-major);
//   * two threads issue tcgen05.mma: warp 5 the S products (S(j) as soon as
//     K_j is in and PV(j-3) has freed the buffer), warp 6 the P V products
//     (as soon as P(j) and V_j are ready).  Every wait or commit stalls its
//     issuing thread for longer than one 128x128x16 MMA runs, so one thread
//     alone leaves the tensor core idle between groups; with two, one
//     thread's synchronisation overlaps the other's MMAs.  Warp 4 is the TMA
//     producer;
//   * warps 0-3 run the softmax, one query row per thread (TMEM lane = row),
//     so row max and row sum need no shuffles and no cross-warp exchange;
//     with one softmax warp per scheduler, its ALU work overlaps its own
//     exponentials on the MUFU pipe;
//   * base-2 exponentials with scale*log2(e) folded in; O is rescaled only
//     when a row max grows by more than 2^8 (the same stale max is used for
//     l and O, so the result is exact), and only after the previous P V
//     product has completed; the LSE is converted back to natural log;
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
constexpr int kThreads = 224;            // 7 warps
constexpr int kSoftmaxThreads = 128;     // warps 0-3: one query row per thread
constexpr int kProducerWarp = 4;
constexpr int kSWarp = 5;                // issues S = Q K^T
constexpr int kPVWarp = 6;               // issues O += P V
constexpr int kSBuf = 3;                 // S buffers in TMEM
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when max grows > 2^8

template <int D>
struct PrefillSmem {
  static constexpr int kTileBytes = 128 * D * 2;       // one Q, K or V tile
  static constexpr int kChunkBytes = 128 * 128;        // 128 rows x 64 bf16 (one swizzle span)
  static constexpr int kKSlots = D == 128 ? 2 : 4;
  static constexpr int kVSlots = D == 128 ? 3 : 6;
  static constexpr int kQ = 0;
  static constexpr int kK = kTileBytes;
  static constexpr int kV = kK + kKSlots * kTileBytes;
  static constexpr int kBar = kV + kVSlots * kTileBytes;
  // barriers: q_full, k_full/k_empty[K slots], v_full/v_empty[V slots], s_full[3],
  // p_full[3], pv_done[3], o_full, drain_s, drain_pv
  static constexpr int kNumBars = 1 + 2 * kKSlots + 2 * kVSlots + 3 * kSBuf + 1 + 2;
  static constexpr int kMisc = kBar + kNumBars * 8;            // tmem base, abort flag
  static constexpr int kUsed = kMisc + 16;
  static constexpr int kAlloc = kUsed + 1024;                  // + alignment slack
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

struct PrefillParams {
  float* o;
  float* lse;
  int batch, n_q_heads, n_kv_heads, seqlen;
  float sl2;  // scale * log2(e)
  int causal;
  int n_q_tiles;  // ceil(seqlen / 128)
  uint32_t* err_word;
  uint64_t timeout_ns;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using L = PrefillSmem<D>;
  constexpr int RK = L::kKSlots, RV = L::kVSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item: longest causal rows first; adjacent CTAs share kv heads ----
  const int BH = p.batch * p.n_q_heads;
  const int qt = p.n_q_tiles - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int bidx = bh / p.n_q_heads, h = bh % p.n_q_heads;
  const int kvh = h / (p.n_q_heads / p.n_kv_heads);
  const int N = p.seqlen;
  const int q0 = qt * kBM;
  const int n = p.causal ? (qt + 1) : (N + kBN - 1) / kBN;  // key tiles visited (>= 1)

  // Barrier layout.
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const int kQFull = 0, kKFull = 1, kKEmpty = kKFull + RK, kVFull = kKEmpty + RK,
            kVEmpty = kVFull + RV, kSFull = kVEmpty + RV, kPFull = kSFull + kSBuf,
            kPVDone = kPFull + kSBuf, kOFull = kPVDone + kSBuf, kDrainS = kOFull + 1,
            kDrainPV = kDrainS + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kMisc + 4);

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    mbar_init(bar(kQFull), 1);
    for (int i = 0; i < RK; ++i) {
      mbar_init(bar(kKFull + i), 1);
      mbar_init(bar(kKEmpty + i), 1);
    }
    for (int i = 0; i < RV; ++i) {
      mbar_init(bar(kVFull + i), 1);
      mbar_init(bar(kVEmpty + i), 1);
    }
    for (int i = 0; i < kSBuf; ++i) {
      mbar_init(bar(kSFull + i), 1);
      mbar_init(bar(kPFull + i), kSoftmaxThreads);
      mbar_init(bar(kPVDone + i), 1);
    }
    mbar_init(bar(kOFull), 1);
    mbar_init(bar(kDrainS), 1);
    mbar_init(bar(kDrainPV), 1);
    fence_mbar_init();
  }
  if (warp == kSWarp) {
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
  // TMEM columns: S buffers [0,128), [128,256), [256,384) | O [384, 384+D)
  const uint32_t tO = tmem + 384u;
  const WaitCtl ctl{abort_flag, p.err_word, p.timeout_ns};
  const int zq = bidx * p.n_q_heads + h;      // Q / O tensor-map "plane"
  const int zk = bidx * p.n_kv_heads + kvh;   // K / V tensor-map plane
  const uint32_t id_s = idesc_bf16_f32(kBM, kBN, false, false);  // Q, K both K-major
  const uint32_t id_pv = idesc_bf16_f32(kBM, D, false, true);    // V is MN-major
  const uint32_t dhi = sw128_desc_hi(1024);

  if (warp == kProducerWarp) {
    // ============================ TMA producer ============================
    // Load order K0, K1, V0, K2, V1, K3, ...: the order the two issuing
    // threads need the tiles.  K_j's slot is reused once S(j - RK) is done,
    // V_j's once PV(j - RV) is done.
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(kQFull), (uint32_t)L::kTileBytes);
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem_u32(smem + L::kQ + c * L::kChunkBytes), &tm_q, bar(kQFull), c * 64, q0, zq);
      int nk = 0, nv = 0;  // tiles issued
      auto load = [&](bool is_k, int j) -> bool {
        const int R = is_k ? RK : RV, slot = j % R;
        const int full = (is_k ? kKFull : kVFull) + slot, empty = (is_k ? kKEmpty : kVEmpty) + slot;
        if (j >= R && !mbar_wait(bar(empty), ((j / R) - 1) & 1, ctl)) return false;
        mbar_arrive_expect_tx(bar(full), (uint32_t)L::kTileBytes);
        const int base = is_k ? L::kK : L::kV;
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem_u32(smem + base + slot * L::kTileBytes + c * L::kChunkBytes),
                      is_k ? &tm_k : &tm_v, bar(full), c * 64, j * kBN, zk);
        if (is_k) ++nk; else ++nv;
        return true;
      };
      bool ok = true;
      for (int j = 0; ok && j < min(n, 2); ++j) ok = load(true, j);
      for (int j = 0; ok && j < n; ++j) {
        ok = load(false, j);
        if (ok && j + 2 < n) ok = load(true, j + 2);
      }
      if (*abort_flag) {
        // Let copies already in flight land before the CTA's memory is released.
        volatile uint32_t no_abort = 0u;
        WaitCtl drain{&no_abort, p.err_word, p.timeout_ns};
        mbar_wait(bar(kQFull), 0, drain);
        for (int j = max(0, nk - RK); j < nk; ++j) mbar_wait(bar(kKFull + j % RK), (j / RK) & 1, drain);
        for (int j = max(0, nv - RV); j < nv; ++j) mbar_wait(bar(kVFull + j % RV), (j / RV) & 1, drain);
      }
    }
  } else if (warp == kSWarp) {
    // ============================ S = Q K^T issuer ============================
    if (lane == 0) {
      const uint32_t q_lo = sw128_desc_lo(smem_u32(smem + L::kQ), 16);
      const uint32_t k_lo0 = sw128_desc_lo(smem_u32(smem + L::kK), 16);
      bool ok = mbar_wait(bar(kQFull), 0, ctl);
      for (int j = 0; ok && j < n; ++j) {
        const int b = j % kSBuf, slot = j % RK;
        // Buffer b last held P(j-3): PV(j-3) must have read it.
        if (j >= kSBuf && !mbar_wait(bar(kPVDone + b), ((j / kSBuf) - 1) & 1, ctl)) { ok = false; break; }
        if (!mbar_wait(bar(kKFull + slot), (j / RK) & 1, ctl)) { ok = false; break; }
        const uint32_t kb = k_lo0 + (uint32_t)((slot * L::kTileBytes) >> 4);
        const uint32_t dS = tmem + (uint32_t)(b * 128);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kChunkBytes + (kk & 3) * 32) >> 4;
          mma_ss_lo(dS, q_lo + off, kb + off, dhi, id_s, kk > 0);
        }
        mma_commit(bar(kSFull + b));
        mma_commit(bar(kKEmpty + slot));
      }
      // Before TMEM can be freed every issued MMA must have finished.
      mma_commit(bar(kDrainS));
      volatile uint32_t no_abort = 0u;
      WaitCtl drain{&no_abort, p.err_word, p.timeout_ns};
      mbar_wait(bar(kDrainS), 0, drain);
    }
    __syncwarp();
  } else if (warp == kPVWarp) {
    // ============================ O += P V issuer ============================
    if (lane == 0) {
      const uint32_t v_lo0 = sw128_desc_lo(smem_u32(smem + L::kV), L::kChunkBytes);
      bool ok = true;
      for (int j = 0; ok && j < n; ++j) {
        const int b = j % kSBuf, slot = j % RV;
        if (!mbar_wait(bar(kPFull + b), (j / kSBuf) & 1, ctl)) { ok = false; break; }
        tc_fence_after();  // P(j) was written to TMEM by the softmax threads
        if (!mbar_wait(bar(kVFull + slot), (j / RV) & 1, ctl)) { ok = false; break; }
        // B = V tile rows [16kk, 16kk+16): 16 rows x 128 B per k step; the
        // 64-column halves of the head dimension are one chunk apart (LBO).
        const uint32_t vb = v_lo0 + (uint32_t)((slot * L::kTileBytes) >> 4);
        const uint32_t aP = tmem + (uint32_t)(b * 128);
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts_lo(tO, aP + kk * 8, vb + ((kk * 16 * 128) >> 4), dhi, id_pv, kk > 0 ? 1u : acc0);
        mma_commit(bar(kVEmpty + slot));
        mma_commit(bar(kPVDone + b));
        if (j == n - 1) mma_commit(bar(kOFull));
      }
      mma_commit(bar(kDrainPV));
      volatile uint32_t no_abort = 0u;
      WaitCtl drain{&no_abort, p.err_word, p.timeout_ns};
      mbar_wait(bar(kDrainPV), 0, drain);
    }
    __syncwarp();
  } else {
    // ============================ softmax warps ============================
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int row = warp * 32 + lane;               // row within the tile (= TMEM lane)
    const int q_row = q0 + row;
    const float sl2 = p.sl2;
    const uint32_t tOm = tO + lane_base;
    float m = -INFINITY, l = 0.f;   // running max (log2 domain) and sum of the row
    bool ok = true;
    for (int j = 0; ok && j < n; ++j) {
      const int b = j % kSBuf;
      if (!mbar_wait_warp(bar(kSFull + b), (j / kSBuf) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tSm = tmem + (uint32_t)(b * 128) + lane_base;
      // The whole S row: four 32-column loads in flight, one wait.
      float s[kBN];
      {
        uint32_t r[kBN / 32][32];
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) tmem_ld32(tSm + c * 32, r[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[c][i]);
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
      // packed into bf16 pairs over the first 64 columns of the buffer; the row
      // sum uses four packed chains.
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
      if (rescale_o) {
        // O must hold every P V product up to tile j-1 before it is rescaled.
        const int bp = (j - 1) % kSBuf;
        if (!mbar_wait_warp(bar(kPVDone + bp), ((j - 1) / kSBuf) & 1, ctl)) { ok = false; break; }
        tc_fence_after();
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
      mbar_arrive(bar(kPFull + b));
    }
    // ---- epilogue: O = acc / l, LSE = (m + log2 l) ln 2 ----
    if (ok) ok = mbar_wait_warp(bar(kOFull), 0, ctl);
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

  // ---- teardown: every TMEM reader and both MMA drains are done ----
  tc_fence_before();
  __syncthreads();
  if (warp == kSWarp) {
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
  pp.n_q_tiles = (a.seqlen + kBM - 1) / kBM;
  pp.err_word = ctx.err_word;
  pp.timeout_ns = ctx.timeout_ns;
  const unsigned grid = (unsigned)pp.n_q_tiles * (unsigned)(a.batch * a.n_q_heads);
  prefill_kernel<D><<<grid, kThreads, L::kAlloc, ctx.stream>>>(mq, mk, mv, pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const LaunchCtx& ctx) {
  return a.head_dim == 128 ? launch_prefill_t<128>(a, ctx) : launch_prefill_t<64>(a, ctx);
}

}  // namespace attn
