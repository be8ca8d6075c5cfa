// Split-KV single-token decode and the LSE combine, sm_103a.
//
// Page "FlashAttention for inference: tiled prefill and split-KV decoding",
// section "Decode: a different bottleneck": the key/value sequence of each
// (sequence, kv head) is split into chunks, one thread block per chunk; each
// block loads every key/value row of its chunk once and uses it for all
// g = n_q / n_kv query heads of that kv head (GQA-aware sharing), streams a
// paged or contiguous cache, and writes its partial output with its
// log-sum-exp.  A second small kernel merges the partials by their LSE
// weights (section "The online softmax, with every symbol defined", combining
// partial results; the merge rule of section "Minimal implementation").
//
// Design for GB300.  Decode is HBM-bound, so the kernel is built to stream:
//   * a producer warp feeds a ring of 64-token stages with tiled TMA copies
//     (128-byte swizzle): one box of 64 tokens x 64 dims (8 KB) for a
//     contiguous cache, one box of 16 tokens (2 KB) per 16-token group of a
//     paged cache whose block size is a multiple of 16.  Other block sizes
//     fall back to plain loads by the producer warp;
//   * four consumer warps each take 16 tokens of a stage.  With g query rows
//     sharing the rows, q K^T and P V are small dense products (M = 16 padded
//     rows); they run on mma.sync m16n8k16 (bf16 in, fp32 accumulate) so the
//     ALU work stays far below the memory time;
//   * ldmatrix reads the swizzled rows without bank conflicts; row max / row
//     sum use quad shuffles; the output is rescaled only when a row max grows
//     by more than 2^8 (exact: the same stale max is used for l and O); at the
//     end the warps merge their (m, l, O) states through shared memory.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

#ifndef ATTN_DECODE_STAGES
#define ATTN_DECODE_STAGES 3
#endif
constexpr int kStageTokens = 64;   // tokens per ring stage
constexpr int kStages = ATTN_DECODE_STAGES;
constexpr int kConsumerWarps = 4;  // 16 tokens each per stage
constexpr int kMaxRowGroups = 4;   // query rows per kv head: up to 4 groups of 16
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// How the producer fills a stage.
enum LoadMode : int { kLoadBox64 = 0, kLoadBox16 = 1, kLoadPlain = 2 };

template <int D>
struct DecodeSmem {
  static constexpr int kHalves = D / 64;                       // 128-byte swizzle spans per row
  static constexpr int kHalfBytes = kStageTokens * 128;        // 64 rows x 128 B
  static constexpr int kTileBytes = kHalves * kHalfBytes;      // K (or V) of one stage
  static constexpr int kStageBytes = 2 * kTileBytes;           // K then V
  static constexpr int kQRowBytes = D * 2 + 16;                // padded q rows
  static constexpr int kRing = 0;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kBarOff = kRingBytes;                   // 2*kStages barriers
  static constexpr int kMiscOff = kBarOff + 2 * kStages * 8;
  static constexpr int kQOff = kMiscOff + 16;                  // 16 q rows per row group
  // Dynamic shared memory for `groups` row groups of 16 query rows.
  static constexpr int total(int groups) { return kQOff + groups * 16 * kQRowBytes + 1024; }
  // Merge scratch reuses the ring once the stream is done: per warp 16 rows of
  // D floats at a padded pitch (64-bit stores from a quad land in distinct
  // bank pairs), then per warp and row m and l, then per row the warps' weights.
  static constexpr int kMergePitch = D + 8;                            // floats
  static constexpr int kMergeO = 0;                                    // [warps][16][pitch]
  static constexpr int kMergeM = kConsumerWarps * 16 * kMergePitch * 4;  // [warps][16]
  static constexpr int kMergeL = kMergeM + kConsumerWarps * 16 * 4;      // [warps][16]
  static constexpr int kMergeF = kMergeL + kConsumerWarps * 16 * 4;      // [warps][16]
  static_assert(kMergeF + kConsumerWarps * 16 * 4 <= kRingBytes, "merge scratch fits in the ring");
};

// Byte offset of (row, 16-byte chunk c) inside one 128-byte-swizzled span.
__device__ __forceinline__ uint32_t swz(int row, int c) {
  return (uint32_t)(row * 128 + ((c ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
// L2 prefetch of one box: a hint, with no shared memory and no barrier.
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int c0, int c1, int c2,
                                                int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");
}

struct DecodeKParams {
  DecodeArgs a;
  int mode;  // LoadMode
  uint32_t* err_word;
  uint64_t timeout_ns;
};

template <int D>
__global__ void __launch_bounds__(kThreads)
decode_splitkv_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const DecodeKParams kp) {
  using L = DecodeSmem<D>;
  const DecodeArgs& a = kp.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int S = a.num_splits;
  const int g = a.n_q_heads / a.n_kv_heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Inputs may come from the previous kernel on the stream: wait for it before
  // the first global read; then let the next kernel (the combine) begin its
  // launch while this grid streams.  Early cache streaming: the caller has
  // stated that the previous kernel writes neither kv_lens, the block table
  // nor the cache, so the wait moves to the reads of q (consumers) and the
  // first write; the producer fills the ring meanwhile.
  const bool early = a.early_cache != 0;
  if (!early) grid_dep_wait();
  grid_dep_launch();
  // Contiguous cache: before kv_lens arrives, ask L2 for the first stage of
  // this split as the host's max_kv_len places it (kv_len's placement when
  // the two are equal).  A hint only: the copies below read whatever range
  // kv_len gives.
  if (kp.mode == kLoadBox64 && a.k_new == nullptr && a.window_left < 0 && threadIdx.x == 0) {
    const int per_h = (a.max_kv_len + S - 1) / S;
    const int chunk_h = (per_h + kSplitGranule - 1) / kSplitGranule * kSplitGranule;
    const long long t0_h = (long long)split * chunk_h;
    if (t0_h < a.max_kv_len) {
#pragma unroll
      for (int h = 0; h < L::kHalves; ++h) {
        tma_prefetch_4d(&tm_k, h * 64, kvh, (int)t0_h, b);
        tma_prefetch_4d(&tm_v, h * 64, kvh, (int)t0_h, b);
      }
    }
  }
  // ---- this split's token range (split rule: see the C header) ----
  const bool paged = a.block_table != nullptr;
  const bool append = a.k_new != nullptr;
  const long long capacity =
      paged ? (long long)a.max_blocks_per_seq * a.block_size : (long long)a.max_kv_len;
  int len = a.kv_lens[b];  // tokens already cached
  bool len_ok = true;
  if (len < 0 || (long long)len + (append ? 1 : 0) > capacity) {
    if (threadIdx.x == 0 && split == 0) atomicOr(kp.err_word, kErrKvLen);
    len = len < 0 ? 0 : (int)capacity - (append ? 1 : 0);
    len_ok = false;  // attend over the clamped length, write nothing
  }
  const int pos_new = len;  // the appended token's position
  if (append) len += 1;     // the new token attends to itself too
  // A sliding window keeps tokens lo_tok .. len-1; the splits cover
  // [lo16, len) with lo16 = lo_tok rounded down to the split granule, and
  // tokens below lo_tok are masked.
  const int lo_tok = a.window_left >= 0 ? max(0, len - 1 - a.window_left) : 0;
  const int lo16 = lo_tok / kSplitGranule * kSplitGranule;
  const int n_att = len - lo16;
  const int per = (n_att + S - 1) / S;
  const int chunk = (per + kSplitGranule - 1) / kSplitGranule * kSplitGranule;
  const int t0 = lo16 + min(split * chunk, n_att);
  const int t1 = lo16 + min(min(split * chunk, n_att) + chunk, n_att);
  const int n_tok = t1 - t0;

  float* o_out = a.o_partial + (((size_t)split * a.batch + b) * a.n_q_heads + (size_t)kvh * g) * D;
  float* lse_out = a.lse_partial + ((size_t)split * a.batch + b) * a.n_q_heads + (size_t)kvh * g;
  if (n_tok <= 0) {  // empty split: o = 0, lse = -inf
    if (early) grid_dep_wait();
    for (int i = threadIdx.x; i < g * D; i += blockDim.x) o_out[i] = 0.f;
    for (int i = threadIdx.x; i < g; i += blockDim.x) lse_out[i] = -INFINITY;
    return;
  }
  const int n_stage_iters = (n_tok + kStageTokens - 1) / kStageTokens;

  // ---- decode with append: the split that holds the new position writes
  // the new key / value row of this kv head into the cache (page "FlashAttention
  // for inference", section "Minimal implementation": the decode call appends
  // the new keys and values in place).  The write is fenced against the async
  // proxy and the block synchronises below before the producer's first copy,
  // so the copies that cover the position read the new row.  No other block
  // reads that position.
  if (append && len_ok && pos_new >= t0 && pos_new < t1 && threadIdx.x < 2 * (D / 8)) {
    const bool is_v = threadIdx.x >= D / 8;
    const int c = threadIdx.x % (D / 8);  // 16-byte chunk of the row
    long long row = -1;                   // (token, kv head) row index in the cache
    if (paged) {
      const int blk = a.block_table[(size_t)b * a.max_blocks_per_seq + pos_new / a.block_size];
      if (blk >= 0 && blk < a.num_blocks)
        row = ((long long)blk * a.block_size + pos_new % a.block_size) * a.n_kv_heads + kvh;
      else if (c == 0 && !is_v)
        atomicOr(kp.err_word, kErrBlockIndex);
    } else {
      row = ((long long)b * a.max_kv_len + pos_new) * a.n_kv_heads + kvh;
    }
    if (row >= 0) {
      const uint4 val = reinterpret_cast<const uint4*>(
          (is_v ? a.v_new : a.k_new) + ((size_t)b * a.n_kv_heads + kvh) * D)[c];
      uint16_t* dst = const_cast<uint16_t*>(is_v ? a.v_cache : a.k_cache) + (size_t)row * D;
      reinterpret_cast<uint4*>(dst)[c] = val;
      fence_proxy_async_global();
    }
  }

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + L::kMiscOff);
  const uint32_t full0 = smem_u32(&bars[0]);
  const uint32_t empty0 = smem_u32(&bars[kStages]);
  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl ctl{abort_flag, kp.err_word, kp.timeout_ns};

  if (warp == 0) {
    // ================= producer: stream rows into the ring =================
    const int32_t* table = paged ? a.block_table + (size_t)b * a.max_blocks_per_seq : nullptr;
    if (lane == 0 && kp.mode != kLoadPlain) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    for (int it = 0; it < n_stage_iters; ++it) {
      const int st = it % kStages;
      if (it >= kStages) {
        if (!mbar_wait_warp(empty0 + 8 * st, ((it / kStages) - 1) & 1, ctl)) break;
      }
      const int base = t0 + it * kStageTokens;
      const int cnt = min(kStageTokens, t1 - base);
      uint8_t* sk = smem + L::kRing + st * L::kStageBytes;
      uint8_t* sv = sk + L::kTileBytes;
      if (kp.mode == kLoadBox64) {
        // Contiguous cache viewed as (D, n_kv, L, B): one 64-token box per half.
        if (lane == 0) {
          mbar_arrive_expect_tx(full0 + 8 * st, (uint32_t)L::kStageBytes);
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h) {
            tma_load_4d(smem_u32(sk + h * L::kHalfBytes), &tm_k, full0 + 8 * st, h * 64, kvh, base, b);
            tma_load_4d(smem_u32(sv + h * L::kHalfBytes), &tm_v, full0 + 8 * st, h * 64, kvh, base, b);
          }
        }
      } else if (kp.mode == kLoadBox16) {
        // Paged cache viewed as (D, n_kv, block_size, num_blocks): one box per
        // 16-token group (a group never straddles a block: both are 16-aligned).
        const int groups = (cnt + 15) >> 4;
        if (lane == 0)
          mbar_arrive_expect_tx(full0 + 8 * st, (uint32_t)groups * 16u * 2u * (uint32_t)D * 2u);
        __syncwarp();
        if (lane < groups) {
          const int t = base + 16 * lane;
          int blk = table[t / a.block_size];
          if (blk < 0 || blk >= a.num_blocks) {
            atomicOr(kp.err_word, kErrBlockIndex);
            blk = 0;  // keep the copy in bounds; the result is flagged invalid
          }
          const int slot = t % a.block_size;
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h) {
            tma_load_4d(smem_u32(sk + h * L::kHalfBytes + lane * 2048), &tm_k, full0 + 8 * st,
                        h * 64, kvh, slot, blk);
            tma_load_4d(smem_u32(sv + h * L::kHalfBytes + lane * 2048), &tm_v, full0 + 8 * st,
                        h * 64, kvh, slot, blk);
          }
        }
      } else {
        // Any other block size: plain 16-byte loads into the swizzled layout.
        for (int i = lane; i < cnt * (D / 8); i += 32) {
          const int r = i / (D / 8), c = i % (D / 8);
          const int t = base + r;
          size_t row;
          if (paged) {
            int blk = table[t / a.block_size];
            if (blk < 0 || blk >= a.num_blocks) {
              atomicOr(kp.err_word, kErrBlockIndex);
              blk = 0;
            }
            row = (size_t)blk * a.block_size + (t % a.block_size);
          } else {
            row = (size_t)b * a.max_kv_len + t;
          }
          const size_t off = (row * a.n_kv_heads + kvh) * D + (size_t)c * 8;
          const uint4 kval = *reinterpret_cast<const uint4*>(a.k_cache + off);
          const uint4 vval = *reinterpret_cast<const uint4*>(a.v_cache + off);
          const uint32_t o = (c >> 3) * L::kHalfBytes + swz(r, c & 7);
          *reinterpret_cast<uint4*>(sk + o) = kval;
          *reinterpret_cast<uint4*>(sv + o) = vval;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(full0 + 8 * st);
      }
    }
    // Wait for copies still in flight before the CTA may leave (abort path only:
    // on the normal path the consumers have waited on every stage).
    if (*abort_flag && lane == 0) {
      volatile uint32_t no_abort = 0u;
      WaitCtl drain{&no_abort, kp.err_word, kp.timeout_ns};
      for (int it = max(0, n_stage_iters - kStages); it < n_stage_iters; ++it)
        mbar_wait(full0 + 8 * (it % kStages), (it / kStages) & 1, drain);
    }
  } else {
    // ================= consumers =================
    const int cw = warp - 1;
    const int ctid = threadIdx.x - 32;
    // Row groups: the g query rows in groups of 16 (G = 1, 2 or 4).  The
    // four warps split into G teams, one per group; a team's warps share the
    // stage's four 16-token sub-blocks, so every K/V row is still read from
    // memory once and used for all g rows.
    const int G = g <= 16 ? 1 : (g <= 32 ? 2 : 4);
    const int team = 4 / G;              // warps per row group
    const int rg = cw / team;            // this warp's row group
    const int rg_row0 = rg * 16;         // its first query row
    uint8_t* sq = smem + L::kQOff;
    // q rows of this kv head's g query heads; rows g .. 16 G - 1 are zero.
    if (early) grid_dep_wait();  // q (and below, the slopes) may come from the previous grid
    const uint16_t* qsrc = a.q + ((size_t)b * a.n_q_heads + (size_t)kvh * g) * D;
    for (int i = ctid; i < 16 * G * (D / 8); i += 32 * kConsumerWarps) {
      const int r = i / (D / 8), c = i % (D / 8);
      uint4 val = make_uint4(0, 0, 0, 0);
      if (r < g) val = *reinterpret_cast<const uint4*>(qsrc + (size_t)r * D + c * 8);
      *reinterpret_cast<uint4*>(sq + r * L::kQRowBytes + c * 16) = val;
    }
    consumer_sync();
    // Q as A fragments, one set per 16-wide k step of the head dimension.
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int r = rg_row0 + (lane & 15);
      const int c = kk * 16 + (lane >> 4) * 8;
      ldsm_x4(smem_u32(sq + r * L::kQRowBytes + c * 2), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    }
    // With soft-capping the scores become tanh(s * scale / softcap) and the
    // factor softcap (times log2 e) moves into sl2.
    const bool capped = a.softcap > 0.f;
    const float sl2 = capped ? a.softcap * kLog2e : a.scale * kLog2e;
    const float cap_in2 = capped ? 2.f * kLog2e * a.scale / a.softcap : 0.f;
    // ALiBi: rows gid and gid + 8 are query heads kvh * g + row; their slopes
    // in log2 units.  The scores are then biased and scaled in place, so the
    // softmax below uses a unit scale (sl2x).
    const bool alibi = a.alibi_slopes != nullptr;
    float al2[2] = {0.f, 0.f};
    if (alibi) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = rg_row0 + (lane >> 2) + 8 * r;
        if (row < g) al2[r] = a.alibi_slopes[kvh * g + row] * kLog2e;
      }
    }
    const float sl2x = alibi ? 1.f : sl2;
    float m_r[2] = {-INFINITY, -INFINITY};  // running max (log2 domain) of rows gid, gid+8
    float l_r[2] = {0.f, 0.f};
    float acc[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    const int quad = lane & 3;

    for (int it = 0; it < n_stage_iters; ++it) {
      const int st = it % kStages;
      if (!mbar_wait_warp(full0 + 8 * st, (it / kStages) & 1, ctl)) break;
      const int base = t0 + it * kStageTokens;
      const int cnt = min(kStageTokens, t1 - base);
      // This warp's 16-token sub-blocks of the stage: one with a single row
      // group, two or four when its team shares the stage.
#pragma unroll 1
      for (int sb = cw % team; sb < 4; sb += team) {
      const int vc = min(16, cnt - sb * 16);  // valid tokens of this sub-block
      if (vc > 0) {
        uint8_t* sk = smem + L::kRing + st * L::kStageBytes;
        uint8_t* sv = sk + L::kTileBytes;
        const int r0 = sb * 16;  // the sub-block's first row in the stage
        if (vc < 16) {  // rows past the end: zero V so 0 * (old data) stays 0
          for (int i = lane; i < (16 - vc) * (D / 8); i += 32) {
            const int r = r0 + vc + i / (D / 8), c = i % (D / 8);
            *reinterpret_cast<uint4*>(sv + (c >> 3) * L::kHalfBytes + swz(r, c & 7)) =
                make_uint4(0, 0, 0, 0);
          }
          __syncwarp();
        }
        // ---- S = q K^T for 16 tokens (two n-tiles of 8) ----
        float s[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // lanes 0-7: tokens 0-7 @ d 16kk; 8-15: tokens 0-7 @ d+8; 16-23: tokens 8-15 @ d; 24-31: tokens 8-15 @ d+8
          const int r = r0 + (lane & 7) + ((lane >> 4) << 3);
          const int c = kk * 2 + ((lane >> 3) & 1);  // 16-byte chunk index over the row
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_u32(sk + (c >> 3) * L::kHalfBytes + swz(r, c & 7)), b0, b1, b2, b3);
          mma16816(s[0], qa[kk], b0, b1);
          mma16816(s[1], qa[kk], b2, b3);
        }
        if (capped) {
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[n][e] = tanh_from_exp2(s[n][e] * cap_in2);
        }
        if (alibi) {
          // s -> s scale log2 e - slope log2 e (len - 1 - token)
#pragma unroll
          for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tok = base + r0 + n * 8 + quad * 2 + (e & 1);
              s[n][e] = fmaf(s[n][e], sl2, -al2[e >> 1] * static_cast<float>(len - 1 - tok));
            }
        }
        // ---- mask tokens past the end or left of the window, online softmax update ----
        const int lo_rel = lo_tok - (base + r0);  // first token of the warp's 16 in the window
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = n * 8 + quad * 2 + (e & 1);
            if (tok >= vc || tok < lo_rel) s[n][e] = -INFINITY;
            mx[e >> 1] = fmaxf(mx[e >> 1], s[n][e]);
          }
        bool grow = false;
        float m_new[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
          mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
          m_new[r] = fmaxf(m_r[r], mx[r] * sl2x);  // -inf only while every token was masked
          grow |= m_new[r] - m_r[r] > kRescaleThreshold;  // true at the first unmasked token
        }
        // Keep the stale max unless some row of the warp grew by more than 2^8.
        const bool rescale = __any_sync(0xffffffffu, grow);
        float corr[2] = {1.f, 1.f};
        if (rescale) {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            corr[r] = ex2_approx(m_r[r] - m_new[r]);  // exp2(-inf) = 0 on the first stage
            m_r[r] = m_new[r];
          }
        }
        float rs[2] = {0.f, 0.f};
        uint32_t pa[4];
        // Rows that have seen only masked tokens keep m = -inf: reference 0.
        const float mr0 = m_r[0] == -INFINITY ? 0.f : m_r[0];
        const float mr1 = m_r[1] == -INFINITY ? 0.f : m_r[1];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          const float p0 = ex2_approx(fmaf(s[n][0], sl2x, -mr0));
          const float p1 = ex2_approx(fmaf(s[n][1], sl2x, -mr0));
          const float p2 = ex2_approx(fmaf(s[n][2], sl2x, -mr1));
          const float p3 = ex2_approx(fmaf(s[n][3], sl2x, -mr1));
          rs[0] += p0 + p1;
          rs[1] += p2 + p3;
          pa[2 * n + 0] = pack_bf16x2(p0, p1);  // row gid,   tokens 8n + 2q, +1
          pa[2 * n + 1] = pack_bf16x2(p2, p3);  // row gid+8
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 1);
          rs[r] += __shfl_xor_sync(0xffffffffu, rs[r], 2);
          l_r[r] = l_r[r] * corr[r] + rs[r];
        }
        if (rescale) {
#pragma unroll
          for (int j = 0; j < D / 8; ++j) {
            acc[j][0] *= corr[0];
            acc[j][1] *= corr[0];
            acc[j][2] *= corr[1];
            acc[j][3] *= corr[1];
          }
        }
        // A fragment of P: {row g tok 2q..}, {row g+8 tok 2q..}, {row g tok 8+2q..}, {row g+8 tok 8+2q..}
        const uint32_t pfrag[4] = {pa[0], pa[1], pa[2], pa[3]};
        // ---- O += P V ----
#pragma unroll
        for (int j = 0; j < D / 16; ++j) {
          // lanes 0-7: tok 0-7 @ d 16j; 8-15: tok 8-15 @ 16j; 16-23: tok 0-7 @ 16j+8; 24-31: tok 8-15 @ 16j+8
          const int r = r0 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int c = j * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(sv + (c >> 3) * L::kHalfBytes + swz(r, c & 7)), b0, b1, b2, b3);
          mma16816(acc[2 * j + 0], pfrag, b0, b1);
          mma16816(acc[2 * j + 1], pfrag, b2, b3);
        }
        if (vc < 16) fence_proxy_async_smem();  // generic writes above precede the next copy
      }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
    }

    // ================= merge the consumer warps' states =================
    consumer_sync();  // every warp is done reading the ring
    float* mo = reinterpret_cast<float*>(smem + L::kMergeO);
    float* mm = reinterpret_cast<float*>(smem + L::kMergeM);
    float* ml = reinterpret_cast<float*>(smem + L::kMergeL);
    float* mf = reinterpret_cast<float*>(smem + L::kMergeF);
    const int gid = lane >> 2;
    if (quad == 0) {
      mm[cw * 16 + gid] = m_r[0];
      mm[cw * 16 + gid + 8] = m_r[1];
      ml[cw * 16 + gid] = l_r[0];
      ml[cw * 16 + gid + 8] = l_r[1];
    }
    float* mow = mo + (size_t)cw * 16 * L::kMergePitch;
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      const int col = j * 8 + quad * 2;
      *reinterpret_cast<float2*>(&mow[gid * L::kMergePitch + col]) = make_float2(acc[j][0], acc[j][1]);
      *reinterpret_cast<float2*>(&mow[(gid + 8) * L::kMergePitch + col]) =
          make_float2(acc[j][2], acc[j][3]);
    }
    consumer_sync();
    // Per row: the common max over its team's warps, each warp's weight
    // e^(m_w - m) / l, and the LSE.  Row r belongs to row group r / 16, whose
    // team is warps (r / 16) * team .. + team - 1, at local row r % 16.
    if (ctid < g && !*abort_flag) {
      const int r = ctid, lr = r & 15, w0 = (r >> 4) * team;
      float m = -INFINITY;
      for (int w = w0; w < w0 + team; ++w) m = fmaxf(m, mm[w * 16 + lr]);
      float lsum = 0.f;
      for (int w = w0; w < w0 + team; ++w) {
        const float f = ex2_approx(mm[w * 16 + lr] - m);  // 0 for a warp that saw no token
        lsum += f * ml[w * 16 + lr];
        mf[w * 16 + lr] = f;
      }
      const float inv = 1.f / lsum;
      for (int w = w0; w < w0 + team; ++w) mf[w * 16 + lr] *= inv;
      lse_out[r] = (m + __log2f(lsum)) * kLn2;
    }
    consumer_sync();
    if (!*abort_flag) {
      for (int e = ctid; e < g * (D / 4); e += 32 * kConsumerWarps) {
        const int r = e / (D / 4), c = (e % (D / 4)) * 4;
        const int lr = r & 15, w0 = (r >> 4) * team;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = w0; w < w0 + team; ++w) {
          const float fw = mf[w * 16 + lr];
          const float4 v = *reinterpret_cast<const float4*>(
              &mo[((size_t)w * 16 + lr) * L::kMergePitch + c]);
          o.x = fmaf(fw, v.x, o.x);
          o.y = fmaf(fw, v.y, o.y);
          o.z = fmaf(fw, v.z, o.z);
          o.w = fmaf(fw, v.w, o.w);
        }
        *reinterpret_cast<float4*>(o_out + (size_t)r * D + c) = o;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Combine: one 512-thread block per (sequence, query head).  Every thread
// loads its share of the splits (eight at a time, all in flight together),
// merges them with a running max, then the block merges the threads'
// states: one memory round trip for up to 8 * 16 splits.
// ---------------------------------------------------------------------------
constexpr int kCombineWarps = 16;
constexpr int kCombineBatch = 8;

template <int D>
__global__ void __launch_bounds__(32 * kCombineWarps) combine_kernel(const CombineArgs a) {
  constexpr int kVec = D / 4;                       // float4 per partial row
  constexpr int kLanesPerRow = kVec < 32 ? kVec : 32;
  constexpr int kPerLane = kVec / kLanesPerRow;     // float4 per lane (2 for head_dim 256)
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;   // splits handled per warp step
  constexpr int kStep = kCombineWarps * kRowsPerWarp;
  const int bh = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.num_splits;
  const size_t stride_s = (size_t)a.batch * a.n_q_heads;
  const int sub = lane / kLanesPerRow, li = lane % kLanesPerRow;
  __shared__ float s_max[kCombineWarps], s_sum[kCombineWarps];
  __shared__ float4 s_o[kCombineWarps][kRowsPerWarp][kVec];
  // The next kernel may begin its launch at once: it waits for this grid
  // before it reads what this grid writes or overwrites the partials (a decode
  // with early cache streaming only fills its ring before that wait).
  grid_dep_launch();
  grid_dep_wait();    // the partials come from the decode kernel before us

  float m = -INFINITY, wsum = 0.f;  // running max / weight sum (natural-log domain)
  float4 acc[kPerLane];
#pragma unroll
  for (int e = 0; e < kPerLane; ++e) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = warp * kRowsPerWarp + sub; s0 < S; s0 += kCombineBatch * kStep) {
    float w[kCombineBatch];
    float4 v[kCombineBatch][kPerLane];
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      const int s = s0 + u * kStep;
      w[u] = -INFINITY;
#pragma unroll
      for (int e = 0; e < kPerLane; ++e) v[u][e] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s < S) {
        const size_t idx = (size_t)s * stride_s + bh;
        w[u] = a.lse_partial[idx];
#pragma unroll
        for (int e = 0; e < kPerLane; ++e)
          v[u][e] = reinterpret_cast<const float4*>(a.o_partial + idx * D)[li + e * kLanesPerRow];
      }
    }
    float mb = m;
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) mb = fmaxf(mb, w[u]);
    if (mb != -INFINITY) {
      const float c = ex2_approx((m - mb) * kLog2e);  // 0 while m is -inf
#pragma unroll
      for (int e = 0; e < kPerLane; ++e) {
        acc[e].x *= c; acc[e].y *= c; acc[e].z *= c; acc[e].w *= c;
      }
      wsum *= c;
#pragma unroll
      for (int u = 0; u < kCombineBatch; ++u) {
        const float ew = ex2_approx((w[u] - mb) * kLog2e);  // 0 for an empty split
#pragma unroll
        for (int e = 0; e < kPerLane; ++e) {
          acc[e].x = fmaf(ew, v[u][e].x, acc[e].x);
          acc[e].y = fmaf(ew, v[u][e].y, acc[e].y);
          acc[e].z = fmaf(ew, v[u][e].z, acc[e].z);
          acc[e].w = fmaf(ew, v[u][e].w, acc[e].w);
        }
        wsum += ew;
      }
      m = mb;
    }
  }
  // Block merge: the common max, then every thread's state rescaled to it.
  float mx = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) s_max[warp] = mx;
  __syncthreads();
  mx = s_max[0];
#pragma unroll
  for (int w = 1; w < kCombineWarps; ++w) mx = fmaxf(mx, s_max[w]);
  float4* out = reinterpret_cast<float4*>(a.o + (size_t)bh * D);
  if (mx == -INFINITY) {  // every split empty
    for (int i = threadIdx.x; i < D / 4; i += blockDim.x) out[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (threadIdx.x == 0) a.lse[bh] = -INFINITY;
    return;
  }
  const float f = ex2_approx((m - mx) * kLog2e);  // 0 for a thread that saw only empty splits
#pragma unroll
  for (int e = 0; e < kPerLane; ++e) {
    acc[e].x *= f; acc[e].y *= f; acc[e].z *= f; acc[e].w *= f;
    s_o[warp][sub][li + e * kLanesPerRow] = acc[e];
  }
  float ws = li == 0 ? wsum * f : 0.f;  // each split's weight counted once per sub-row
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
  if (lane == 0) s_sum[warp] = ws;
  __syncthreads();
  float W = 0.f;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) W += s_sum[w];
  for (int i = threadIdx.x; i < kVec; i += blockDim.x) {
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int w = 0; w < kCombineWarps; ++w)
      for (int r = 0; r < kRowsPerWarp; ++r) {
        const float4 v = s_o[w][r][i];
        t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
      }
    const float inv = 1.f / W;
    out[i] = make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
  }
  if (threadIdx.x == 0) a.lse[bh] = mx + logf(W);
}

__global__ void wait_selftest_kernel(uint32_t* err_word, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0u;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl ctl{&abort_flag, err_word, timeout_ns};
  mbar_wait(smem_u32(&bar), 0, ctl);  // no one arrives: must give up after timeout_ns
  __syncthreads();
  if (threadIdx.x == 0) mbar_arrive(smem_u32(&bar));  // complete the phase before exit
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// A (D, n_kv, rows, planes) bf16 cache with boxes of 64 dims x 1 head x box_rows x 1.
bool make_cache_map(CUtensorMap* m, const void* base, int D, int n_kv, long long rows,
                    long long planes, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)n_kv, (cuuint64_t)rows, (cuuint64_t)planes};
  cuuint64_t row = (cuuint64_t)D * 2;
  cuuint64_t strides[3] = {row, row * (cuuint64_t)n_kv, row * (cuuint64_t)n_kv * (cuuint64_t)rows};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_decode_t(const DecodeArgs& a, const LaunchCtx& ctx) {
  using L = DecodeSmem<D>;
  static bool configured[64] = {};  // the attribute is per device
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_splitkv_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::total(kMaxRowGroups));
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  const int gq = a.n_q_heads / a.n_kv_heads;  // at most 64 (validated)
  const int groups = gq <= 16 ? 1 : (gq <= 32 ? 2 : 4);
  DecodeKParams kp;
  kp.a = a;
  kp.err_word = ctx.err_word;
  kp.timeout_ns = ctx.timeout_ns;
  CUtensorMap mk, mv;
  std::memset(&mk, 0, sizeof(mk));
  std::memset(&mv, 0, sizeof(mv));
  if (a.block_table == nullptr) {
    kp.mode = kLoadBox64;
    if (!make_cache_map(&mk, a.k_cache, D, a.n_kv_heads, a.max_kv_len, a.batch, 64) ||
        !make_cache_map(&mv, a.v_cache, D, a.n_kv_heads, a.max_kv_len, a.batch, 64))
      return cudaErrorInvalidValue;
  } else if (a.block_size % 16 == 0) {
    kp.mode = kLoadBox16;
    if (!make_cache_map(&mk, a.k_cache, D, a.n_kv_heads, a.block_size, a.num_blocks, 16) ||
        !make_cache_map(&mv, a.v_cache, D, a.n_kv_heads, a.block_size, a.num_blocks, 16))
      return cudaErrorInvalidValue;
  } else {
    kp.mode = kLoadPlain;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_splits, a.n_kv_heads, a.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::total(groups);
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_splitkv_kernel<D>, mk, mv, kp);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, const LaunchCtx& ctx) {
  if (a.head_dim == 256) return launch_decode_t<256>(a, ctx);
  return a.head_dim == 128 ? launch_decode_t<128>(a, ctx) : launch_decode_t<64>(a, ctx);
}

cudaError_t launch_combine(const CombineArgs& a, const LaunchCtx& ctx) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.batch * (unsigned)a.n_q_heads);
  cfg.blockDim = dim3(32 * kCombineWarps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.head_dim == 256) return cudaLaunchKernelEx(&cfg, combine_kernel<256>, a);
  return a.head_dim == 128 ? cudaLaunchKernelEx(&cfg, combine_kernel<128>, a)
                           : cudaLaunchKernelEx(&cfg, combine_kernel<64>, a);
}

cudaError_t launch_wait_selftest(const LaunchCtx& ctx) {
  wait_selftest_kernel<<<1, 32, 0, ctx.stream>>>(ctx.err_word, ctx.timeout_ns);
  return cudaGetLastError();
}

}  // namespace attn
