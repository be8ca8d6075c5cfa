// FP8 (e4m3) block quantisation with incoherent processing, sm_103a.
//
// Page "FlashAttention for inference: tiled prefill and split-KV decoding",
// section "Interaction with post-trained models": FlashAttention-3's FP8
// path lowers the error of naive FP8 attention by block quantisation and
// incoherent processing.  These kernels prepare the inputs of the FP8
// prefill: optionally rotate each row by diag(signs) H / sqrt(d) (H the
// Sylvester Hadamard matrix; the same rotation for Q and K leaves Q K^T
// unchanged), then quantise blocks of rows to e4m3 with scale amax / 448.
//
// Layout of the work: blocks of 128 rows of a plane, eight warps of 16 rows
// each.  Within a warp, LPR consecutive lanes share a row: lane l holds
// elements [E c, E c + E) (c = l % LPR, E = d / LPR) of the rows l / LPR +
// k (32 / LPR), k = 0, 1, ...  Row-major codes take LPR = 2 (64 elements per
// lane at head_dim 128: six of the rotation's seven butterfly stages inside
// the lane), in persistent CTAs that walk a list of blocks and stage each in
// shared memory with asynchronous copies, two blocks ahead, so that loads
// overlap the arithmetic.  Packed sequences take LPR = 4 with direct loads.
// The transposed output takes LPR = 32, one CTA per block, so that a lane
// holds 16 consecutive rows of each of its
// elements and writes them as 16 consecutive bytes.  Butterflies with
// stride h < E pair elements inside a lane; larger strides pair lane l with
// lane l ^ (h / E) through a shuffle, the lower index taking u + v and the
// upper u - v (u the lower element, v the upper), written as
// fma(+-1, own, partner), which rounds exactly like that sum or difference.
// Every step is the float32 operation, in the order, of the definition:
// signs multiply, butterflies with stride 1, 2, 4, ..., d/2, one multiply
// by the float32 value of 1/sqrt(d); the scale and its inverse are
// IEEE-rounded float32 divisions; codes are rounded to nearest e4m3, ties to
// even, saturating.
//
// One scale per plane: a first pass takes each block's amax and combines
// them per plane with an integer atomic max on the float's bits (amax >= 0,
// where the bit patterns order like the values); the second pass quantises;
// a last, one-thread-per-plane pass turns the stored amax into the scale.
#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "attn_internal.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kBlockRows = 128;                 // rows per CTA
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kWarpRows = kBlockRows / kWarps;  // 16 rows per warp
constexpr float kE4M3Max = 448.f;

__device__ __forceinline__ uint32_t e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Lane geometry: E elements per lane, RW rows per warp-wide step, RPL rows
// per lane.
template <int D, int LPR>
struct Geom {
  static constexpr int E = D / LPR;
  static constexpr int RW = 32 / LPR;
  static constexpr int RPL = kWarpRows / RW;
  static_assert(E % 2 == 0 && RPL >= 1, "lane geometry");
};

// The lane's rows (row0w + k RW + lane / LPR, k < RPL) as raw bf16 pairs from
// global memory: w[k][i] holds elements E c + 2 i and E c + 2 i + 1 (c = lane %
// LPR) of row k; zero from row_end on.
template <int D, int LPR>
__device__ __forceinline__ void load_raw(const QuantArgs& a, int plane, int row0w, int lane,
                                         uint32_t (&w)[Geom<D, LPR>::RPL][Geom<D, LPR>::E / 2],
                                         int row_end) {
  using G = Geom<D, LPR>;
  constexpr int E = G::E;
  const int c = lane % LPR;
#pragma unroll
  for (int k = 0; k < G::RPL; ++k) {
    const int row = row0w + k * G::RW + lane / LPR;
    if (row < row_end) {
      const uint16_t* src = a.x + ((size_t)plane * a.rows + row) * D + c * E;
      if constexpr (E >= 8) {
#pragma unroll
        for (int i = 0; i < E / 8; ++i) {
          const uint4 u = reinterpret_cast<const uint4*>(src)[i];
          w[k][4 * i] = u.x; w[k][4 * i + 1] = u.y; w[k][4 * i + 2] = u.z; w[k][4 * i + 3] = u.w;
        }
      } else if constexpr (E == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(src);
        w[k][0] = u.x; w[k][1] = u.y;
      } else {
        w[k][0] = *reinterpret_cast<const uint32_t*>(src);
      }
    } else {
#pragma unroll
      for (int i = 0; i < E / 2; ++i) w[k][i] = 0u;
    }
  }
}

// Blocks of 128 rows staged in shared memory: row r of the block takes D * 2
// bytes, its 16-byte chunk j stored at chunk stage_chunk<D>(r, j) of the row.
// The reads below give two lanes to a row, so the eight lanes of a 16-byte
// load phase read the same chunk slot of four consecutive rows, which would
// all fall on the same banks (rows are 128 or 256 bytes); the permutation
// (an XOR within each group of eight chunks, by the row and the half of the
// row) puts those eight reads, and the copies' writes, on distinct banks.
template <int D>
__device__ __forceinline__ int stage_chunk(int r, int j) {
  if constexpr (D == 128)
    return j ^ (((r & 3) << 1) | (j >> 3));
  else
    return j ^ (r & 3);
}

template <int D>
constexpr int stage_bytes() {
  return kBlockRows * D * 2;
}

// Copies rows [r0, r1) of a plane into a stage (r0 is the block's first row),
// one 16-byte chunk per thread and step; the caller commits the group.
template <int D>
__device__ __forceinline__ void stage_rows(const QuantArgs& a, int plane, int r0, int r1,
                                           uint32_t sbuf) {
  constexpr int kCpr = D * 2 / 16;  // chunks per row
  const int n = (r1 - r0) * kCpr;
  const uint16_t* src = a.x + ((size_t)plane * a.rows + r0) * D;
  for (int idx = threadIdx.x; idx < n; idx += kThreads) {
    const int r = idx / kCpr, j = idx % kCpr;
    cp_async16(sbuf + (uint32_t)(r * D * 2 + stage_chunk<D>(r, j) * 16),
               src + (size_t)r * D + j * 8);
  }
}

// load_raw's result (two lanes per row) from a staged block; lrow0w is
// row0w's row within the block.
template <int D>
__device__ __forceinline__ void load_raw_staged(const uint8_t* stage, int lrow0w, int row0w,
                                                int lane,
                                                uint32_t (&w)[Geom<D, 2>::RPL][Geom<D, 2>::E / 2],
                                                int row_end) {
  using G = Geom<D, 2>;
  constexpr int E = G::E;  // whole chunks: 64 or 32 elements
  const int c = lane % 2;
#pragma unroll
  for (int k = 0; k < G::RPL; ++k) {
    const int dr = k * G::RW + lane / 2;
    if (row0w + dr < row_end) {
      const int lr = lrow0w + dr;
      const uint8_t* rowp = stage + lr * (D * 2);
#pragma unroll
      for (int i = 0; i < E / 8; ++i) {
        const uint4 u =
            *reinterpret_cast<const uint4*>(rowp + stage_chunk<D>(lr, c * (E / 8) + i) * 16);
        w[k][4 * i] = u.x; w[k][4 * i + 1] = u.y; w[k][4 * i + 2] = u.z; w[k][4 * i + 3] = u.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < E / 2; ++i) w[k][i] = 0u;
    }
  }
}

// The rows as float32, rotated when signs (global memory, or shared memory
// and 16-byte aligned when SMEM_SIGNS) are given: x[k][e] is element
// E (lane % LPR) + e of the lane's row k.
template <int D, int LPR, bool SMEM_SIGNS = false>
__device__ __forceinline__ void rotate_rows(const float* signs, float inv_sqrt_d, int lane,
                                            const uint32_t (&w)[Geom<D, LPR>::RPL][Geom<D, LPR>::E / 2],
                                            float (&x)[Geom<D, LPR>::RPL][Geom<D, LPR>::E]) {
  using G = Geom<D, LPR>;
  constexpr int E = G::E;
  const int c = lane % LPR;
#pragma unroll
  for (int k = 0; k < G::RPL; ++k)
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
      x[k][2 * i] = __uint_as_float(w[k][i] << 16);
      x[k][2 * i + 1] = __uint_as_float(w[k][i] & 0xffff0000u);
    }
  if (signs == nullptr) return;
  // Pairs of elements go through the packed two-lane float32 instructions
  // (each half rounded on its own, as the scalar operation).
  float2 sg[E / 2];
  if constexpr (SMEM_SIGNS) {
#pragma unroll
    for (int e = 0; e < E; e += 4) {
      const float4 t = *reinterpret_cast<const float4*>(signs + c * E + e);
      sg[e / 2] = make_float2(t.x, t.y);
      sg[e / 2 + 1] = make_float2(t.z, t.w);
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; e += 2) sg[e / 2] = make_float2(signs[c * E + e], signs[c * E + e + 1]);
  }
  const float2 neg1 = make_float2(-1.f, -1.f);
  const float2 isd = make_float2(inv_sqrt_d, inv_sqrt_d);
#pragma unroll
  for (int k = 0; k < G::RPL; ++k) {
    float* xr = x[k];
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 t = mul2(make_float2(xr[e], xr[e + 1]), sg[e / 2]);
      xr[e] = t.x;
      xr[e + 1] = t.y;
    }
    // strides inside the lane: (u, v) -> (u + v, u - v), u - v as fma(-1, v, u)
    if constexpr (E == 2) {
      const float u = xr[0], v = xr[1];
      xr[0] = __fadd_rn(u, v);
      xr[1] = __fsub_rn(u, v);
    } else {
      // stride 1: butterflies (e, e + 1) and (e + 2, e + 3) side by side
#pragma unroll
      for (int e = 0; e < E; e += 4) {
        const float2 u = make_float2(xr[e], xr[e + 2]), v = make_float2(xr[e + 1], xr[e + 3]);
        const float2 sm = add2(u, v), df = fma2(neg1, v, u);
        xr[e] = sm.x; xr[e + 1] = df.x; xr[e + 2] = sm.y; xr[e + 3] = df.y;
      }
      // stride h >= 2: butterflies (e, e + h) and (e + 1, e + 1 + h) side by side
#pragma unroll
      for (int h = 2; h < E; h <<= 1)
#pragma unroll
        for (int e = 0; e < E; e += 2)
          if ((e & h) == 0) {
            const float2 u = make_float2(xr[e], xr[e + 1]), v = make_float2(xr[e + h], xr[e + h + 1]);
            const float2 sm = add2(u, v), df = fma2(neg1, v, u);
            xr[e] = sm.x; xr[e + 1] = sm.y; xr[e + h] = df.x; xr[e + h + 1] = df.y;
          }
    }
    // strides across the row's lanes: the lower element becomes own + partner,
    // the upper partner - own, both as fma(+-1, own, partner)
#pragma unroll
    for (int hl = 1; hl < LPR; hl <<= 1) {
      const float sgn = (lane & hl) ? -1.f : 1.f;
      const float2 sgn2 = make_float2(sgn, sgn);
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        const float y0 = __shfl_xor_sync(0xffffffffu, xr[e], hl);
        const float y1 = __shfl_xor_sync(0xffffffffu, xr[e + 1], hl);
        const float2 t = fma2(sgn2, make_float2(xr[e], xr[e + 1]), make_float2(y0, y1));
        xr[e] = t.x;
        xr[e + 1] = t.y;
      }
    }
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 t = mul2(make_float2(xr[e], xr[e + 1]), isd);
      xr[e] = t.x;
      xr[e + 1] = t.y;
    }
  }
}

// The lane's rows from global memory, rotated when signs are given (zero from
// row_end on).
template <int D, int LPR>
__device__ __forceinline__ void load_rows(const QuantArgs& a, int plane, int row0w, int lane,
                                          float (&x)[Geom<D, LPR>::RPL][Geom<D, LPR>::E],
                                          int row_end) {
  uint32_t w[Geom<D, LPR>::RPL][Geom<D, LPR>::E / 2];
  load_raw<D, LPR>(a, plane, row0w, lane, w, row_end);
  rotate_rows<D, LPR>(a.signs, a.inv_sqrt_d, lane, w, x);
}

// Largest |x| over the CTA's rows (every thread gets it).
template <int D, int LPR>
__device__ __forceinline__ float block_amax(const float (&x)[Geom<D, LPR>::RPL][Geom<D, LPR>::E],
                                            float* red) {
  using G = Geom<D, LPR>;
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < G::RPL; ++k)
#pragma unroll
    for (int e = 0; e < G::E; ++e) m = fmaxf(m, fabsf(x[k][e]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  float b = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) b = fmaxf(b, red[w]);
  return b;
}

// Codes of the lane's rows: row-major (row, d) with LPR = 4, or transposed
// (d, row) with LPR = 32.
template <int D, int LPR>
__device__ __forceinline__ void store_codes(const QuantArgs& a, int plane, int row0w, int lane,
                                            const float (&x)[Geom<D, LPR>::RPL][Geom<D, LPR>::E],
                                            float inv, int row_end) {
  using G = Geom<D, LPR>;
  constexpr int E = G::E;
  const int c = lane % LPR;
  const float2 inv2 = make_float2(inv, inv);
  // codes of element pairs: bits 0-7 element e, bits 8-15 element e + 1
  uint32_t pr[G::RPL][E / 2];
#pragma unroll
  for (int k = 0; k < G::RPL; ++k)
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 t = mul2(make_float2(x[k][e], x[k][e + 1]), inv2);
      pr[k][e / 2] = e4m3x2(t.y, t.x);
    }
  if constexpr (LPR != 32) {
#pragma unroll
    for (int k = 0; k < G::RPL; ++k) {
      const int row = row0w + k * G::RW + lane / LPR;
      if (row >= row_end) continue;
      uint8_t* dst = a.codes + ((size_t)plane * a.rows + row) * D + c * E;
      uint32_t wd[E / 4];
#pragma unroll
      for (int i = 0; i < E / 4; ++i) wd[i] = pr[k][2 * i] | (pr[k][2 * i + 1] << 16);
      if constexpr (E >= 16) {
#pragma unroll
        for (int i = 0; i < E / 16; ++i)
          reinterpret_cast<uint4*>(dst)[i] = make_uint4(wd[4 * i], wd[4 * i + 1], wd[4 * i + 2], wd[4 * i + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < E / 4; ++i) reinterpret_cast<uint32_t*>(dst)[i] = wd[i];
      }
    }
  } else {
    // (plane, d, rows): the lane's 16 rows (row0w ..) of element d are 16
    // consecutive bytes.
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int sh = (e & 1) * 8;
      uint8_t* dst = a.codes + ((size_t)plane * D + (size_t)(c * E + e)) * a.rows + row0w;
      if ((a.rows & 15) == 0 && row0w + kWarpRows <= a.rows) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          w[q] = 0;
#pragma unroll
          for (int b = 0; b < 4; ++b) w[q] |= ((pr[4 * q + b][e / 2] >> sh) & 0xffu) << (8 * b);
        }
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
      } else {
#pragma unroll
        for (int k = 0; k < G::RPL; ++k)
          if (row0w + k < a.rows) dst[k] = (uint8_t)(pr[k][e / 2] >> sh);
      }
    }
  }
}

// One scale per block of 128 rows: amax, scale and codes in one pass, for
// block `blk` of `plane` (nblk blocks per plane).
template <int D, int LPR>
__device__ __forceinline__ void quantize_block(const QuantArgs& a, int plane, int blk, int nblk,
                                               float* red) {
  using G = Geom<D, LPR>;
  const int lane = threadIdx.x & 31;
  const int row0w = blk * kBlockRows + (threadIdx.x >> 5) * kWarpRows;
  float x[G::RPL][G::E];
  load_rows<D, LPR>(a, plane, row0w, lane, x, a.rows);
  float amax = block_amax<D, LPR>(x, red);
  if (amax == 0.f) amax = 1.f;
  if (threadIdx.x == 0) a.scales[(size_t)plane * nblk + blk] = __fdiv_rn(amax, kE4M3Max);
  store_codes<D, LPR>(a, plane, row0w, lane, x, __fdiv_rn(kE4M3Max, amax), a.rows);
}

// Packed sequences: CTA (T, plane) quantises tile T of the list of every
// sequence's 128-row tiles (tiles start at their sequence's first row), its
// scale at column T.  One warp first reads cu_seqlens, clamps each sequence
// into [0, rows] as the packed prefill does, and scans the tile counts.
template <int D>
__global__ void __launch_bounds__(kThreads) packed_block_kernel(const QuantArgs a) {
  using G = Geom<D, 4>;
  __shared__ float red[kWarps];
  __shared__ int seq_start[kMaxVarlenSeqs], seq_end[kMaxVarlenSeqs], prefix[kMaxVarlenSeqs + 1];
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int base = 0; base < a.num_seqs; base += 32) {
      const int s = base + lane;
      int st = 0, en = 0;
      if (s < a.num_seqs) {
        st = min(max(a.cu_seqlens[s], 0), a.rows);
        en = min(max(a.cu_seqlens[s + 1], st), a.rows);
      }
      int incl = (en - st + kBlockRows - 1) / kBlockRows;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (s < a.num_seqs) {
        seq_start[s] = st;
        seq_end[s] = en;
        prefix[s + 1] = carry + incl;
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) prefix[0] = 0;
  }
  __syncthreads();
  const int T = blockIdx.x, plane = blockIdx.y;
  if (T >= prefix[a.num_seqs]) return;  // beyond the last tile
  int lo = 0, hi = a.num_seqs - 1;       // the last sequence whose tiles start at or before T
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= T) lo = mid; else hi = mid - 1;
  }
  const int r0 = seq_start[lo] + (T - prefix[lo]) * kBlockRows;
  const int r1 = min(r0 + kBlockRows, seq_end[lo]);
  const int lane = threadIdx.x & 31;
  const int row0w = r0 + (threadIdx.x >> 5) * kWarpRows;
  float x[G::RPL][G::E];
  load_rows<D, 4>(a, plane, row0w, lane, x, r1);
  float amax = block_amax<D, 4>(x, red);
  if (amax == 0.f) amax = 1.f;
  if (threadIdx.x == 0) a.scales[(size_t)plane * a.tiles + T] = __fdiv_rn(amax, kE4M3Max);
  store_codes<D, 4>(a, plane, row0w, lane, x, __fdiv_rn(kE4M3Max, amax), r1);
}

template <int D, int LPR>
__global__ void __launch_bounds__(kThreads) quantize_block_kernel(const QuantArgs a) {
  __shared__ float red[kWarps];
  quantize_block<D, LPR>(a, blockIdx.y, blockIdx.x, gridDim.x, red);
}

// Blocks of 128 rows with two lanes per row, staged through shared memory:
// block b of the concatenated lists (q's blocks, then k's: codes and one
// scale per block; then v's: the block's amax folded into its plane's).  Any
// list may be empty (planes = 0).  Persistent CTAs walk the blocks b =
// blockIdx.x + i gridDim.x; kStages stages keep the copies of the next
// blocks in flight while a block is rotated, reduced and written.
constexpr int kStages = 3;

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
staged_blocks_kernel(const __grid_constant__ QuantArgs q, const __grid_constant__ QuantArgs k,
                     const __grid_constant__ QuantArgs v, int nblk) {
  using G = Geom<D, 2>;
  extern __shared__ __align__(16) uint8_t stage_mem[];
  __shared__ float red[kWarps];
  __shared__ __align__(16) float sgn[3][D];  // each list's signs, read 4 at a time
  const uint32_t sbase = smem_u32(stage_mem);
  for (int i = threadIdx.x; i < 3 * D; i += kThreads) {
    const float* g = i < D ? q.signs : (i < 2 * D ? k.signs : v.signs);
    sgn[i / D][i % D] = g != nullptr ? g[i % D] : 0.f;
  }  // visible after the first __syncthreads below
  // 64-bit list indices: planes x blocks may exceed the int range
  const long long nq = (long long)q.planes * nblk, nk = (long long)k.planes * nblk;
  const long long total = nq + nk + (long long)v.planes * nblk;
  const long long step = gridDim.x;
  // list index -> (tensor, plane, block)
  auto locate = [&](long long b, int& which, int& plane, int& blk) {
    which = b < nq ? 0 : (b < nq + nk ? 1 : 2);
    const long long lb = which == 0 ? b : (which == 1 ? b - nq : b - nq - nk);
    plane = static_cast<int>(lb / nblk);
    blk = static_cast<int>(lb - (long long)plane * nblk);
  };
  auto args = [&](int which) -> const QuantArgs& { return which == 0 ? q : (which == 1 ? k : v); };
  auto issue = [&](long long b, int stage) {
    int which, plane, blk;
    locate(b, which, plane, blk);
    const QuantArgs& a = args(which);
    const int r0 = blk * kBlockRows;
    stage_rows<D>(a, plane, r0, min(r0 + kBlockRows, a.rows),
                  sbase + (uint32_t)(stage * stage_bytes<D>()));
  };
#pragma unroll 1
  for (int s = 0; s < kStages - 1; ++s) {
    const long long b = blockIdx.x + s * step;
    if (b < total) issue(b, s);
    cp_async_commit();  // possibly empty: every thread counts the same groups
  }
  const int lane = threadIdx.x & 31;
  const int lrow0w = (threadIdx.x >> 5) * kWarpRows;
  int it = 0;
#pragma unroll 1
  for (long long b = blockIdx.x; b < total; ++it, b += step) {
    cp_async_wait<kStages - 2>();  // this thread's copies of block b have landed
    __syncthreads();               // everyone's have; the stage read in the last round is free
    {
      const long long bn = b + (kStages - 1) * step;
      if (bn < total) issue(bn, (it + kStages - 1) % kStages);
      cp_async_commit();
    }
    int which, plane, blk;
    locate(b, which, plane, blk);
    const QuantArgs& a = args(which);
    const int row0w = blk * kBlockRows + lrow0w;
    float x[G::RPL][G::E];
    {
      uint32_t w[G::RPL][G::E / 2];
      load_raw_staged<D>(stage_mem + (it % kStages) * stage_bytes<D>(), lrow0w, row0w, lane, w,
                         a.rows);
      if (a.signs != nullptr)
        rotate_rows<D, 2, true>(sgn[which], a.inv_sqrt_d, lane, w, x);
      else
        rotate_rows<D, 2>(nullptr, a.inv_sqrt_d, lane, w, x);
    }
    float amax = block_amax<D, 2>(x, red);
    if (which == 2) {
      if (threadIdx.x == 0)
        atomicMax(reinterpret_cast<unsigned int*>(a.scales) + plane, __float_as_uint(amax));
    } else {
      if (amax == 0.f) amax = 1.f;
      if (threadIdx.x == 0) a.scales[(size_t)plane * nblk + blk] = __fdiv_rn(amax, kE4M3Max);
      store_codes<D, 2>(a, plane, row0w, lane, x, __fdiv_rn(kE4M3Max, amax), a.rows);
    }
  }
  cp_async_wait<0>();
}

// Launches staged_blocks_kernel over the three lists: at most two CTAs per SM
// (the stages take 3 x 32 KB at head_dim 128), no more CTAs than blocks.
template <int D>
cudaError_t launch_staged(const QuantArgs& q, const QuantArgs& k, const QuantArgs& v, int nblk,
                          const LaunchCtx& ctx) {
  constexpr int kSmem = kStages * stage_bytes<D>();
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(staged_blocks_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev] = true;
  }
  const long long total = (long long)(q.planes + k.planes + v.planes) * nblk;
  const int grid = (int)std::min<long long>(total, 2LL * std::max(ctx.num_sms, 1));
  if (grid < 1) return cudaSuccess;
  staged_blocks_kernel<D><<<grid, kThreads, kSmem, ctx.stream>>>(q, k, v, nblk);
  return cudaGetLastError();
}

// Pass 2: the codes, from the plane's amax.
template <int D, int LPR>
__global__ void __launch_bounds__(kThreads) plane_codes_kernel(const QuantArgs a) {
  using G = Geom<D, LPR>;
  const int plane = blockIdx.y, lane = threadIdx.x & 31;
  const int row0w = blockIdx.x * kBlockRows + (threadIdx.x >> 5) * kWarpRows;
  float x[G::RPL][G::E];
  load_rows<D, LPR>(a, plane, row0w, lane, x, a.rows);
  float amax = __uint_as_float(reinterpret_cast<const unsigned int*>(a.scales)[plane]);
  if (amax == 0.f) amax = 1.f;
  store_codes<D, LPR>(a, plane, row0w, lane, x, __fdiv_rn(kE4M3Max, amax), a.rows);
}

// Pass 3: amax -> scale, in place.
__global__ void plane_scale_kernel(const QuantArgs a) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= a.planes) return;
  float amax = __uint_as_float(reinterpret_cast<const unsigned int*>(a.scales)[p]);
  if (amax == 0.f) amax = 1.f;
  a.scales[p] = __fdiv_rn(amax, kE4M3Max);
}

template <int D, int LPR>
cudaError_t launch_quantize_t(const QuantArgs& a, const LaunchCtx& ctx) {
  const int nblk = (a.rows + kBlockRows - 1) / kBlockRows;
  const dim3 grid((unsigned)nblk, (unsigned)a.planes);
  QuantArgs none = a;
  none.planes = 0;
  if (a.block_rows > 0) {
    if constexpr (LPR == 4) {
      return launch_staged<D>(a, none, none, nblk, ctx);
    } else {
      quantize_block_kernel<D, LPR><<<grid, kThreads, 0, ctx.stream>>>(a);
      return cudaGetLastError();
    }
  }
  cudaError_t e = cudaMemsetAsync(a.scales, 0, (size_t)a.planes * sizeof(float), ctx.stream);
  if (e != cudaSuccess) return e;
  e = launch_staged<D>(none, none, a, nblk, ctx);
  if (e != cudaSuccess) return e;
  plane_codes_kernel<D, LPR><<<grid, kThreads, 0, ctx.stream>>>(a);
  plane_scale_kernel<<<(a.planes + 127) / 128, 128, 0, ctx.stream>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_quantize_d(const QuantArgs& a, const LaunchCtx& ctx) {
  if (a.cu_seqlens) {
    packed_block_kernel<D><<<dim3((unsigned)a.tiles, (unsigned)a.planes), kThreads, 0,
                             ctx.stream>>>(a);
    return cudaGetLastError();
  }
  return a.transpose ? launch_quantize_t<D, 32>(a, ctx) : launch_quantize_t<D, 4>(a, ctx);
}

// Q, K (block scales, rotated when signs are given) and V (plane scales,
// transposed): the first pass of all three in one launch, then V's codes and
// scales.
template <int D>
cudaError_t launch_quantize_qkv_d(const QuantArgs& q, const QuantArgs& k, const QuantArgs& v,
                                  const LaunchCtx& ctx) {
  const int nblk = (q.rows + kBlockRows - 1) / kBlockRows;
  cudaError_t e = cudaMemsetAsync(v.scales, 0, (size_t)v.planes * sizeof(float), ctx.stream);
  if (e != cudaSuccess) return e;
  e = launch_staged<D>(q, k, v, nblk, ctx);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)nblk, (unsigned)v.planes);
  plane_codes_kernel<D, 32><<<grid, kThreads, 0, ctx.stream>>>(v);
  plane_scale_kernel<<<(v.planes + 127) / 128, 128, 0, ctx.stream>>>(v);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const QuantArgs& a, const LaunchCtx& ctx) {
  return a.head_dim == 128 ? launch_quantize_d<128>(a, ctx) : launch_quantize_d<64>(a, ctx);
}

cudaError_t launch_quantize_qkv(const QuantArgs& q, const QuantArgs& k, const QuantArgs& v,
                                const LaunchCtx& ctx) {
  return q.head_dim == 128 ? launch_quantize_qkv_d<128>(q, k, v, ctx)
                           : launch_quantize_qkv_d<64>(q, k, v, ctx);
}

}  // namespace attn
