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
// Layout of the work: one CTA per block of 128 rows of a plane, eight warps
// of 16 rows each.  Within a warp, LPR consecutive lanes share a row: lane l
// holds elements [E c, E c + E) (c = l % LPR, E = d / LPR) of the rows
// l / LPR + k (32 / LPR), k = 0, 1, ...  Row-major output takes LPR = 4 (32
// elements per lane at head_dim 128: 64-byte loads, five of the rotation's
// seven butterfly stages inside the lane); the transposed output takes
// LPR = 32, so that a lane holds 16 consecutive rows of each of its
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

// The lane's rows (row0w + k RW + lane / LPR, k < RPL; zero from row_end on),
// rotated when signs are given: x[k][e] is element E (lane % LPR) + e.
template <int D, int LPR>
__device__ __forceinline__ void load_rows(const QuantArgs& a, int plane, int row0w, int lane,
                                          float (&x)[Geom<D, LPR>::RPL][Geom<D, LPR>::E],
                                          int row_end) {
  using G = Geom<D, LPR>;
  constexpr int E = G::E;
  const int c = lane % LPR;
#pragma unroll
  for (int k = 0; k < G::RPL; ++k) {
    const int row = row0w + k * G::RW + lane / LPR;
    if (row < row_end) {
      const uint16_t* src = a.x + ((size_t)plane * a.rows + row) * D + c * E;
      uint32_t w[E / 2];
      if constexpr (E >= 8) {
#pragma unroll
        for (int i = 0; i < E / 8; ++i) {
          const uint4 u = reinterpret_cast<const uint4*>(src)[i];
          w[4 * i] = u.x; w[4 * i + 1] = u.y; w[4 * i + 2] = u.z; w[4 * i + 3] = u.w;
        }
      } else if constexpr (E == 4) {
        const uint2 u = *reinterpret_cast<const uint2*>(src);
        w[0] = u.x; w[1] = u.y;
      } else {
        w[0] = *reinterpret_cast<const uint32_t*>(src);
      }
#pragma unroll
      for (int i = 0; i < E / 2; ++i) {
        x[k][2 * i] = __uint_as_float(w[i] << 16);
        x[k][2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) x[k][e] = 0.f;
    }
  }
  if (a.signs == nullptr) return;
  // Pairs of elements go through the packed two-lane float32 instructions
  // (each half rounded on its own, as the scalar operation).
  float2 sg[E / 2];
#pragma unroll
  for (int e = 0; e < E; e += 2) sg[e / 2] = make_float2(a.signs[c * E + e], a.signs[c * E + e + 1]);
  const float2 neg1 = make_float2(-1.f, -1.f);
  const float2 isd = make_float2(a.inv_sqrt_d, a.inv_sqrt_d);
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

// One scale per plane, pass 1: block `blk`'s amax folded into the plane's,
// kept as float bits in scales[plane] (zeroed before the launch).
template <int D>
__device__ __forceinline__ void plane_amax_block(const QuantArgs& a, int plane, int blk,
                                                 float* red) {
  using G = Geom<D, 4>;
  const int lane = threadIdx.x & 31;
  const int row0w = blk * kBlockRows + (threadIdx.x >> 5) * kWarpRows;
  float x[G::RPL][G::E];
  load_rows<D, 4>(a, plane, row0w, lane, x, a.rows);
  const float amax = block_amax<D, 4>(x, red);
  if (threadIdx.x == 0)
    atomicMax(reinterpret_cast<unsigned int*>(a.scales) + plane, __float_as_uint(amax));
}

template <int D>
__global__ void __launch_bounds__(kThreads) plane_amax_kernel(const QuantArgs a) {
  __shared__ float red[kWarps];
  plane_amax_block<D>(a, blockIdx.y, blockIdx.x, red);
}

// Q and K with block scales and V's plane amax in one launch: CTA b takes
// block b of the concatenated lists (Q blocks, then K blocks, then V blocks).
template <int D>
__global__ void __launch_bounds__(kThreads) qkv_pass1_kernel(const QuantArgs q, const QuantArgs k,
                                                             const QuantArgs v, int nblk) {
  __shared__ float red[kWarps];
  int b = blockIdx.x;
  const int nq = q.planes * nblk, nk = k.planes * nblk;
  if (b < nq) {
    quantize_block<D, 4>(q, b / nblk, b % nblk, nblk, red);
  } else if ((b -= nq) < nk) {
    quantize_block<D, 4>(k, b / nblk, b % nblk, nblk, red);
  } else {
    b -= nk;
    plane_amax_block<D>(v, b / nblk, b % nblk, red);
  }
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
  const dim3 grid((unsigned)((a.rows + kBlockRows - 1) / kBlockRows), (unsigned)a.planes);
  if (a.block_rows > 0) {
    quantize_block_kernel<D, LPR><<<grid, kThreads, 0, ctx.stream>>>(a);
    return cudaGetLastError();
  }
  cudaError_t e = cudaMemsetAsync(a.scales, 0, (size_t)a.planes * sizeof(float), ctx.stream);
  if (e != cudaSuccess) return e;
  plane_amax_kernel<D><<<grid, kThreads, 0, ctx.stream>>>(a);
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
  const unsigned blocks = (unsigned)((q.planes + k.planes + v.planes) * nblk);
  qkv_pass1_kernel<D><<<blocks, kThreads, 0, ctx.stream>>>(q, k, v, nblk);
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
