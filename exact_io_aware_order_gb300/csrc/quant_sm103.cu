// FP8 (e4m3) block quantisation with incoherent processing, sm_103a.
//
// Page "FlashAttention for inference: tiled prefill and split-KV decoding",
// section "Interaction with post-trained models": FlashAttention-3's FP8
// path lowers the error of naive FP8 attention by block quantisation and
// incoherent processing.  This kernel prepares the inputs of the FP8
// prefill: optionally rotates each row by diag(signs) H / sqrt(d) (H the
// Sylvester Hadamard matrix; the same rotation for Q and K leaves Q K^T
// unchanged), then quantises blocks of rows to e4m3 with scale amax / 448.
//
// One thread per row, one CTA per block of 128 rows (or per plane when the
// whole plane shares one scale, looping over its rows twice: amax, codes).
// The rotation runs as in-register butterflies, stride 1, 2, 4, ..., d/2,
// then one multiply by the float32 value of 1/sqrt(d); the scale and its
// inverse are IEEE-rounded float32 divisions; codes are rounded to nearest
// e4m3, ties to even, saturating.  The transposed output (plane, d, rows)
// is written by consecutive threads to consecutive bytes.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kQRows = 128;  // rows per CTA pass (one per thread)
constexpr float kE4M3Max = 448.f;

__device__ __forceinline__ uint32_t e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Loads row `row` of the plane (zero past the end) as float32, optionally
// rotated.
template <int D>
__device__ __forceinline__ void load_row(const QuantArgs& a, int plane, int row, float (&x)[D]) {
  if (row < a.rows) {
    const uint4* src = reinterpret_cast<const uint4*>(a.x + ((size_t)plane * a.rows + row) * D);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const uint4 u = src[c];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[c * 8 + 2 * i] = __uint_as_float(w[i] << 16);
        x[c * 8 + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < D; ++i) x[i] = 0.f;
  }
  if (a.signs) {
#pragma unroll
    for (int i = 0; i < D; ++i) x[i] = __fmul_rn(x[i], a.signs[i]);
#pragma unroll
    for (int h = 1; h < D; h <<= 1)
#pragma unroll
      for (int b = 0; b < D; b += 2 * h)
#pragma unroll
        for (int i = 0; i < h; ++i) {
          const float u = x[b + i], v = x[b + i + h];
          x[b + i] = __fadd_rn(u, v);
          x[b + i + h] = __fsub_rn(u, v);
        }
    // float32 value of 1/sqrt(d), rounded once from the exact value by the host
#pragma unroll
    for (int i = 0; i < D; ++i) x[i] = __fmul_rn(x[i], a.inv_sqrt_d);
  }
}

template <int D>
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int w = 1; w < kQRows / 32; ++w) m = fmaxf(m, red[w]);
  return m;
}

template <int D>
__device__ __forceinline__ void store_row(const QuantArgs& a, int plane, int row,
                                          const float (&x)[D], float inv) {
  if (row >= a.rows) return;
  uint32_t wds[D / 4];
#pragma unroll
  for (int i = 0; i < D / 4; ++i) {
    const uint32_t lo = e4m3x2(__fmul_rn(x[4 * i + 1], inv), __fmul_rn(x[4 * i], inv));
    const uint32_t hi = e4m3x2(__fmul_rn(x[4 * i + 3], inv), __fmul_rn(x[4 * i + 2], inv));
    wds[i] = lo | (hi << 16);  // element k of the row in byte k
  }
  if (!a.transpose) {
    uint4* dst = reinterpret_cast<uint4*>(a.codes + ((size_t)plane * a.rows + row) * D);
#pragma unroll
    for (int c = 0; c < D / 16; ++c)
      dst[c] = make_uint4(wds[4 * c], wds[4 * c + 1], wds[4 * c + 2], wds[4 * c + 3]);
  } else {
    // (plane, d, rows): column `row` of each d-row; a warp writes 32 bytes.
    uint8_t* dst = a.codes + (size_t)plane * D * a.rows + row;
#pragma unroll
    for (int k = 0; k < D; ++k) dst[(size_t)k * a.rows] = (uint8_t)(wds[k >> 2] >> (8 * (k & 3)));
  }
}

template <int D>
__global__ void __launch_bounds__(kQRows) quantize_kernel(const QuantArgs a) {
  __shared__ float red[kQRows / 32];
  const int plane = blockIdx.y;
  float x[D];
  if (a.block_rows > 0) {
    // One scale per block of 128 rows: this CTA's block.
    const int row = blockIdx.x * kQRows + threadIdx.x;
    load_row<D>(a, plane, row, x);
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < D; ++i) m = fmaxf(m, fabsf(x[i]));
    float amax = block_max<D>(m, red);
    if (amax == 0.f) amax = 1.f;
    const float inv = __fdiv_rn(kE4M3Max, amax);
    if (threadIdx.x == 0) a.scales[(size_t)plane * gridDim.x + blockIdx.x] = __fdiv_rn(amax, kE4M3Max);
    store_row<D>(a, plane, row, x, inv);
  } else {
    // One scale for the whole plane: amax over every row, then the codes.
    float m = 0.f;
    for (int r0 = 0; r0 < a.rows; r0 += kQRows) {
      load_row<D>(a, plane, r0 + threadIdx.x, x);
#pragma unroll
      for (int i = 0; i < D; ++i) m = fmaxf(m, fabsf(x[i]));
    }
    float amax = block_max<D>(m, red);
    if (amax == 0.f) amax = 1.f;
    const float inv = __fdiv_rn(kE4M3Max, amax);
    if (threadIdx.x == 0) a.scales[plane] = __fdiv_rn(amax, kE4M3Max);
    for (int r0 = 0; r0 < a.rows; r0 += kQRows) {
      load_row<D>(a, plane, r0 + threadIdx.x, x);
      store_row<D>(a, plane, r0 + threadIdx.x, x, inv);
    }
  }
}

}  // namespace

cudaError_t launch_quantize(const QuantArgs& a, const LaunchCtx& ctx) {
  const unsigned nb = a.block_rows > 0 ? (unsigned)((a.rows + kQRows - 1) / kQRows) : 1u;
  const dim3 grid(nb, (unsigned)a.planes);
  if (a.head_dim == 128)
    quantize_kernel<128><<<grid, kQRows, 0, ctx.stream>>>(a);
  else
    quantize_kernel<64><<<grid, kQRows, 0, ctx.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace attn
