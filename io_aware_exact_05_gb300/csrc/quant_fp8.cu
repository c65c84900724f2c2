// quant_fp8.cu -- per-head e4m3 quantisation of bf16 attention operands, with
// the optional rotation of incoherent processing.
//
// FP8 computation and incoherent processing are the FlashAttention-3
// techniques of "Flash Attention: Revolutionizing Transformer Efficiency"
// (section FlashAttention-3, items 2 and 3).  A head X [n][128] is encoded as
// codes c = round_e4m3(y * 448 / amax(|y|)) with descale = amax / 448, where
// y = X, or for incoherent processing y = X diag(s) H_128 / sqrt(128) with H
// the Sylvester Hadamard matrix and s a vector of signs (the same rotation
// for Q and K leaves Q K^T unchanged and spreads large entries over the row).
// The Hadamard product is unnormalised in the kernel (y' = sqrt(128) y); the
// factor cancels in the codes and is folded into the descale.
//
// Two passes over X (the head's maximum is needed before any code): an amax
// kernel writes one partial maximum per 128-row block, and the quantise
// kernel reduces its head's partials, then writes the codes, row-major or
// transposed ([128][n], for V).  Each warp holds one row at a time, four
// consecutive values per lane, and transforms it with two in-register and
// five shuffle butterfly stages.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm100.cuh"

namespace attn {
namespace {

constexpr int kD = 128;          // head dim
constexpr int kRows = 128;       // rows per block
constexpr int kThreads = 256;    // 8 warps x 16 rows
constexpr int kRowsPerWarp = kRows / (kThreads / 32);
constexpr int kTilePitch = kRows + 16;   // bytes per row of the transpose tile

__device__ __forceinline__ void unpack_row4(const uint2 u, float (&v)[4]) {
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  v[0] = __low2float(a);
  v[1] = __high2float(a);
  v[2] = __low2float(b);
  v[3] = __high2float(b);
}

// y = H (s o x) for the 128 values of a row, value 4 * lane + e in v[e]
// (Sylvester order: bit 0 and 1 of the index are e, bits 2..6 the lane).
__device__ __forceinline__ void hadamard128(float (&v)[4], const float (&s)[4], int lane) {
#pragma unroll
  for (int e = 0; e < 4; ++e) v[e] *= s[e];
  const float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2;
  v[2] = a0 - a2;
  v[1] = a1 + a3;
  v[3] = a1 - a3;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, v[e], m);
      v[e] = upper ? (o - v[e]) : (v[e] + o);
    }
  }
}

__device__ __forceinline__ void load_signs(const float* __restrict__ signs, int lane,
                                           float (&s)[4]) {
#pragma unroll
  for (int e = 0; e < 4; ++e) s[e] = signs ? signs[4 * lane + e] : 1.0f;
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) v = fmaxf(v, red[w]);
  return v;
}

// partial[bh * nblk + blockIdx.x] = max |y| over rows [128 blockIdx.x, +128)
__global__ void __launch_bounds__(kThreads, 3)
fp8_amax_kernel(const __nv_bfloat16* __restrict__ X, const float* __restrict__ signs,
                float* __restrict__ partial, int n, int nblk) {
  __shared__ float red[kThreads / 32];
  const int bh = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float s[4];
  load_signs(signs, lane, s);
  const int r0 = blockIdx.x * kRows + warp * kRowsPerWarp;
  const __nv_bfloat16* base = X + ((size_t)bh * n) * kD + 4 * lane;
  // all rows' loads in flight before any arithmetic (8 bytes a row per lane)
  uint2 raw[kRowsPerWarp];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i)
    raw[i] = (r0 + i < n) ? __ldg(reinterpret_cast<const uint2*>(base + (size_t)(r0 + i) * kD))
                          : make_uint2(0u, 0u);
  float mx = 0.0f;
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    float v[4];
    unpack_row4(raw[i], v);
    if (signs) hadamard128(v, s, lane);
#pragma unroll
    for (int e = 0; e < 4; ++e) mx = fmaxf(mx, fabsf(v[e]));
  }
  mx = block_max(mx, red);
  if (threadIdx.x == 0) partial[(size_t)bh * nblk + blockIdx.x] = mx;
}

template <bool TRANSPOSE>
__global__ void __launch_bounds__(kThreads, 3)
fp8_quant_kernel(const __nv_bfloat16* __restrict__ X, const float* __restrict__ signs,
                 const float* __restrict__ partial, uint8_t* __restrict__ X8,
                 float* __restrict__ descale, int n, int nblk, float descale_factor) {
  __shared__ float red[kThreads / 32];
  __shared__ __align__(16) uint8_t tile[TRANSPOSE ? kD * kTilePitch : 16];
  const int bh = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  float amax = 0.0f;
  for (int i = threadIdx.x; i < nblk; i += kThreads)
    amax = fmaxf(amax, partial[(size_t)bh * nblk + i]);
  amax = block_max(amax, red);
  // correctly rounded whatever the fast-math flags: the codes are defined by
  // the float32 product x * fl(448 / amax)
  const float inv = amax > 0.0f ? __fdiv_rn(448.0f, amax) : 1.0f;
  if (blockIdx.x == 0 && threadIdx.x == 0)
    descale[bh] = amax > 0.0f ? __fmul_rn(__fdiv_rn(amax, 448.0f), descale_factor) : 1.0f;

  float s[4];
  load_signs(signs, lane, s);
  const int rl0 = warp * kRowsPerWarp;
  const int r0 = blockIdx.x * kRows + rl0;
  const __nv_bfloat16* base = X + ((size_t)bh * n) * kD + 4 * lane;
  // all rows' loads in flight before any arithmetic (8 bytes a row per lane)
  uint2 raw[kRowsPerWarp];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i)
    raw[i] = (r0 + i < n) ? __ldg(reinterpret_cast<const uint2*>(base + (size_t)(r0 + i) * kD))
                          : make_uint2(0u, 0u);
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    float v[4];
    unpack_row4(raw[i], v);
    if (signs) hadamard128(v, s, lane);
    const uint32_t c = sm100::pack_e4m3x4(__fmul_rn(v[0], inv), __fmul_rn(v[1], inv),
                                          __fmul_rn(v[2], inv), __fmul_rn(v[3], inv));
    if (!TRANSPOSE) {
      if (r0 + i < n)
        reinterpret_cast<uint32_t*>(X8 + ((size_t)bh * n + r0 + i) * kD)[lane] = c;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) tile[(4 * lane + e) * kTilePitch + rl0 + i] = (c >> (8 * e)) & 0xFF;
    }
  }
  if (TRANSPOSE) {
    __syncthreads();
    // X8 is [bh][128][n]: row dd gets this block's 128 columns, 16 bytes a thread
    const int n0 = blockIdx.x * kRows;
#pragma unroll
    for (int k = 0; k < kD * kRows / 16 / kThreads; ++k) {
      const int idx = threadIdx.x + k * kThreads;
      const int dd = idx >> 3, c16 = (idx & 7) * 16;
      if (n0 + c16 < n)
        *reinterpret_cast<uint4*>(X8 + ((size_t)bh * kD + dd) * n + n0 + c16) =
            *reinterpret_cast<const uint4*>(&tile[dd * kTilePitch + c16]);
    }
  }
}

}  // namespace

size_t quant_fp8_workspace_bytes(int BH, int n) {
  return (size_t)BH * ((n + kRows - 1) / kRows) * sizeof(float);
}

cudaError_t launch_quant_fp8(const void* X, void* X8, float* descale, int BH, int n, bool transpose,
                             const float* signs, float* partial, cudaStream_t st) {
  const int nblk = (n + kRows - 1) / kRows;
  const dim3 grid(nblk, BH);
  const auto* x = static_cast<const __nv_bfloat16*>(X);
  fp8_amax_kernel<<<grid, kThreads, 0, st>>>(x, signs, partial, n, nblk);
  note_launch();
  // the kernel's Hadamard product is sqrt(128) times the orthonormal one
  const float factor = signs ? 0.088388347648318440f : 1.0f;   // 1 / sqrt(128)
  if (transpose)
    fp8_quant_kernel<true><<<grid, kThreads, 0, st>>>(x, signs, partial,
                                                      static_cast<uint8_t*>(X8), descale, n, nblk,
                                                      factor);
  else
    fp8_quant_kernel<false><<<grid, kThreads, 0, st>>>(x, signs, partial,
                                                       static_cast<uint8_t*>(X8), descale, n,
                                                       nblk, factor);
  note_launch();
  return cudaGetLastError();
}

}  // namespace attn
