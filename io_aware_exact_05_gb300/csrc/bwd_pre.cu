// bwd_pre.cu -- bandwidth-bound helpers of the bf16 backward pass.
//
// delta_kernel: D_i = dO_i . O_i in fp32 (the row term of
//   dS = P o (dP - D), since sum_j P_ij dP_ij = dO_i . O_i), the log2-scaled
//   logsumexp LSE2_i = LSE_i * log2(e) that the tensor-core kernels use to
//   recompute P_ij = 2^(s_ij * scale * log2(e) - LSE2_i), and (optionally) a
//   zeroed fp32 dQ accumulator.  Row statistics are written with a row stride
//   padded to a multiple of 128 so every 128-row tile starts 512-byte aligned;
//   padded rows get LSE2 = +inf (so P = 0) and D = 0.
// dq_convert_kernel: fp32 dQ accumulator -> bf16 dQ.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"

namespace attn {
namespace {

__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) {
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&v);
  return __bfloat1622float2(b);
}

template <int D>
__global__ void __launch_bounds__(256)
delta_kernel(const __nv_bfloat16* __restrict__ O, const __nv_bfloat16* __restrict__ dO,
             const float* __restrict__ LSE, float* __restrict__ Dv, float* __restrict__ LSE2,
             float* __restrict__ dQacc, int n, int n_pad, int total_rows_pad) {
  constexpr int TPR = D / 8;            // threads per row, 8 bf16 (16 B) each
  constexpr int RPB = 256 / TPR;        // rows per block
  const int sub = threadIdx.x % TPR;
  const int prow = blockIdx.x * RPB + threadIdx.x / TPR;   // padded row index
  if (prow >= total_rows_pad) return;
  const int bh = prow / n_pad;
  const int i = prow - bh * n_pad;
  float acc = 0.f;
  const bool valid = i < n;
  const size_t row = (size_t)bh * n + i;
  if (valid) {
    const uint4 a = *reinterpret_cast<const uint4*>(O + row * D + sub * 8);
    const uint4 b = *reinterpret_cast<const uint4*>(dO + row * D + sub * 8);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 x = bf2_to_f2(av[t]), y = bf2_to_f2(bv[t]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
    if (dQacc) {
      float4* z = reinterpret_cast<float4*>(dQacc + row * D + sub * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int o = TPR / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (sub == 0) {
    Dv[prow] = valid ? acc : 0.f;
    // +inf (P = 0) on padded rows and on rows that kept no score (LSE = -inf)
    const float lse = valid ? LSE[row] : -INFINITY;
    LSE2[prow] = lse == -INFINITY ? INFINITY : lse * 1.4426950408889634f;
  }
}

__global__ void __launch_bounds__(256)
dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ out, size_t n8) {
  const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[2 * t];
  const float4 b = reinterpret_cast<const float4*>(acc)[2 * t + 1];
  __nv_bfloat162 r[4];
  r[0] = __floats2bfloat162_rn(a.x, a.y);
  r[1] = __floats2bfloat162_rn(a.z, a.w);
  r[2] = __floats2bfloat162_rn(b.x, b.y);
  r[3] = __floats2bfloat162_rn(b.z, b.w);
  reinterpret_cast<uint4*>(out)[t] = *reinterpret_cast<uint4*>(r);
}

}  // namespace

cudaError_t launch_delta_bf16(const void* O, const void* dO, const float* LSE, float* Dv,
                              float* LSE2, float* dQacc, int BH, int n, int n_pad, int d,
                              cudaStream_t st) {
  const int rows = BH * n_pad;
  const auto* o = static_cast<const __nv_bfloat16*>(O);
  const auto* g = static_cast<const __nv_bfloat16*>(dO);
  switch (d) {
    case 64:
      delta_kernel<64><<<ceil_div(rows, 32), 256, 0, st>>>(o, g, LSE, Dv, LSE2, dQacc, n, n_pad,
                                                          rows);
      note_launch();
      break;
    case 128:
      delta_kernel<128><<<ceil_div(rows, 16), 256, 0, st>>>(o, g, LSE, Dv, LSE2, dQacc, n, n_pad,
                                                           rows);
      note_launch();
      break;
    case 256:
      delta_kernel<256><<<ceil_div(rows, 8), 256, 0, st>>>(o, g, LSE, Dv, LSE2, dQacc, n, n_pad,
                                                          rows);
      note_launch();
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const float* acc, void* dQ, size_t elems, cudaStream_t st) {
  const size_t n8 = elems / 8;
  if (n8 == 0) return cudaSuccess;
  dq_convert_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, st>>>(
      acc, static_cast<__nv_bfloat16*>(dQ), n8);
  note_launch();
  return cudaGetLastError();
}

}  // namespace attn
