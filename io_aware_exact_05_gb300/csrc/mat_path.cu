// mat_path.cu -- row kernels of the materialise-P comparison path.
//
// This path keeps every n x n matrix in HBM, the way standard attention does
// ("Flash Attention: Revolutionizing Transformer Efficiency", "Standard
// attention": the score matrix is written to HBM and read back for the
// softmax) and the way the small-cache backward algorithm of "On the
// fine-grained I/O complexity of attention backward passes" (Methodology,
// step 3) reads and writes the n x n attention matrices explicitly.
//
// mat_softmax_kernel : P = softmax(S) row by row (S already scaled, fp32),
//                      causal mask applied before the maximum, P in bf16,
//                      LSE_i = m_i + ln l_i.
// mat_dsoftmax_kernel: dS = P o (dP - D) elementwise (bf16 out).
#include <cuda_bf16.h>
#include <math.h>

#include "kernels.h"

namespace attn {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
  for (int w = 1; w < kThreads / 32; ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
  return v;
}

// One CTA per row; n % 4 == 0.
__global__ void __launch_bounds__(kThreads)
mat_softmax_kernel(const float* __restrict__ S, __nv_bfloat16* __restrict__ P,
                   float* __restrict__ LSE, int n, int causal) {
  __shared__ float red[kThreads / 32];
  const int i = blockIdx.x;
  const size_t row = (size_t)blockIdx.y * n + i;
  const float* s = S + row * n;
  __nv_bfloat16* p = P + row * n;
  const int jend = causal ? i + 1 : n;   // columns j < jend are kept
  float m = -INFINITY;
  for (int j = threadIdx.x * 4; j < jend; j += kThreads * 4) {
    const float4 x = *reinterpret_cast<const float4*>(s + j);
    m = fmaxf(m, x.x);
    if (j + 1 < jend) m = fmaxf(m, x.y);
    if (j + 2 < jend) m = fmaxf(m, x.z);
    if (j + 3 < jend) m = fmaxf(m, x.w);
  }
  m = block_reduce(m, true, red);
  float l = 0.f;
  for (int j = threadIdx.x * 4; j < jend; j += kThreads * 4) {
    const float4 x = *reinterpret_cast<const float4*>(s + j);
    l += expf(x.x - m);
    if (j + 1 < jend) l += expf(x.y - m);
    if (j + 2 < jend) l += expf(x.z - m);
    if (j + 3 < jend) l += expf(x.w - m);
  }
  l = block_reduce(l, false, red);
  const float inv = 1.f / l;
  for (int j = threadIdx.x * 4; j < n; j += kThreads * 4) {
    const float4 x = *reinterpret_cast<const float4*>(s + j);
    const float v0 = j < jend ? expf(x.x - m) * inv : 0.f;
    const float v1 = j + 1 < jend ? expf(x.y - m) * inv : 0.f;
    const float v2 = j + 2 < jend ? expf(x.z - m) * inv : 0.f;
    const float v3 = j + 3 < jend ? expf(x.w - m) * inv : 0.f;
    __nv_bfloat162 a = __floats2bfloat162_rn(v0, v1), b = __floats2bfloat162_rn(v2, v3);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p + j) = u;
  }
  if (threadIdx.x == 0) LSE[row] = m + logf(l);
}

// dS = P o (dP - D_i); 8 elements per thread; n % 8 == 0.  dS may alias P
// (each thread reads its 8 elements before writing them).
__global__ void __launch_bounds__(kThreads)
mat_dsoftmax_kernel(const __nv_bfloat16* P, const float* __restrict__ dP,
                    const float* __restrict__ Dv, __nv_bfloat16* dS, int n,
                    size_t total8) {
  const size_t t = (size_t)blockIdx.x * kThreads + threadIdx.x;
  if (t >= total8) return;
  const size_t e = t * 8;
  const size_t row = e / n;
  const float Di = Dv[row];
  const uint4 pv = *reinterpret_cast<const uint4*>(P + e);
  const float4 a = *reinterpret_cast<const float4*>(dP + e);
  const float4 b = *reinterpret_cast<const float4*>(dP + e + 4);
  const float g[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  const uint32_t pw[4] = {pv.x, pv.y, pv.z, pv.w};
  uint32_t out[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t w = pw[k];
    const float2 pf = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&w));
    __nv_bfloat162 r = __floats2bfloat162_rn(pf.x * (g[2 * k] - Di), pf.y * (g[2 * k + 1] - Di));
    out[k] = *reinterpret_cast<uint32_t*>(&r);
  }
  *reinterpret_cast<uint4*>(dS + e) = make_uint4(out[0], out[1], out[2], out[3]);
}

}  // namespace

cudaError_t launch_mat_softmax(const float* S, void* P, float* LSE, int BH, int n, float scale,
                               int causal, cudaStream_t st) {
  (void)scale;   // S arrives already scaled by the GEMM
  dim3 grid(n, BH);
  mat_softmax_kernel<<<grid, kThreads, 0, st>>>(S, static_cast<__nv_bfloat16*>(P), LSE, n,
                                                causal);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_mat_dsoftmax(const void* P, const float* dP, const float* Dv, void* dS, int BH,
                                int n, cudaStream_t st) {
  const size_t total8 = (size_t)BH * n * n / 8;
  mat_dsoftmax_kernel<<<(unsigned)((total8 + kThreads - 1) / kThreads), kThreads, 0, st>>>(
      static_cast<const __nv_bfloat16*>(P), dP, Dv, static_cast<__nv_bfloat16*>(dS), n, total8);
  note_launch();
  return cudaGetLastError();
}

}  // namespace attn
