// simt_f32.cu -- exact fp32 attention forward/backward on the CUDA cores.
//
// One warp owns one output row.  The forward walks the keys of its query row
// keeping the running maximum m and running sum l of the online softmax
// ("Flash Attention: Revolutionizing Transformer Efficiency", "The
// mathematics behind Flash Attention", formulas 1 and 2, with the
// previous sum l_old carried into the update).  The backward recomputes
// p_ij = exp(s_ij - LSE_i) from the saved logsumexp instead of storing P
// ("Chapter 3.1 -- The cost of attention", section 5) and forms
// dS_ij = p_ij (dO_i . v_j - D_i).  No tensor cores: fp32 FFMA throughout, so
// results stay within fp32 rounding of the exact values.
#include <cuda_runtime.h>
#include <math.h>

#include "kernels.h"

namespace attn {
namespace {

constexpr int kRowsPerBlock = 8;   // one warp per row
constexpr int kMaxPerLane = 8;     // d <= 256

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kRowsPerBlock * 32)
fwd_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
               const float* __restrict__ V, float* __restrict__ O, float* __restrict__ LSE,
               HeadMap hm, const uint8_t* __restrict__ bmask, int n, int d, float scale,
               int causal) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  const size_t bh = blockIdx.y;
  const size_t bkv = hm.kv_of((int)bh);
  if (row >= n) return;
  const float* q = Q + (bh * n + row) * d;
  const float* k = K + bkv * n * d;
  const float* v = V + bkv * n * d;
  // block-sparse pattern (null: dense): the 128-block row of this query
  const uint8_t* brow = bmask ? bmask + (size_t)(row / 128) * ((n + 127) / 128) : nullptr;
  float qr[kMaxPerLane], acc[kMaxPerLane];
#pragma unroll
  for (int t = 0; t < kMaxPerLane; ++t) {
    const int c = lane + 32 * t;
    qr[t] = c < d ? q[c] : 0.f;
    acc[t] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int jend = causal ? row + 1 : n;
  for (int j = 0; j < jend; ++j) {
    if (brow && !brow[j / 128]) continue;   // key outside the kept blocks
    const float* kj = k + (size_t)j * d;
    float part = 0.f;
#pragma unroll
    for (int t = 0; t < kMaxPerLane; ++t) {
      const int c = lane + 32 * t;
      if (c < d) part = fmaf(qr[t], kj[c], part);
    }
    const float s = scale * warp_sum(part);
    const float m_new = fmaxf(m, s);
    const float alpha = expf(m - m_new);   // 0 on the first key (m = -inf)
    const float p = expf(s - m_new);
    l = l * alpha + p;
    const float* vj = v + (size_t)j * d;
#pragma unroll
    for (int t = 0; t < kMaxPerLane; ++t) {
      const int c = lane + 32 * t;
      if (c < d) acc[t] = fmaf(p, vj[c], acc[t] * alpha);
    }
    m = m_new;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;   // no kept key: O = 0, LSE = -inf
  float* o = O + (bh * n + row) * d;
#pragma unroll
  for (int t = 0; t < kMaxPerLane; ++t) {
    const int c = lane + 32 * t;
    if (c < d) o[c] = acc[t] * inv;
  }
  if (lane == 0) LSE[bh * n + row] = l > 0.f ? m + logf(l) : -INFINITY;
}

// D_i = dO_i . O_i for fp32 tensors (one warp per row).
__global__ void __launch_bounds__(kRowsPerBlock * 32)
delta_f32_kernel(const float* __restrict__ O, const float* __restrict__ dO,
                 float* __restrict__ Dv, int rows, int d) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float* o = O + (size_t)row * d;
  const float* g = dO + (size_t)row * d;
  float part = 0.f;
  for (int c = lane; c < d; c += 32) part = fmaf(o[c], g[c], part);
  part = warp_sum(part);
  if (lane == 0) Dv[row] = part;
}

// dQ_i = scale * sum_j p_ij (dO_i . v_j - D_i) k_j   (one warp per query row)
__global__ void __launch_bounds__(kRowsPerBlock * 32)
bwd_dq_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                  const float* __restrict__ V, const float* __restrict__ dO,
                  const float* __restrict__ LSE, const float* __restrict__ Dv,
                  float* __restrict__ dQ, HeadMap hm, const uint8_t* __restrict__ bmask, int n,
                  int d, float scale, int causal) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  const size_t bh = blockIdx.y;
  const size_t bkv = hm.kv_of((int)bh);
  if (row >= n) return;
  const float* q = Q + (bh * n + row) * d;
  const float* g = dO + (bh * n + row) * d;
  const float* k = K + bkv * n * d;
  const float* v = V + bkv * n * d;
  const float lse = LSE[bh * n + row];
  const float Di = Dv[bh * n + row];
  const uint8_t* brow = bmask ? bmask + (size_t)(row / 128) * ((n + 127) / 128) : nullptr;
  float qr[kMaxPerLane], gr[kMaxPerLane], acc[kMaxPerLane];
#pragma unroll
  for (int t = 0; t < kMaxPerLane; ++t) {
    const int c = lane + 32 * t;
    qr[t] = c < d ? q[c] : 0.f;
    gr[t] = c < d ? g[c] : 0.f;
    acc[t] = 0.f;
  }
  const int jend = causal ? row + 1 : n;
  for (int j = 0; j < jend; ++j) {
    if (brow && !brow[j / 128]) continue;   // key outside the kept blocks
    const float* kj = k + (size_t)j * d;
    const float* vj = v + (size_t)j * d;
    float ps = 0.f, pd = 0.f;
#pragma unroll
    for (int t = 0; t < kMaxPerLane; ++t) {
      const int c = lane + 32 * t;
      if (c < d) {
        ps = fmaf(qr[t], kj[c], ps);
        pd = fmaf(gr[t], vj[c], pd);
      }
    }
    const float s = scale * warp_sum(ps);
    const float dp = warp_sum(pd);
    const float p = expf(s - lse);
    const float ds = p * (dp - Di);
#pragma unroll
    for (int t = 0; t < kMaxPerLane; ++t) {
      const int c = lane + 32 * t;
      if (c < d) acc[t] = fmaf(ds, kj[c], acc[t]);
    }
  }
  float* out = dQ + (bh * n + row) * d;
#pragma unroll
  for (int t = 0; t < kMaxPerLane; ++t) {
    const int c = lane + 32 * t;
    if (c < d) out[c] = scale * acc[t];
  }
}

// dV_j = sum_i p_ij dO_i ; dK_j = scale * sum_i dS_ij q_i  (one warp per key row;
// the sums run over every query head that reads this key/value head)
__global__ void __launch_bounds__(kRowsPerBlock * 32)
bwd_dkdv_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                    const float* __restrict__ V, const float* __restrict__ dO,
                    const float* __restrict__ LSE, const float* __restrict__ Dv,
                    float* __restrict__ dK, float* __restrict__ dV, HeadMap hm,
                    const uint8_t* __restrict__ bmask, int n, int d, float scale, int causal) {
  const int lane = threadIdx.x & 31;
  const int col = blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  const size_t bkv = blockIdx.y;
  if (col >= n) return;
  const float* kj = K + (bkv * n + col) * d;
  const float* vj = V + (bkv * n + col) * d;
  float kr[kMaxPerLane], vr[kMaxPerLane], ak[kMaxPerLane], av[kMaxPerLane];
#pragma unroll
  for (int t = 0; t < kMaxPerLane; ++t) {
    const int c = lane + 32 * t;
    kr[t] = c < d ? kj[c] : 0.f;
    vr[t] = c < d ? vj[c] : 0.f;
    ak[t] = 0.f;
    av[t] = 0.f;
  }
  for (int m = 0; m < hm.group; ++m) {
    const size_t bh = hm.q_of((int)bkv, m);
    const float* q = Q + bh * n * d;
    const float* g = dO + bh * n * d;
    for (int i = causal ? col : 0; i < n; ++i) {
      if (bmask && !bmask[(size_t)(i / 128) * ((n + 127) / 128) + col / 128]) continue;
      const float* qi = q + (size_t)i * d;
      const float* gi = g + (size_t)i * d;
      float ps = 0.f, pd = 0.f;
#pragma unroll
      for (int t = 0; t < kMaxPerLane; ++t) {
        const int c = lane + 32 * t;
        if (c < d) {
          ps = fmaf(qi[c], kr[t], ps);
          pd = fmaf(gi[c], vr[t], pd);
        }
      }
      const float s = scale * warp_sum(ps);
      const float dp = warp_sum(pd);
      const float p = expf(s - LSE[bh * n + i]);
      const float ds = p * (dp - Dv[bh * n + i]);
#pragma unroll
      for (int t = 0; t < kMaxPerLane; ++t) {
        const int c = lane + 32 * t;
        if (c < d) {
          av[t] = fmaf(p, gi[c], av[t]);
          ak[t] = fmaf(ds, qi[c], ak[t]);
        }
      }
    }
  }
  float* ok = dK + (bkv * n + col) * d;
  float* ov = dV + (bkv * n + col) * d;
#pragma unroll
  for (int t = 0; t < kMaxPerLane; ++t) {
    const int c = lane + 32 * t;
    if (c < d) {
      ok[c] = scale * ak[t];
      ov[c] = av[t];
    }
  }
}

}  // namespace

cudaError_t launch_fwd_f32(const float* Q, const float* K, const float* V, float* O, float* LSE,
                           int BH, const HeadMap& hm, const uint8_t* bmask, int n, int d,
                           float scale, int causal, cudaStream_t st) {
  dim3 grid(ceil_div(n, kRowsPerBlock), BH);
  fwd_f32_kernel<<<grid, kRowsPerBlock * 32, 0, st>>>(Q, K, V, O, LSE, hm, bmask, n, d, scale,
                                                      causal);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_delta_f32(const float* O, const float* dO, float* Dv, int BH, int n, int d,
                             cudaStream_t st) {
  const int rows = BH * n;
  delta_f32_kernel<<<ceil_div(rows, kRowsPerBlock), kRowsPerBlock * 32, 0, st>>>(O, dO, Dv, rows,
                                                                                 d);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv_f32(const float* Q, const float* K, const float* V, const float* dO,
                                const float* LSE, const float* Dv, float* dK, float* dV, int BH,
                                const HeadMap& hm, const uint8_t* bmask, int n, int d, float scale,
                                int causal, cudaStream_t st) {
  dim3 grid(ceil_div(n, kRowsPerBlock), BH / hm.group);
  bwd_dkdv_f32_kernel<<<grid, kRowsPerBlock * 32, 0, st>>>(Q, K, V, dO, LSE, Dv, dK, dV, hm, bmask,
                                                           n, d, scale, causal);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_f32(const float* Q, const float* K, const float* V, const float* dO,
                              const float* LSE, const float* Dv, float* dQ, int BH,
                              const HeadMap& hm, const uint8_t* bmask, int n, int d, float scale,
                              int causal, cudaStream_t st) {
  dim3 grid(ceil_div(n, kRowsPerBlock), BH);
  bwd_dq_f32_kernel<<<grid, kRowsPerBlock * 32, 0, st>>>(Q, K, V, dO, LSE, Dv, dQ, hm, bmask, n, d,
                                                         scale, causal);
  note_launch();
  return cudaGetLastError();
}

}  // namespace attn
