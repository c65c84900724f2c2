// bwd_kv128.cu -- key-tile attention backward for head dim 128, software-
// pipelined two query tiles deep.
//
// One CTA owns 128 keys of one head (the TMEM lanes) and walks the query
// tiles (64 queries each) that can see them.  For every query tile u, with
// c = scale * log2(e) and LSE2 = LSE * log2(e):
//   S^T  = K Q_u^T                (SS-MMA, M = 128 keys, N = 64 queries)
//   P^T  = 2^(S^T c - LSE2)       (registers; bf16 copy back into TMEM)
//   dV  += P^T dO_u               (TS-MMA: A = P^T read from TMEM)
//   dP^T = V dO_u^T               (SS-MMA)
//   dS^T = P^T o (dP^T - D)       (registers; bf16 copy into shared memory)
//   dK  += dS^T Q_u               (SS-MMA: A = dS^T, K-major over queries)
//   dQ_u^T = K^T dS^T             (SS-MMA: M = d on the lanes, N = 64 queries)
// These are the chain-rule steps of the backward pass that recomputes the
// attention matrix instead of storing it ("Chapter 3.1 -- The cost of
// attention", section 5; "Flash Attention: Revolutionizing Transformer
// Efficiency", key idea 2).
//
// Tensor memory (512 columns): dV [0,128), dK [128,256), S^T in two 64-column
// slots [256,384), dP^T [384,448), dQ^T [448,512).  Shared memory: K and V
// tiles, a 3-deep ring of (Q tile, LSE2, D), a 2-deep ring of dO tiles, two
// dS^T buffers and a 64 x 128 fp32 dQ staging tile.
//
// The MMA issuer runs, per tile u,  dV(u) | dP(u+1) | dK(u), dQ^T(u) | S(u+2):
// S of the tile after next is already in TMEM while the compute warps finish
// tile u, so they go from dS(u) straight to the exponentials of u+1.  The dQ
// warpgroup reads each dQ^T tile out of TMEM, stages it as fp32 [64][128] in
// shared memory and adds it into the fp32 dQ accumulator with one TMA bulk
// reduce-add.  Every wait is bounded (mbar_wait).
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm100.cuh"

namespace attn {
namespace {

using namespace sm100;

__device__ __forceinline__ uint8_t* align_1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void store_row32_bf16(__nv_bfloat16* dst, const uint32_t (&r)[32],
                                                 float mul) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    reinterpret_cast<uint4*>(dst)[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
}

template <bool DQ>
struct Kv128 {
  static constexpr int D = 128, BNK = 128, BM = 64, NKB = 2;
  static constexpr int QST = 3, GST = 2;
  static constexpr uint32_t KV_BYTES = BNK * D * 2;           // 32 KB
  static constexpr uint32_t QT_BYTES = BM * D * 2;            // 16 KB
  static constexpr uint32_t QSLOT = QT_BYTES + 1024;          // Q + LSE2 (+0) + D (+512)
  static constexpr uint32_t DS_BYTES = BM * BNK * 2;          // 16 KB
  static constexpr uint32_t K_OFF = 0, V_OFF = KV_BYTES;
  static constexpr uint32_t Q_OFF = 2 * KV_BYTES;
  static constexpr uint32_t G_OFF = Q_OFF + QST * QSLOT;
  static constexpr uint32_t DS_OFF = G_OFF + GST * QT_BYTES;
  static constexpr uint32_t QS_OFF = DS_OFF + 2 * DS_BYTES;
  static constexpr uint32_t QS_BYTES = DQ ? BM * D * 4 : 0;
  static constexpr uint32_t BAR_OFF = QS_OFF + QS_BYTES;
  static constexpr uint32_t SMEM = BAR_OFF + 256 + 1024;
  static constexpr int DV_COL = 0, DK_COL = 128, S_COL = 256, DP_COL = 384, DQ_COL = 448;
  static constexpr int NTHREADS = DQ ? 512 : 384;
  static_assert(SMEM <= 232448, "shared memory budget");
};

// barrier indices
enum : int { P_KV = 0, P_QF = 1, P_QE = 4, P_GF = 7, P_GE = 9, P_SF = 11, P_DPF = 13, P_PR = 14,
             P_DPE = 15, P_DSR = 16, P_DSE = 17, P_DQF = 19, P_DQE = 20, P_ACC = 21, P_DRAIN = 22 };

template <bool DQ>
__global__ void __launch_bounds__(Kv128<DQ>::NTHREADS, 1)
bwd_kv128_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                 const __grid_constant__ CUtensorMap tmdQ, const float* __restrict__ LSE2,
                 const float* __restrict__ Dv, __nv_bfloat16* __restrict__ dK,
                 __nv_bfloat16* __restrict__ dV, int n, int n_pad, float scale, float scale_log2,
                 int causal, KernelCtl ctl) {
  using C = Kv128<DQ>;
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1k(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::BAR_OFF + 192);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 200);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kt = blockIdx.x, bh = blockIdx.y;
  const int k0 = kt * C::BNK;
  const int nq = (n + C::BM - 1) / C::BM;
  const int i_start = causal ? (k0 / C::BM) : 0;
  const int cnt = nq - i_start;   // query tiles that see these keys (>= 1)

  if (threadIdx.x == 0) {
    mbar_init(bar(P_KV), 1);
    for (int s = 0; s < C::QST; ++s) { mbar_init(bar(P_QF + s), 1); mbar_init(bar(P_QE + s), 1); }
    for (int s = 0; s < C::GST; ++s) { mbar_init(bar(P_GF + s), 1); mbar_init(bar(P_GE + s), 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(bar(P_SF + s), 1); mbar_init(bar(P_DSE + s), 1); }
    mbar_init(bar(P_DPF), 1);
    mbar_init(bar(P_PR), 256);
    mbar_init(bar(P_DPE), 256);
    mbar_init(bar(P_DSR), 256);
    mbar_init(bar(P_DQF), 1);
    mbar_init(bar(P_DQE), 128);
    mbar_init(bar(P_ACC), 1);
    mbar_init(bar(P_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
  }
  if (warp == 2) tmem_alloc<512>(smem_u32(tmem_slot));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------ producer
      mbar_expect_tx(bar(P_KV), 2 * C::KV_BYTES);
#pragma unroll
      for (int kb = 0; kb < C::NKB; ++kb) {
        tma_load_3d(sb + C::K_OFF + kb * (C::BNK * 128), &tmK, kb * 64, k0, bh, bar(P_KV));
        tma_load_3d(sb + C::V_OFF + kb * (C::BNK * 128), &tmV, kb * 64, k0, bh, bar(P_KV));
      }
      int last_q[C::QST], last_g[C::GST];
      for (int s = 0; s < C::QST; ++s) last_q[s] = -1;
      for (int s = 0; s < C::GST; ++s) last_g[s] = -1;
      for (int u = 0; u < cnt; ++u) {
        const int q0 = (i_start + u) * C::BM;
        const int qs = u % C::QST, gs = u % C::GST;
        if (!mbar_wait(bar(P_QE + qs), ((u / C::QST) & 1) ^ 1, abort_flag, ctl, SITE_BWD_Q_EMPTY))
          break;
        const uint32_t qa = sb + C::Q_OFF + qs * C::QSLOT;
        mbar_expect_tx(bar(P_QF + qs), C::QT_BYTES + 2 * C::BM * 4);
#pragma unroll
        for (int kb = 0; kb < C::NKB; ++kb)
          tma_load_3d(qa + kb * (C::BM * 128), &tmQ, kb * 64, q0, bh, bar(P_QF + qs));
        bulk_load(qa + C::QT_BYTES, LSE2 + (size_t)bh * n_pad + q0, C::BM * 4, bar(P_QF + qs));
        bulk_load(qa + C::QT_BYTES + 512, Dv + (size_t)bh * n_pad + q0, C::BM * 4, bar(P_QF + qs));
        last_q[qs] = u;
        if (!mbar_wait(bar(P_GE + gs), ((u / C::GST) & 1) ^ 1, abort_flag, ctl, SITE_BWD_Q_EMPTY))
          break;
        const uint32_t ga = sb + C::G_OFF + gs * C::QT_BYTES;
        mbar_expect_tx(bar(P_GF + gs), C::QT_BYTES);
#pragma unroll
        for (int kb = 0; kb < C::NKB; ++kb)
          tma_load_3d(ga + kb * (C::BM * 128), &tmdO, kb * 64, q0, bh, bar(P_GF + gs));
        last_g[gs] = u;
      }
      if (*abort_flag) {   // let issued copies land before the CTA may exit
        volatile int no_abort = 0;
        mbar_wait(bar(P_KV), 0, &no_abort, ctl, SITE_BWD_KV);
        for (int s = 0; s < C::QST; ++s)
          if (last_q[s] >= 0)
            mbar_wait(bar(P_QF + s), (last_q[s] / C::QST) & 1, &no_abort, ctl, SITE_BWD_Q_FULL);
        for (int s = 0; s < C::GST; ++s)
          if (last_g[s] >= 0)
            mbar_wait(bar(P_GF + s), (last_g[s] / C::GST) & 1, &no_abort, ctl, SITE_BWD_Q_FULL);
      }
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t id_s = idesc_bf16(128, C::BM, false, false);   // K/V and Q/dO K-major
      constexpr uint32_t id_acc = idesc_bf16(128, D, false, true);      // A K-major, B MN-major
      constexpr uint32_t id_dq = idesc_bf16(128, C::BM, true, true);    // both MN-major
      const uint32_t ka = sb + C::K_OFF, va = sb + C::V_OFF;
      auto qaddr = [&](int u) { return sb + C::Q_OFF + (u % C::QST) * C::QSLOT; };
      auto gaddr = [&](int u) { return sb + C::G_OFF + (u % C::GST) * C::QT_BYTES; };
      // S^T(u) = K Q(u)^T into slot u & 1
      auto issue_s = [&](int u) -> bool {
        if (!mbar_wait(bar(P_QF + u % C::QST), (u / C::QST) & 1, abort_flag, ctl, SITE_BWD_Q_FULL))
          return false;
        tc_fence_after();
        const uint32_t qa = qaddr(u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::S_COL + (u & 1) * C::BM,
                 sdesc_sw128(ka + (kk >> 2) * (C::BNK * 128) + (kk & 3) * 32, 16, 1024),
                 sdesc_sw128(qa + (kk >> 2) * (C::BM * 128) + (kk & 3) * 32, 16, 1024), id_s, kk > 0);
        tc_commit(bar(P_SF + (u & 1)));
        return true;
      };
      // dP^T(u) = V dO(u)^T
      auto issue_dp = [&](int u) -> bool {
        if (!mbar_wait(bar(P_GF + u % C::GST), (u / C::GST) & 1, abort_flag, ctl, SITE_BWD_Q_FULL))
          return false;
        tc_fence_after();
        const uint32_t ga = gaddr(u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::DP_COL,
                 sdesc_sw128(va + (kk >> 2) * (C::BNK * 128) + (kk & 3) * 32, 16, 1024),
                 sdesc_sw128(ga + (kk >> 2) * (C::BM * 128) + (kk & 3) * 32, 16, 1024), id_s, kk > 0);
        tc_commit(bar(P_DPF));
        return true;
      };
      bool ok = mbar_wait(bar(P_KV), 0, abort_flag, ctl, SITE_BWD_KV);
      if (ok) ok = issue_s(0);
      if (ok) ok = issue_dp(0);
      if (ok && cnt > 1) ok = issue_s(1);
      for (int u = 0; ok && u < cnt; ++u) {
        const int b = u & 1;
        const uint32_t qa = qaddr(u), ga = gaddr(u);
        const uint32_t dsa = sb + C::DS_OFF + b * C::DS_BYTES;
        // dV += P^T dO(u): P^T from TMEM slot b, where compute half h wrote
        // queries [32h, 32h+32) packed into columns [32h, 32h+16)
        if (!(ok = mbar_wait(bar(P_PR), u & 1, abort_flag, ctl, SITE_BWD_P_READY))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk) {
          const uint32_t acol = (kk >> 1) * 32 + (kk & 1) * 8;
          mma_ts(tmem + C::DV_COL, tmem + C::S_COL + b * C::BM + acol,
                 sdesc_sw128(ga + kk * 2048, C::BM * 128, 1024), id_acc, (u > 0 || kk > 0));
        }
        // dP^T(u+1) once the compute warps have read dP^T(u)
        if (u + 1 < cnt) {
          if (!(ok = mbar_wait(bar(P_DPE), u & 1, abort_flag, ctl, SITE_BWD_DS_FREE))) break;
          if (!(ok = issue_dp(u + 1))) break;
        }
        if (!(ok = mbar_wait(bar(P_DSR), u & 1, abort_flag, ctl, SITE_BWD_DS_READY))) break;
        tc_fence_after();
        // dK += dS^T Q(u)   (dS^T in smem, K-major over the 64 queries)
#pragma unroll
        for (int kk = 0; kk < C::BM / 16; ++kk)
          mma_ss(tmem + C::DK_COL, sdesc_sw128(dsa + kk * 32, 16, 1024),
                 sdesc_sw128(qa + kk * 2048, C::BM * 128, 1024), id_acc, (u > 0 || kk > 0));
        if (DQ) {
          if (u >= 1) {
            if (!(ok = mbar_wait(bar(P_DQE), (u - 1) & 1, abort_flag, ctl, SITE_BWD_DQ_FREE))) break;
            tc_fence_after();
          }
          // dQ^T(u) = K^T dS^T   (M = d, N = 64 queries, contraction over the 128 keys)
#pragma unroll
          for (int kk = 0; kk < C::BNK / 16; ++kk)
            mma_ss(tmem + C::DQ_COL, sdesc_sw128(ka + kk * 2048, C::BNK * 128, 1024),
                   sdesc_sw128(dsa + kk * 2048, C::BNK * 128, 1024), id_dq, kk > 0);
          tc_commit(bar(P_DQF));
        }
        tc_commit(bar(P_QE + u % C::QST));
        tc_commit(bar(P_GE + u % C::GST));
        tc_commit(bar(P_DSE + b));
        if (u + 2 < cnt) {
          if (!(ok = issue_s(u + 2))) break;
        }
      }
      tc_commit(bar(P_ACC));
      if (*abort_flag) {
        tc_commit(bar(P_DRAIN));
        volatile int no_abort = 0;
        mbar_wait(bar(P_DRAIN), 0, &no_abort, ctl, SITE_BWD_ACC_DONE);
      }
    }
    __syncwarp();
  } else if (warp < 12) {
    // ---------------------------------------------------------------- compute
    const int q = warp & 3, h = (warp - 4) >> 2;
    const int r = q * 32 + lane;          // key row (TMEM lane)
    const int key = k0 + r;
    constexpr int NC = 32;                // queries of this thread: [32h, 32h+32)
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint32_t dp_addr = tmem + lane_off + C::DP_COL + h * NC;
    bool ok = true;
    for (int u = 0; u < cnt; ++u) {
      const int b = u & 1;
      const int q0 = (i_start + u) * C::BM;
      const uint8_t* qp = smem + C::Q_OFF + (u % C::QST) * C::QSLOT;
      const float* lse2 = reinterpret_cast<const float*>(qp + C::QT_BYTES) + h * NC;
      const float* dd = reinterpret_cast<const float*>(qp + C::QT_BYTES + 512) + h * NC;
      const uint32_t s_addr = tmem + lane_off + C::S_COL + b * C::BM + h * NC;
      ok = mbar_wait(bar(P_QF + u % C::QST), (u / C::QST) & 1, abort_flag, ctl, SITE_BWD_Q_FULL);
      ok = ok && mbar_wait(bar(P_SF + b), (u >> 1) & 1, abort_flag, ctl, SITE_BWD_S_FULL);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const bool masked = causal && (k0 + C::BNK - 1 > q0);
      const int qbase = q0 + h * NC;
      float p[NC];
      {
        uint32_t rr[32];
        tmem_ld32(s_addr, rr);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float v = ex2(fmaf(__uint_as_float(rr[i]), scale_log2, -lse2[i]));
          if (masked && key > qbase + i) v = 0.f;
          p[i] = v;
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(p[2 * i], p[2 * i + 1]);
        tmem_st16(s_addr, pk);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(bar(P_PR));
      ok = mbar_wait(bar(P_DPF), u & 1, abort_flag, ctl, SITE_BWD_DP_FULL);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t ds[16];
      {
        uint32_t rr[32];
        tmem_ld32(dp_addr, rr);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bar(P_DPE));        // the dP^T columns may be overwritten
#pragma unroll
        for (int i = 0; i < 16; ++i)
          ds[i] = pack_bf16x2(p[2 * i] * (__uint_as_float(rr[2 * i]) - dd[2 * i]),
                              p[2 * i + 1] * (__uint_as_float(rr[2 * i + 1]) - dd[2 * i + 1]));
      }
      if (u >= 2) {
        ok = mbar_wait(bar(P_DSE + b), ((u >> 1) - 1) & 1, abort_flag, ctl, SITE_BWD_DS_FREE);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      // dS^T row of key r: [128 keys][64 queries] bf16, 128-byte swizzle;
      // this half's 32 queries are chunks 4h .. 4h+3
      uint8_t* dsb = smem + C::DS_OFF + b * C::DS_BYTES;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(dsb + sw128_offset(r, h * 4 + c)) =
            make_uint4(ds[4 * c], ds[4 * c + 1], ds[4 * c + 2], ds[4 * c + 3]);
      fence_proxy_async_smem();
      mbar_arrive(bar(P_DSR));
    }
    // ---- epilogue: half 0 writes dV, half 1 writes dK (scaled)
    if (ok) {
      ok = mbar_wait(bar(P_ACC), 0, abort_flag, ctl, SITE_BWD_ACC_DONE);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const uint32_t src = tmem + lane_off + (h == 0 ? C::DV_COL : C::DK_COL);
      __nv_bfloat16* dst = (h == 0 ? dV : dK) + ((size_t)bh * n + key) * D;
      const float mul = h == 0 ? 1.f : scale;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(src + c0, rr);
        tmem_ld_wait();
        if (key < n) store_row32_bf16(dst + c0, rr, mul);
      }
    }
  } else if (DQ) {
    // ---------------------------------------------------------------- dQ warpgroup
    const int q = warp & 3;
    const int r = q * 32 + lane;          // d column (TMEM lane of dQ^T)
    const int et = threadIdx.x - 384;     // 0..127 within this warpgroup
    float* stage = reinterpret_cast<float*>(smem + C::QS_OFF);
    for (int u = 0; u < cnt; ++u) {
      bool ok = mbar_wait(bar(P_DQF), u & 1, abort_flag, ctl, SITE_BWD_DQ_FULL);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t src = tmem + ((uint32_t)(q * 32) << 16) + C::DQ_COL;
      uint32_t a[32], c[32];
      tmem_ld32(src, a);
      tmem_ld32(src + 32, c);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(bar(P_DQE));            // the dQ^T columns may be refilled
      if (et == 0) bulk_wait_read_all();  // the previous reduce has read the stage
      named_bar_sync(1, 128);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        stage[i * D + r] = scale * __uint_as_float(a[i]);
        stage[(32 + i) * D + r] = scale * __uint_as_float(c[i]);
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (et == 0) {
        tma_reduce_add_3d(&tmdQ, smem_u32(stage), 0, (i_start + u) * C::BM, bh);
        bulk_commit_group();
      }
    }
    if (et == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc<512>(tmem);
}

template <bool DQ>
int launch(const void* Q, const void* K, const void* V, const void* dO, const float* LSE2,
           const float* Dv, float* dQacc, void* dK, void* dV, int BH, int n, int n_pad,
           float scale, int causal, const KernelCtl& ctl, cudaStream_t st) {
  using C = Kv128<DQ>;
  CUtensorMap tq, tk, tv, tg, tdq;
  if (!make_tmap_bf16(&tq, Q, 128, n, BH, 64, C::BM) ||
      !make_tmap_bf16(&tk, K, 128, n, BH, 64, C::BNK) ||
      !make_tmap_bf16(&tv, V, 128, n, BH, 64, C::BNK) ||
      !make_tmap_bf16(&tg, dO, 128, n, BH, 64, C::BM))
    return ATTN_ERR_CUDA;
  if (DQ) {
    if (!make_tmap_f32(&tdq, dQacc, 128, n, BH, 128, C::BM)) return ATTN_ERR_CUDA;
  } else {
    tdq = tq;   // not read
  }
  auto kern = bwd_kv128_kernel<DQ>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  dim3 grid(ceil_div(n, C::BNK), BH);
  kern<<<grid, C::NTHREADS, C::SMEM, st>>>(tq, tk, tv, tg, tdq, LSE2, Dv,
                                           static_cast<__nv_bfloat16*>(dK),
                                           static_cast<__nv_bfloat16*>(dV), n, n_pad, scale,
                                           scale * 1.4426950408889634f, causal, ctl);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

int launch_bwd_kv128_tc(const void* Q, const void* K, const void* V, const void* dO,
                        const float* LSE2, const float* Dv, float* dQacc, void* dK, void* dV,
                        int BH, int n, int n_pad, float scale, int causal, const KernelCtl& ctl,
                        cudaStream_t st) {
  if (dQacc)
    return launch<true>(Q, K, V, dO, LSE2, Dv, dQacc, dK, dV, BH, n, n_pad, scale, causal, ctl, st);
  return launch<false>(Q, K, V, dO, LSE2, Dv, dQacc, dK, dV, BH, n, n_pad, scale, causal, ctl, st);
}

}  // namespace attn
