// fwd_fp8.cu -- exact-attention forward with FP8 (e4m3) operands, head dim 128.
//
// The pages name FP8 computation as a FlashAttention-3 technique, together
// with quantisation-error reduction ("Flash Attention: Revolutionizing
// Transformer Efficiency", section FlashAttention-3, items 2-3).  This is the
// forward of fwd_tc.cu (online softmax over KV tiles, scores only in tensor
// memory: "Chapter 3.1 -- The cost of attention", section 5) with both
// products on the FP8 tensor cores (tcgen05 kind::f8f6f4, twice the bf16
// rate):
//   S   = Q K^T               e4m3 x e4m3 -> fp32 (SS-MMA, K = 32 per MMA)
//   P   = 2^(S c - m)         fp32 in registers, quantised to e4m3 in TMEM
//   O  += P V                 e4m3 (TMEM) x e4m3 -> fp32 (TS-MMA)
// with c = scale * descale_q[h] * descale_k[h] * log2(e) and O scaled by
// descale_v[h] / l at the end (descales per head, read from device memory, so
// that they can come from the quantiser without a host round trip).  The row sum l is taken over the fp32 values of
// P.  P stays below 2^8 (the running maximum is only kept while the new one
// exceeds it by at most 8 in log2 units), well inside e4m3's range (448).
// V is taken transposed (Vt: [d][n] per head) so that every FP8 operand is
// K-major.
//
// Roles and pipeline as fwd_tc.cu (two 128-row query tiles per CTA ping-pong
// two S slots; warp 0 loads Q and K, warp 3 loads Vt, warp 1 issues the MMAs
// from the whole warp with an elected lane, warpgroups 1 and 2 run the
// softmax of one tile each).  All waits are bounded.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm100.cuh"

namespace attn {
namespace {

using namespace sm100;

struct Fp8Cfg {
  static constexpr int D = 128, BM = 128, BN = 128, QT = 2;
  static constexpr int KST = 4, VST = 4;
  static constexpr uint32_t Q_BYTES = BM * D;          // 16 KB: [128 rows][128 B]
  static constexpr uint32_t K_BYTES = BN * D;          // 16 KB
  static constexpr uint32_t V_BYTES = D * BN;          // 16 KB: Vt tile [128 d][128 keys]
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = Q_OFF + QT * Q_BYTES;
  static constexpr uint32_t V_OFF = K_OFF + KST * K_BYTES;
  static constexpr uint32_t BAR_OFF = V_OFF + VST * V_BYTES;
  static constexpr uint32_t SMEM = BAR_OFF + 256 + 1024;
  static constexpr int S_COL = 0, O_COL = 2 * BN;
  static_assert(SMEM <= 232448, "shared memory budget");
};

enum : int { F_Q = 0, F_KF = 1, F_KE = 5, F_VF = 9, F_VE = 13, F_SF = 17, F_PF = 19, F_OD = 21,
             F_DRAIN = 23 };   // 24 barriers: 192 bytes

struct TileRange {
  int last0, last1;
};

// unit k -> (query tile t, KV tile j): pairs (0, j), (1, j) while both tiles
// need j, then tile 1 alone (it never needs fewer tiles than tile 0)
__device__ __forceinline__ int2 unit_of(int k, const TileRange& tr) {
  if (tr.last1 < 0) return make_int2(0, k);
  const int pairs = tr.last0 + 1;
  if (k < 2 * pairs) return make_int2(k & 1, k >> 1);
  return make_int2(1, k - pairs);
}
__device__ __forceinline__ int pos_of(int t, int j, const TileRange& tr) {
  return min(j, tr.last0 + 1) + min(j, tr.last1 + 1) + ((t == 1 && j <= tr.last0) ? 1 : 0);
}
// PV of unit k is followed by S of unit k + 2; when that is the same tile's
// next step, the S commit covers the PV, which then gets no commit of its own
// (both sides evaluate this to keep the O-done phases in step).
__device__ __forceinline__ bool pv_implied(int t, int j, const TileRange& tr) {
  const int last = t == 0 ? tr.last0 : tr.last1;
  return j < last && pos_of(t, j + 1, tr) == pos_of(t, j, tr) + 2;
}

__global__ void __launch_bounds__(384, 1)
fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmVt, __nv_bfloat16* __restrict__ O,
               float* __restrict__ LSE, const float* __restrict__ dsq,
               const float* __restrict__ dsk, const float* __restrict__ dsv, int n,
               float scale_log2_base, int causal, KernelCtl ctl) {
  using C = Fp8Cfg;
  static_assert(C::KST <= F_KE - F_KF && C::KST <= F_VF - F_KE && C::VST <= F_VE - F_VF &&
                    C::VST <= F_SF - F_VE,
                "ring deeper than its barrier slots");
  constexpr int D = C::D, BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::BAR_OFF + 192);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 200);

  const int warp = warp_id_uniform(), lane = threadIdx.x & 31;
  // Causal (tiles of unequal length): heads vary fastest in the grid, in
  // groups of 8 (the last group may be smaller), and tiles slowest, longest
  // first, so the long tiles of every head of a group start early while only
  // that group's K and V are in flight (kept in L2).  Otherwise tiles vary
  // fastest, which keeps a head's K and V shared in L2 by CTAs that run
  // together.
  const bool heads_fast = causal;
  int head_ix = heads_fast ? blockIdx.x : blockIdx.y;
  int tile_pos = heads_fast ? (int)blockIdx.y : (int)blockIdx.x;
  if (causal) {
    constexpr int kHeadGroup = 8;
    const int nh = (int)gridDim.x, nt = (int)gridDim.y;
    const int L = (int)(blockIdx.x + gridDim.x * blockIdx.y);
    const int full = nh / kHeadGroup, per = kHeadGroup * nt;
    if (L < full * per) {
      tile_pos = (L % per) / kHeadGroup;
      head_ix = (L / per) * kHeadGroup + (L % per) % kHeadGroup;
    } else {
      const int rest = nh - full * kHeadGroup, Lr = L - full * per;
      tile_pos = Lr / rest;
      head_ix = full * kHeadGroup + Lr % rest;
    }
  }
  const int bh = head_ix;
  const int ntile = heads_fast ? gridDim.y : gridDim.x;
  const int tile_ix = tile_pos;
  const int cta = causal ? (ntile - 1 - tile_ix) : tile_ix;
  const int row0 = cta * (C::QT * C::BM);
  const int nkv = (n + BN - 1) / BN;
  TileRange tr;
  {
    int last[2] = {-1, -1};
    for (int t = 0; t < C::QT; ++t) {
      const int r0 = row0 + t * C::BM;
      if (r0 < n) last[t] = causal ? min(nkv - 1, (r0 + C::BM - 1) / BN) : nkv - 1;
    }
    tr.last0 = last[0];
    tr.last1 = last[1];
  }
  const int jmax = max(tr.last0, tr.last1);

  if (threadIdx.x == 0) {
    mbar_init(bar(F_Q), 1);
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(bar(F_KF + s), 1);
      mbar_init(bar(F_KE + s), 1);
    }
    for (int s = 0; s < C::VST; ++s) {
      mbar_init(bar(F_VF + s), 1);
      mbar_init(bar(F_VE + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(F_SF + s), 1);
      mbar_init(bar(F_PF + s), 128);
      mbar_init(bar(F_OD + s), 1);
    }
    mbar_init(bar(F_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVt);
  }
  if (warp == 2) tmem_alloc<512>(smem_u32(tmem_slot));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 88;");
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------- producer: Q, then K tiles
      uint32_t qbytes = 0;
      for (int t = 0; t < C::QT; ++t)
        if (row0 + t * C::BM < n) qbytes += C::Q_BYTES;
      mbar_expect_tx(bar(F_Q), qbytes);
      for (int t = 0; t < C::QT; ++t)
        if (row0 + t * C::BM < n)
          tma_load_3d(sb + C::Q_OFF + t * C::Q_BYTES, &tmQ, 0, row0 + t * C::BM, bh, bar(F_Q));
      int last_k[C::KST];
      for (int s = 0; s < C::KST; ++s) last_k[s] = -1;
      for (int j = 0; j <= jmax; ++j) {
        const int s = j % C::KST;
        if (!mbar_wait(bar(F_KE + s), ((j / C::KST) & 1) ^ 1, abort_flag, ctl, SITE_FWD_KV_EMPTY))
          break;
        mbar_expect_tx(bar(F_KF + s), C::K_BYTES);
        tma_load_3d(sb + C::K_OFF + s * C::K_BYTES, &tmK, 0, j * BN, bh, bar(F_KF + s));
        last_k[s] = j;
      }
      if (*abort_flag) {   // let issued copies land before the CTA may exit
        volatile int no_abort = 0;
        mbar_wait(bar(F_Q), 0, &no_abort, ctl, SITE_FWD_LOAD_Q);
        for (int s = 0; s < C::KST; ++s)
          if (last_k[s] >= 0)
            mbar_wait(bar(F_KF + s), (last_k[s] / C::KST) & 1, &no_abort, ctl, SITE_FWD_K_FULL);
      }
    } else if (warp == 3 && lane == 0) {
      // ---------------------------------------------- producer: Vt tiles
      int last_v[C::VST];
      for (int s = 0; s < C::VST; ++s) last_v[s] = -1;
      for (int j = 0; j <= jmax; ++j) {
        const int s = j % C::VST;
        if (!mbar_wait(bar(F_VE + s), ((j / C::VST) & 1) ^ 1, abort_flag, ctl, SITE_FWD_KV_EMPTY))
          break;
        mbar_expect_tx(bar(F_VF + s), C::V_BYTES);
        tma_load_3d(sb + C::V_OFF + s * C::V_BYTES, &tmVt, j * BN, 0, bh, bar(F_VF + s));
        last_v[s] = j;
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        for (int s = 0; s < C::VST; ++s)
          if (last_v[s] >= 0)
            mbar_wait(bar(F_VF + s), (last_v[s] / C::VST) & 1, &no_abort, ctl, SITE_FWD_V_FULL);
      }
    } else if (warp == 1) {
      // ---------------------------------------------- MMA issuer (whole warp)
      constexpr uint32_t idesc_s = idesc_e4m3(C::BM, BN);   // Q, K K-major
      constexpr uint32_t idesc_o = idesc_e4m3(C::BM, D);    // P (TMEM), Vt K-major
      constexpr uint32_t HI = sdesc_hi(1024);
      const int total = (tr.last0 + 1) + (tr.last1 + 1);
      const uint32_t q_lo = sdesc_lo(sb + C::Q_OFF, 16), k_lo = sdesc_lo(sb + C::K_OFF, 16);
      const uint32_t v_lo = sdesc_lo(sb + C::V_OFF, 16);
      auto first_user = [&](int t, int j) { return t == 0 || j > tr.last0; };
      auto last_user = [&](int t, int j) { return t == 1 || j > tr.last1; };
      bool ok = mbar_wait_warp(bar(F_Q), 0, abort_flag, ctl, SITE_FWD_LOAD_Q);
      // S(k) = Q_t K_j^T into S slot k & 1: four MMAs of 32 e4m3 (32 bytes) of d
      auto issue_s = [&](int k) -> bool {
        const int2 u = unit_of(k, tr);
        const int s = u.y % C::KST;
        if (first_user(u.x, u.y)) {
          if (!mbar_wait_warp(bar(F_KF + s), (u.y / C::KST) & 1, abort_flag, ctl, SITE_FWD_K_FULL))
            return false;
        }
        tc_fence_after();
        uint32_t alo[4], blo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          alo[i] = q_lo + u.x * (C::Q_BYTES >> 4) + 2 * i;
          blo[i] = k_lo + s * (C::K_BYTES >> 4) + 2 * i;
        }
        mma_ss_x4_f8(tmem + C::S_COL + (k & 1) * BN, alo, HI, blo, HI, idesc_s, 0);
        tc_commit(bar(F_SF + (k & 1)));
        if (last_user(u.x, u.y)) tc_commit(bar(F_KE + s));
        return true;
      };
      if (ok && total > 0) ok = issue_s(0);
      if (ok && total > 1) ok = issue_s(1);
      for (int k = 0; ok && k < total; ++k) {
        const int2 u = unit_of(k, tr);
        const int s = u.y % C::VST;
        if (!mbar_wait_warp(bar(F_PF + (k & 1)), (k >> 1) & 1, abort_flag, ctl, SITE_FWD_P_FULL))
          break;
        if (first_user(u.x, u.y)) {
          if (!mbar_wait_warp(bar(F_VF + s), (u.y / C::VST) & 1, abort_flag, ctl, SITE_FWD_V_FULL))
            break;
        }
        tc_fence_after();
        // O_t += P Vt^T: P's 128 keys in 32 columns of slot k & 1, four MMAs of 32 keys
        uint32_t blo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) blo[i] = v_lo + s * (C::V_BYTES >> 4) + 2 * i;
        mma_ts_x4_f8(tmem + C::O_COL + u.x * D, tmem + C::S_COL + (k & 1) * BN, blo, HI, idesc_o,
                     u.y > 0);
        if (!pv_implied(u.x, u.y, tr)) tc_commit(bar(F_OD + u.x));
        if (last_user(u.x, u.y)) tc_commit(bar(F_VE + s));
        if (k + 2 < total) ok = issue_s(k + 2);
      }
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        tc_commit(bar(F_DRAIN));
        volatile int no_abort = 0;
        mbar_wait_warp(bar(F_DRAIN), 0, &no_abort, ctl, SITE_FWD_O_DONE);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax
    asm volatile("setmaxnreg.inc.sync.aligned.u32 208;");
    const float scale_log2 =
        scale_log2_base * (dsq ? dsq[bh] : 1.0f) * (dsk ? dsk[bh] : 1.0f);
    const float descale_v = dsv ? dsv[bh] : 1.0f;
    const int t = (warp >> 2) - 1;
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int row = row0 + t * C::BM + r;
    const int last = (t == 0) ? tr.last0 : tr.last1;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    float m = -INFINITY, l = 0.f;
    int odc = 0;   // O-done phases consumed
    bool ok = true;
    for (int j = 0; j <= last; ++j) {
      const int k = pos_of(t, j, tr);
      const int slot = k & 1;
      ok = mbar_wait_warp(bar(F_SF + slot), (k >> 1) & 1, abort_flag, ctl, SITE_FWD_S_FULL);
      if (!ok) break;
      tc_fence_after();
      const uint32_t sa = tmem + lane_off + C::S_COL + slot * BN;
      uint32_t sr[BN];
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32)
        tmem_ld32(sa + c0, *reinterpret_cast<uint32_t(*)[32]>(&sr[c0]));
      tmem_ld_wait();
      reg_fence<BN>(sr);
      float* s = reinterpret_cast<float*>(sr);
      const int col0 = j * BN;
      if ((col0 + BN > n) || (causal && col0 + BN - 1 > row0 + t * C::BM)) {
        const int lim = causal ? min(n, row + 1) : n;   // columns < lim are kept
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (col0 + c >= lim) s[c] = -INFINITY;
      }
      // row maximum: three-input maxima in four independent chains
      float mx4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int c = 4; c < BN; c += 2) mx4[(c >> 1) & 3] = max3f(mx4[(c >> 1) & 3], s[c], s[c + 1]);
      const float mx = max3f(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
      const float m_cand = mx * scale_log2;
      const float m_new = (m_cand > m + 8.0f) ? m_cand : m;
      const float alpha = ex2(m - m_new);   // 0 on the first tile (m = -inf)
      // exponents and row sum on column pairs (paired fp32 FMA and add)
      const float2 c2 = make_float2(scale_log2, scale_log2);
      const float2 nm2 = make_float2(-m_new, -m_new);
      float2 rs4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                       make_float2(0.f, 0.f)};
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 64) {   // 64 keys -> 16 columns of packed e4m3
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float2 p[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = c0 + 4 * i + 2 * h;
            const float2 x = __ffma2_rn(make_float2(s[c], s[c + 1]), c2, nm2);
            p[h] = make_float2(ex2(x.x), ex2(x.y));
            rs4[(2 * i + h) & 3] = __fadd2_rn(rs4[(2 * i + h) & 3], p[h]);
          }
          pk[i] = pack_e4m3x4(p[0].x, p[0].y, p[1].x, p[1].y);
        }
        tmem_st16(sa + c0 / 4, pk);   // P overwrites the first BN/4 columns of the slot
      }
      const float2 rs2 = __fadd2_rn(__fadd2_rn(rs4[0], rs4[1]), __fadd2_rn(rs4[2], rs4[3]));
      const float rs = rs2.x + rs2.y;
      tmem_st_wait();
      l = l * alpha + rs;
      if (j > 0 && !pv_implied(t, j - 1, tr)) {   // PV of step j-1 done before any rescale
        ok = mbar_wait_warp(bar(F_OD + t), odc & 1, abort_flag, ctl, SITE_FWD_O_DONE);
        if (!ok) break;
        ++odc;
      }
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {   // kept maximum moved
        tc_fence_after();
        const uint32_t oa = tmem + lane_off + C::O_COL + t * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(oa + c0, rr);
          tmem_ld_wait();
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 o2 = __fmul2_rn(
                make_float2(__uint_as_float(rr[i]), __uint_as_float(rr[i + 1])), a2);
            rr[i] = __float_as_uint(o2.x);
            rr[i + 1] = __float_as_uint(o2.y);
          }
          tmem_st32(oa + c0, rr);
        }
        tmem_st_wait();
      }
      m = m_new;
      tc_fence_before();
      mbar_arrive(bar(F_PF + slot));
    }
    if (ok && last >= 0) {
      ok = mbar_wait_warp(bar(F_OD + t), odc & 1, abort_flag, ctl, SITE_FWD_O_DONE);   // last PV
      if (ok) {
        tc_fence_after();
        const float mul = descale_v / l;
        const uint32_t oa = tmem + lane_off + C::O_COL + t * D;
        __nv_bfloat16* orow = O + ((size_t)bh * n + row) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(oa + c0, rr);
          tmem_ld_wait();
          if (row < n) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * mul,
                                  __uint_as_float(rr[2 * i + 1]) * mul);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              reinterpret_cast<uint4*>(orow + c0)[i] =
                  make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
        if (row < n) LSE[(size_t)bh * n + row] = (m + __log2f(l)) * 0.69314718055994531f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc<512>(tmem);
}

}  // namespace

int launch_fwd_fp8(const void* Q8, const void* K8, const void* Vt8, void* O, float* LSE, int BH,
                   int n, float scale, const float* descale_q, const float* descale_k,
                   const float* descale_v, int causal, const KernelCtl& ctl, cudaStream_t st) {
  using C = Fp8Cfg;
  if (n % 16 != 0) return ATTN_ERR_UNSUPPORTED;   // Vt rows of n bytes: 16-byte strides
  CUtensorMap tq, tk, tv;
  if (!make_tmap_u8(&tq, Q8, C::D, n, BH, 128, C::BM) ||
      !make_tmap_u8(&tk, K8, C::D, n, BH, 128, C::BN) ||
      !make_tmap_u8(&tv, Vt8, n, C::D, BH, 128, C::D))
    return ATTN_ERR_CUDA;
  if (cudaFuncSetAttribute(fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  const int ntile = ceil_div(n, C::QT * C::BM);
  dim3 grid = causal ? dim3(BH, ntile) : dim3(ntile, BH);
  fwd_fp8_kernel<<<grid, 384, C::SMEM, st>>>(tq, tk, tv, static_cast<__nv_bfloat16*>(O), LSE,
                                             descale_q, descale_k, descale_v, n,
                                             scale * 1.4426950408889634f, causal, ctl);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn
