// bwd_kv.cuh -- key-tile attention backward for head dims 64 and 128
// (instantiated by bwd_kv128.cu and bwd_kv64.cu).
//
// One CTA owns 128 keys of one head (the TMEM lanes) and walks the 128-query
// tiles that can see them.  For every query tile u, with c = scale * log2(e)
// and LSE2 = LSE * log2(e):
//   S^T  = K Q_u^T                (SS-MMA, M = 128 keys, N = 128 queries)
//   P^T  = 2^(S^T c - LSE2)       (registers; bf16 copy back into TMEM)
//   dV  += P^T dO_u               (TS-MMA: A = P^T read from TMEM)
//   dP^T = V dO_u^T               (SS-MMA)
//   dS^T = P^T o (dP^T - D)       (registers; bf16 copy into shared memory)
//   dK  += dS^T Q_u               (SS-MMA: A = dS^T, K-major over the queries)
//   dQ_u = dS K                   (SS-MMA: A = dS, MN-major; M = 128 queries)
// These are the chain-rule steps of the backward pass that recomputes the
// attention matrix instead of storing it ("Chapter 3.1 -- The cost of
// attention", section 5; "Flash Attention: Revolutionizing Transformer
// Efficiency", key idea 2).
//
// Why 128-query tiles: an SS-MMA of M = 128 rows reads (128 + N) x 16 x 2
// bytes of shared memory per 2 x 128 x N x 16 FLOPs.  At N = 64 the tensor
// cores' operand traffic exceeds their MMA time; at N = 128 it stays below.
//
// Tensor memory: dV [0,D), dK [D,2D), S^T [2D,2D+128), dP^T [2D+128,2D+256)
// (all 512 columns for D = 128).  The dQ tile reuses the dP^T columns once
// the compute warps have read dP^T, so S of the next tile is issued right
// after dV and its exponentials overlap this tile's dK and dQ products.
// dS^T [128 keys][128 queries] is written over the dO tile of its stage
// after dV has consumed dO when D = 128 (the tiles are the same size); for
// D = 64 the stage carries its own dS^T buffer.  dQ is issued
// before dK so that its drain overlaps the dK product.  The dQ warpgroup
// (given 176 registers by setmaxnreg) pulls the whole fp32 dQ tile out of
// TMEM and releases the columns; each 64-row half (two warps) then adds its
// rows into the global fp32 accumulator as four 64 x 32 boxes staged in its
// own 8 KB of shared memory (128-byte swizzle), one TMA bulk reduce-add
// each, so two reduce-adds are in flight.  What sets the period at D = 128
// is the chain through the dP^T columns (dQ(u), its read-out, then
// dP^T(u+1)) followed by the compute warps' dS and dS^T store; the SS
// products read 128 B/clk of shared memory while they run and slow down
// when the tile loads and dQ staging run beside them.
// Every wait is bounded (mbar_wait).
#pragma once
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

template <int D_>
struct KvCfgT {
  static constexpr int D = D_, BNK = 128, BM = 128, NKB = D / 64, STG = 2;
  static constexpr uint32_t KV_BYTES = BNK * D * 2;           // 32 KB (D = 128)
  static constexpr uint32_t QT_BYTES = BM * D * 2;            // 32 KB (D = 128)
  static constexpr uint32_t DS_BYTES = BNK * BM * 2;          // dS^T: 32 KB
  // stage: Q, dO, LSE2 (+0), D (+512), then dS^T when it does not fit over dO
  static constexpr bool DS_OVER_DO = (QT_BYTES == DS_BYTES);
  static constexpr uint32_t DS_OFF = DS_OVER_DO ? QT_BYTES : 2 * QT_BYTES + 1024;
  static constexpr uint32_t STAGE = 2 * QT_BYTES + 1024 + (DS_OVER_DO ? 0 : DS_BYTES);
  static constexpr uint32_t K_OFF = 0, V_OFF = KV_BYTES;
  static constexpr uint32_t ST_OFF = 2 * KV_BYTES;
  // dQ staging: per 64-row half of the tile, QS_NBUF boxes of [64][32] fp32
  // (8 KB each, 128-byte swizzle), so each half keeps QS_NBUF reduce-adds
  // in flight
  static constexpr int QS_NBUF = 2;
  static constexpr uint32_t QS_BOX = 64 * 32 * 4;
  static constexpr uint32_t QS_OFF = ST_OFF + STG * STAGE;
  static constexpr uint32_t QS_BYTES = 2 * QS_NBUF * QS_BOX;
  static constexpr uint32_t BAR_OFF = QS_OFF + QS_BYTES;
  // 1 KB of slack to align the base when it fits; otherwise the kernel checks
  // that the dynamic shared memory starts 1024-byte aligned
  static constexpr uint32_t ALIGN_SLACK = (BAR_OFF + 256 + 1024 <= 232448) ? 1024 : 0;
  static constexpr uint32_t SMEM = BAR_OFF + 256 + ALIGN_SLACK;
  static constexpr int DV_COL = 0, DK_COL = D, S_COL = 2 * D, DP_COL = 2 * D + 128;
  // d = 128: the compute warps read the first 32 LSE2 values of a tile
  // before waiting for S^T, so that their shared-memory latency stays off
  // the chain (D cannot follow: P is live by then, and 128 registers do not
  // hold both)
  static constexpr bool EARLY_LD = (D == 128);
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(STAGE % 1024 == 0, "stages stay 1024-byte aligned for the swizzle");
};

enum : int { B_KV = 0, B_QF = 1, B_QE = 3, B_SF = 5, B_DPF = 6, B_PR = 7, B_DVD = 8, B_DSR = 9,
             B_DQF = 10, B_DQE = 11, B_ACC = 12, B_DRAIN = 13 };

// GROUPED: query heads share key/value heads (compiled separately so that the
// one-head-per-head kernel keeps its simple loops).  SPARSE: a block pattern
// keeps only some query tiles for this key tile; the CTA walks that list
// (every listed tile lies in kept blocks) instead of the dense range.
// KR < 128 (IO study only): the CTA owns the first KR keys of its 128-key
// tile, key tiles start KR keys apart, and the other keys' probabilities are
// set to 0, so the CTA keeps KR keys' worth of K and V on chip and Q and dO
// are streamed 128 / KR times as often.
template <int DH, bool DQ, bool GROUPED, bool SPARSE, int KR = 128>
__global__ void __launch_bounds__(DQ ? 512 : 384, 1)
bwd_kv128_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmdQ, const float* __restrict__ LSE2, const float* __restrict__ Dv,
                  float* __restrict__ dQacc, __nv_bfloat16* __restrict__ dK,
                  __nv_bfloat16* __restrict__ dV, float* __restrict__ dKacc,
                  float* __restrict__ dVacc, HeadMap hm, int gsplit, TileLists tl, int n,
                  int n_pad, float scale, float scale_log2, int causal, KernelCtl ctl) {
  using C = KvCfgT<DH>;
  constexpr int D = DH;
  static_assert(KR == C::BNK || (KR >= 32 && KR < C::BNK && !SPARSE && !GROUPED),
                "owned key rows: a dense, one-head-per-head study instance");
  extern __shared__ uint8_t smem_raw[];
  if constexpr (C::ALIGN_SLACK == 0) {
    // no room to align the layout: it needs the base 1024-byte aligned (the
    // 128-byte swizzle atoms); report and leave before touching anything
    if (smem_u32(smem_raw) & 1023u) {
      if (threadIdx.x == 0) record_error(ctl, ATTN_ERR_CUDA, SITE_BWD_SMEM_ALIGN);
      return;
    }
  }
  uint8_t* smem = align_1k(smem_raw);
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::BAR_OFF + 192);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 200);

  const int warp = warp_id_uniform(), lane = threadIdx.x & 31;
  // Causal or block-sparse (tiles of unequal length): heads vary fastest in
  // the grid and tiles slowest, longest first, so the long tiles of every
  // head start early instead of the last heads' long tiles trailing the rest
  // (CTAs start in grid order).  Otherwise tiles vary fastest, which keeps a
  // head's K and V shared in L2 by CTAs that run together.  The parts of a
  // split group count as heads here (hx = part * key/value heads + head), so
  // the last part's long tiles do not trail either.  Causal and dense, the
  // heads go in groups of kHeadGroup (the last group may be smaller), each
  // group in that order, group after group: only one group's Q, dO and dQ
  // accumulators are then in flight, which keeps them in L2 (DRAM bytes per
  // launch 2.92 -> 0.64 GB on B2 H16 n8192 d128, at the same speed) while
  // every long tile still starts before the short ones of its group.
  const bool heads_fast = causal || SPARSE;
  int kt = heads_fast ? blockIdx.y : blockIdx.x;
  int hx = heads_fast ? blockIdx.x : blockIdx.y;
  if (causal && !SPARSE) {
    constexpr int kHeadGroup = 8;
    const int nh = (int)gridDim.x, ntile = (int)gridDim.y;
    const int L = (int)(blockIdx.x + gridDim.x * blockIdx.y);
    const int full = nh / kHeadGroup, per = kHeadGroup * ntile;
    if (L < full * per) {
      kt = (L % per) / kHeadGroup;
      hx = (L / per) * kHeadGroup + (L % per) % kHeadGroup;
    } else {
      const int rest = nh - full * kHeadGroup, Lr = L - full * per;
      kt = Lr / rest;
      hx = full * kHeadGroup + Lr % rest;
    }
  }
  const int nkvh = (heads_fast ? (int)gridDim.x : (int)gridDim.y) / gsplit;
  const int bh = hx % nkvh;           // key/value head (K, V, dK, dV)
  const int part = hx / nkvh;         // part of the group
  const int k0 = kt * KR;
  const int nq = (n + C::BM - 1) / C::BM;
  const int i_start = causal ? (k0 / C::BM) : 0;
  const int* qlist = SPARSE ? tl.lists + (size_t)kt * tl.stride : nullptr;
  const int cnt = SPARSE ? tl.counts[kt] : nq - i_start;   // query tiles per query head
  auto qtile = [&](int ut) { return SPARSE ? (qlist[ut] & 0xFFFF) : i_start + ut; };
  // The query heads of this key/value head's group are split over gsplit
  // CTAs (part); iteration u visits query tile i_start + u % cnt of
  // query head qbase + u / cnt, so dK and dV accumulate over this CTA's part
  // of the group (over the whole group when gsplit = 1).  Each role runs an
  // outer loop over its heads and an inner loop over the query tiles.
  const int gper = GROUPED ? hm.group / gsplit : 1;
  const int qbase = GROUPED ? hm.q_of(bh, part * gper) : bh;
  const int total = gper * cnt;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_KV), 1);
    for (int s = 0; s < C::STG; ++s) { mbar_init(bar(B_QF + s), 1); mbar_init(bar(B_QE + s), 1); }
    mbar_init(bar(B_SF), 1);
    mbar_init(bar(B_DPF), 1);
    mbar_init(bar(B_PR), 256);
    mbar_init(bar(B_DVD), 1);
    mbar_init(bar(B_DSR), 256);
    mbar_init(bar(B_DQF), 1);
    mbar_init(bar(B_DQE), 128);
    mbar_init(bar(B_ACC), 1);
    mbar_init(bar(B_DRAIN), 1);
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
    if (DQ) asm volatile("setmaxnreg.dec.sync.aligned.u32 80;");
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------ producer
      mbar_expect_tx(bar(B_KV), 2 * C::KV_BYTES);
#pragma unroll
      for (int kb = 0; kb < C::NKB; ++kb) {
        tma_load_3d(sb + C::K_OFF + kb * (C::BNK * 128), &tmK, kb * 64, k0, bh, bar(B_KV));
        tma_load_3d(sb + C::V_OFF + kb * (C::BNK * 128), &tmV, kb * 64, k0, bh, bar(B_KV));
      }
      int last[C::STG] = {-1, -1};
      bool go = true;
      for (int gi = 0, u = 0; go && gi < gper; ++gi) {
        const int bq = qbase + gi;
        for (int ut = 0; ut < cnt; ++ut, ++u) {
          const int s = u % C::STG;
          const int q0 = qtile(ut) * C::BM;
          if (!mbar_wait(bar(B_QE + s), ((u / C::STG) & 1) ^ 1, abort_flag, ctl, SITE_BWD_Q_EMPTY)) {
            go = false;
            break;
          }
          const uint32_t st = sb + C::ST_OFF + s * C::STAGE;
          mbar_expect_tx(bar(B_QF + s), 2 * C::QT_BYTES + 2 * C::BM * 4);
#pragma unroll
          for (int kb = 0; kb < C::NKB; ++kb) {
            tma_load_3d(st + kb * (C::BM * 128), &tmQ, kb * 64, q0, bq, bar(B_QF + s));
            tma_load_3d(st + C::QT_BYTES + kb * (C::BM * 128), &tmdO, kb * 64, q0, bq, bar(B_QF + s));
          }
          bulk_load(st + 2 * C::QT_BYTES, LSE2 + (size_t)bq * n_pad + q0, C::BM * 4, bar(B_QF + s));
          bulk_load(st + 2 * C::QT_BYTES + 512, Dv + (size_t)bq * n_pad + q0, C::BM * 4,
                    bar(B_QF + s));
          if (s == 0) last[0] = u; else last[1] = u;
        }
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        mbar_wait(bar(B_KV), 0, &no_abort, ctl, SITE_BWD_KV);
        if (last[0] >= 0) mbar_wait(bar(B_QF), (last[0] / 2) & 1, &no_abort, ctl, SITE_BWD_Q_FULL);
        if (last[1] >= 0) mbar_wait(bar(B_QF + 1), (last[1] / 2) & 1, &no_abort, ctl, SITE_BWD_Q_FULL);
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // (the whole warp runs the loop; one elected lane issues each MMA/commit)
      constexpr uint32_t id_s = idesc_bf16(128, C::BM, false, false);   // K/V, Q/dO K-major
      constexpr uint32_t id_acc = idesc_bf16(128, D, false, true);      // A K-major, B MN-major
      constexpr uint32_t id_dq = idesc_bf16(128, D, true, true);        // dS, K both MN-major
      // Descriptors from precomputed 32-bit halves; each group of four MMAs is
      // issued from one asm block (the MMA queue is shallow, so scalar work
      // between MMAs costs tensor time).
      constexpr uint32_t HI = sdesc_hi(1024);
      const uint32_t k_km = sdesc_lo(sb + C::K_OFF, 16);              // K tile, K-major
      const uint32_t v_km = sdesc_lo(sb + C::V_OFF, 16);              // V tile, K-major
      const uint32_t k_mn = sdesc_lo(sb + C::K_OFF, C::BNK * 128);    // K tile, MN-major
      const uint32_t st_km = sdesc_lo(sb + C::ST_OFF, 16);            // stage 0, K-major
      const uint32_t st_mn = sdesc_lo(sb + C::ST_OFF, C::BM * 128);   // stage 0, MN-major
      const uint32_t ds_mn = sdesc_lo(sb + C::ST_OFF, C::BNK * 128);  // dS (stage 0), MN-major
      constexpr uint32_t STG16 = C::STAGE >> 4, QT16 = C::QT_BYTES >> 4, DS16 = C::DS_OFF >> 4;
      // K-major operand, 64-wide column box b of a tile with `rows` rows
      auto km4 = [](uint32_t base, int rows, int b, uint32_t (&lo)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) lo[i] = base + b * (rows * 128 / 16) + 2 * i;
      };
      // MN-major operand, K slices 4g .. 4g+3 (16 rows = 2048 bytes each)
      auto mn4 = [](uint32_t base, int g, uint32_t (&lo)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) lo[i] = base + (4 * g + i) * (2048 / 16);
      };
      auto issue_s = [&](int u) -> bool {   // S^T(u) = K Q(u)^T
        if (!mbar_wait_warp(bar(B_QF + u % C::STG), (u / C::STG) & 1, abort_flag, ctl, SITE_BWD_Q_FULL))
          return false;
        tc_fence_after();
        const uint32_t qb = st_km + (u % C::STG) * STG16;
#pragma unroll
        for (int b = 0; b < C::NKB; ++b) {
          uint32_t alo[4], blo[4];
          km4(k_km, C::BNK, b, alo);
          km4(qb, C::BM, b, blo);
          mma_ss_x4(tmem + C::S_COL, alo, HI, blo, HI, id_s, b > 0);
        }
        tc_commit(bar(B_SF));
        return true;
      };
      auto issue_dp = [&](int u) {          // dP^T(u) = V dO(u)^T  (stage already full)
        const uint32_t gb = st_km + (u % C::STG) * STG16 + QT16;
#pragma unroll
        for (int b = 0; b < C::NKB; ++b) {
          uint32_t alo[4], blo[4];
          km4(v_km, C::BNK, b, alo);
          km4(gb, C::BM, b, blo);
          mma_ss_x4(tmem + C::DP_COL, alo, HI, blo, HI, id_s, b > 0);
        }
        tc_commit(bar(B_DPF));
      };
      bool ok = mbar_wait_warp(bar(B_KV), 0, abort_flag, ctl, SITE_BWD_KV);
      if (ok && total > 0) ok = issue_s(0);
      if (ok && total > 0) issue_dp(0);
      for (int u = 0; ok && u < total; ++u) {
        const uint32_t so = (u % C::STG) * STG16;
        // dV += P^T dO(u): P^T in the S columns, half h at [64h, 64h+32)
        if (!(ok = mbar_wait_warp(bar(B_PR), u & 1, abort_flag, ctl, SITE_BWD_P_READY))) break;
        tc_fence_after();
#pragma unroll
        for (int g = 0; g < C::BM / 64; ++g) {
          uint32_t blo[4];
          mn4(st_mn + so + QT16, g, blo);
          mma_ts_x4(tmem + C::DV_COL, tmem + C::S_COL + 64 * g, blo, HI, id_acc, (u > 0 || g > 0));
        }
        tc_commit(bar(B_DVD));
        if (u + 1 < total) {
          if (!(ok = issue_s(u + 1))) break;
        }
        if (!(ok = mbar_wait_warp(bar(B_DSR), u & 1, abort_flag, ctl, SITE_BWD_DS_READY))) break;
        tc_fence_after();
        if (DQ) {
          // dQ(u) = dS K into the dP^T columns (read by the compute warps already);
          // first, so that the dQ warpgroup drains it while dK runs
#pragma unroll
          for (int g = 0; g < C::BNK / 64; ++g) {
            uint32_t alo[4], blo[4];
            mn4(ds_mn + so + DS16, g, alo);
            mn4(k_mn, g, blo);
            mma_ss_x4(tmem + C::DP_COL, alo, HI, blo, HI, id_dq, g > 0);
          }
          tc_commit(bar(B_DQF));
        }
        // dK += dS^T Q(u): dS^T [128 keys][128 queries], K-major
#pragma unroll
        for (int b = 0; b < C::BM / 64; ++b) {
          uint32_t alo[4], blo[4];
          km4(st_km + so + DS16, C::BNK, b, alo);
          mn4(st_mn + so, b, blo);
          mma_ss_x4(tmem + C::DK_COL, alo, HI, blo, HI, id_acc, (u > 0 || b > 0));
        }
        tc_commit(bar(B_QE + u % C::STG));
        if (u + 1 < total) {
          if (DQ) {
            if (!(ok = mbar_wait_warp(bar(B_DQE), u & 1, abort_flag, ctl, SITE_BWD_DQ_FREE))) break;
            tc_fence_after();
          }
          issue_dp(u + 1);   // the stage of u + 1 is full: S(u+1) waited for it
        }
      }
      tc_commit(bar(B_ACC));
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        tc_commit(bar(B_DRAIN));
        volatile int no_abort = 0;
        mbar_wait_warp(bar(B_DRAIN), 0, &no_abort, ctl, SITE_BWD_ACC_DONE);
      }
    }
    __syncwarp();
  } else if (warp < 12) {
    // ---------------------------------------------------------------- compute
    const int q = warp & 3, h = (warp - 4) >> 2;
    const int r = q * 32 + lane;
    const int key = k0 + r;
    constexpr int NC = 64;                 // queries [64h, 64h+64)
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + C::S_COL + h * NC;
    const uint32_t dp_addr = tmem + lane_off + C::DP_COL + h * NC;
    bool ok = true;
    for (int gi = 0, u = 0; ok && gi < gper; ++gi) {
      for (int ut = 0; ut < cnt; ++ut, ++u) {
        const int s = u % C::STG;
        const int q0 = qtile(ut) * C::BM;
        uint8_t* stp = smem + C::ST_OFF + s * C::STAGE;
        const float* lse2 = reinterpret_cast<const float*>(stp + 2 * C::QT_BYTES) + h * NC;
        const float* dd = reinterpret_cast<const float*>(stp + 2 * C::QT_BYTES + 512) + h * NC;
        ok = mbar_wait(bar(B_QF + s), (u / C::STG) & 1, abort_flag, ctl, SITE_BWD_Q_FULL);
        float4 pre[C::EARLY_LD ? 8 : 1];   // EARLY_LD: LSE2 of the first 32 columns
        if constexpr (C::EARLY_LD) {
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) pre[i4] = reinterpret_cast<const float4*>(lse2)[i4];
        }
        ok = ok && mbar_wait(bar(B_SF), u & 1, abort_flag, ctl, SITE_BWD_S_FULL);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const bool masked = causal && (k0 + C::BNK - 1 > q0);
        const int qbase = q0 + h * NC;
        float p[NC];
        if constexpr (D == 64) {
          // both TMEM loads in flight before one wait, LSE2 four at a time
          // (every lane reads the same words), column pairs on the paired
          // fp32 FMA (measured: +3 % at d = 64, -1 % at d = 128)
          uint32_t* pr = reinterpret_cast<uint32_t*>(p);
          tmem_ld32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(pr));
          tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(pr + 32));
          tmem_ld_wait();
          reg_fence<NC>(*reinterpret_cast<uint32_t(*)[NC]>(pr));
          const float4* l4 = reinterpret_cast<const float4*>(lse2);
          const float2 c2 = make_float2(scale_log2, scale_log2);
#pragma unroll
          for (int i4 = 0; i4 < NC / 4; ++i4) {
            const float4 L = l4[i4];
            const float2 x0 = __ffma2_rn(make_float2(p[4 * i4], p[4 * i4 + 1]), c2, make_float2(-L.x, -L.y));
            const float2 x1 = __ffma2_rn(make_float2(p[4 * i4 + 2], p[4 * i4 + 3]), c2,
                                         make_float2(-L.z, -L.w));
            p[4 * i4] = ex2(x0.x);
            p[4 * i4 + 1] = ex2(x0.y);
            p[4 * i4 + 2] = ex2(x1.x);
            p[4 * i4 + 3] = ex2(x1.y);
          }
          if (masked) {
#pragma unroll
            for (int c = 0; c < NC; ++c)
              if (key > qbase + c) p[c] = 0.f;
          }
        } else {
#pragma unroll
          for (int c0 = 0; c0 < NC; c0 += 32) {
            uint32_t rr[32];
            tmem_ld32(s_addr + c0, rr);
            // LSE2 four at a time: one shared-memory wavefront per four words
            // (every lane reads the same ones); 1.110 -> 1.085 ms on the
            // B2 H16 n8192 causal backward, with D read the same way
            const float4* l4 = reinterpret_cast<const float4*>(lse2 + c0);
            tmem_ld_wait();
            {
#pragma unroll
              for (int i4 = 0; i4 < 8; ++i4) {
                const float4 L = (C::EARLY_LD && c0 == 0) ? pre[i4] : l4[i4];
                p[c0 + 4 * i4] = ex2(fmaf(__uint_as_float(rr[4 * i4]), scale_log2, -L.x));
                p[c0 + 4 * i4 + 1] = ex2(fmaf(__uint_as_float(rr[4 * i4 + 1]), scale_log2, -L.y));
                p[c0 + 4 * i4 + 2] = ex2(fmaf(__uint_as_float(rr[4 * i4 + 2]), scale_log2, -L.z));
                p[c0 + 4 * i4 + 3] = ex2(fmaf(__uint_as_float(rr[4 * i4 + 3]), scale_log2, -L.w));
              }
              if (masked) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  if (key > qbase + c0 + i) p[c0 + i] = 0.f;
              }
            }
          }
        }
        if constexpr (KR < C::BNK) {   // keys of the next study tile: no contribution
          if (r >= KR) {
#pragma unroll
            for (int c = 0; c < NC; ++c) p[c] = 0.f;
          }
        }
#pragma unroll
        for (int c0 = 0; c0 < NC; c0 += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(p[c0 + 2 * i], p[c0 + 2 * i + 1]);
          tmem_st16(s_addr + c0 / 2, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_PR));
        ok = mbar_wait(bar(B_DPF), u & 1, abort_flag, ctl, SITE_BWD_DP_FULL);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t ds[NC / 2];
#pragma unroll
        for (int c0 = 0; c0 < NC; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(dp_addr + c0, rr);
          tmem_ld_wait();
          if constexpr (D == 64) {   // D four at a time, paired fp32 subtract and multiply
            const float4* d4 = reinterpret_cast<const float4*>(dd + c0);
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              const float4 Dq = d4[i4];
              const int c = c0 + 4 * i4;
              const float2 x0 = __fmul2_rn(
                  make_float2(p[c], p[c + 1]),
                  __fadd2_rn(make_float2(__uint_as_float(rr[4 * i4]), __uint_as_float(rr[4 * i4 + 1])),
                             make_float2(-Dq.x, -Dq.y)));
              const float2 x1 = __fmul2_rn(
                  make_float2(p[c + 2], p[c + 3]),
                  __fadd2_rn(make_float2(__uint_as_float(rr[4 * i4 + 2]), __uint_as_float(rr[4 * i4 + 3])),
                             make_float2(-Dq.z, -Dq.w)));
              ds[c0 / 2 + 2 * i4] = pack_bf16x2(x0.x, x0.y);
              ds[c0 / 2 + 2 * i4 + 1] = pack_bf16x2(x1.x, x1.y);
            }
          } else {   // D four at a time
            const float4* d4 = reinterpret_cast<const float4*>(dd + c0);
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              const float4 Dq = d4[i4];
              const int c = c0 + 4 * i4;
              ds[c / 2] = pack_bf16x2(p[c] * (__uint_as_float(rr[4 * i4]) - Dq.x),
                                      p[c + 1] * (__uint_as_float(rr[4 * i4 + 1]) - Dq.y));
              ds[c / 2 + 1] = pack_bf16x2(p[c + 2] * (__uint_as_float(rr[4 * i4 + 2]) - Dq.z),
                                          p[c + 3] * (__uint_as_float(rr[4 * i4 + 3]) - Dq.w));
            }
          }
        }
        tc_fence_before();
        // dS^T over dO(u) must wait until dV(u) has read dO; a separate
        // buffer is free (its last readers, dK and dQ of the stage's previous
        // tile, finished before the stage was refilled).  The phase is
        // consumed either way so that parity waits stay one phase behind.
        ok = mbar_wait(bar(B_DVD), u & 1, abort_flag, ctl, SITE_BWD_DS_FREE);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        uint8_t* rowp = stp + C::DS_OFF + h * (C::BNK * 128);   // query block h, key row r
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(rowp + sw128_offset(r, c)) =
              make_uint4(ds[4 * c], ds[4 * c + 1], ds[4 * c + 2], ds[4 * c + 3]);
        fence_proxy_async_smem();
        mbar_arrive(bar(B_DSR));
      }
    }
    if (ok) {
      ok = mbar_wait(bar(B_ACC), 0, abort_flag, ctl, SITE_BWD_ACC_DONE);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const uint32_t src = tmem + lane_off + (h == 0 ? C::DV_COL : C::DK_COL);
      const float mul = h == 0 ? 1.f : scale;
      const size_t row = (size_t)bh * n + key;
      float* acc = GROUPED ? (h == 0 ? dVacc : dKacc) : nullptr;   // set when the group is split
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(src + c0, rr);
        tmem_ld_wait();
        if (SPARSE && total == 0) {   // no kept query tile: dK = dV = 0, TMEM never written
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = 0u;
        }
        if (key < n && (KR == C::BNK || r < KR)) {
          if (acc) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              red_add_v4(acc + row * D + c0 + i, mul * __uint_as_float(rr[i]),
                         mul * __uint_as_float(rr[i + 1]), mul * __uint_as_float(rr[i + 2]),
                         mul * __uint_as_float(rr[i + 3]));
          } else {
            store_row32_bf16((h == 0 ? dV : dK) + row * D + c0, rr, mul);
          }
        }
      }
    }
  } else if (DQ) {
    // ---------------------------------------------------------------- dQ warpgroup
    // Pulls the whole 128 x D fp32 dQ tile out of TMEM (thread = query row)
    // and releases the columns at once.  Each half (warps 2h, 2h+1 of the
    // group: rows [64h, 64h+64)) then adds its rows into the accumulator as
    // D / 32 boxes of 64 x 32 through its own ring of QS_NBUF staging boxes,
    // with its own named barrier and bulk group, so each half keeps QS_NBUF
    // reduce-adds in flight.  Rows past n are clipped by the tensor map; a
    // half that lies wholly past n adds nothing.
    asm volatile("setmaxnreg.inc.sync.aligned.u32 176;");
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int half = q >> 1, hr = r - 64 * half;
    const bool lead = (lane == 0) && (q & 1) == 0;
    const uint32_t src = tmem + ((uint32_t)(q * 32) << 16) + C::DP_COL;
    uint8_t* ring = smem + C::QS_OFF + half * (C::QS_NBUF * C::QS_BOX);
    int slot = 0;
    bool go = true;
    for (int gi = 0, u = 0; go && gi < gper; ++gi) {
      const int bq = qbase + gi;
      for (int ut = 0; ut < cnt; ++ut, ++u) {
        // both warps of the half take the same branch: they meet at named
        // barriers below, which have no time limit
        const bool ok = mbar_wait(bar(B_DQF), u & 1, abort_flag, ctl, SITE_BWD_DQ_FULL);
        if (!named_bar_and(1 + half, 64, ok)) {
          go = false;
          break;
        }
        tc_fence_after();
        uint32_t v[D / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(src + 32 * c, v[c]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(bar(B_DQE));        // the dP^T columns may be refilled now
        const int row0 = qtile(ut) * C::BM + 64 * half;
        if (row0 >= n) continue;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint8_t* stage = ring + slot * C::QS_BOX;
          slot = (slot + 1 == C::QS_NBUF) ? 0 : slot + 1;
          if (lead) bulk_wait_read<C::QS_NBUF - 1>();   // this box's last reduce-add has read it
          named_bar_sync(1 + half, 64);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(stage + sw128_offset(hr, j)) =
                make_float4(scale * __uint_as_float(v[c][4 * j]), scale * __uint_as_float(v[c][4 * j + 1]),
                            scale * __uint_as_float(v[c][4 * j + 2]), scale * __uint_as_float(v[c][4 * j + 3]));
          fence_proxy_async_smem();
          named_bar_sync(1 + half, 64);
          if (lead) {
            tma_reduce_add_3d(&tmdQ, smem_u32(stage), 32 * c, row0, bq);
            bulk_commit_group();
          }
        }
      }
    }
    // The staging buffers must be read before the CTA exits; the reduce-adds
    // themselves complete on their own (the kernel's end orders them before
    // any later work), so the next CTA on this SM starts while they drain.
    if (lead) bulk_wait_read_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc<512>(tmem);
}

template <int DH, bool DQ, bool GROUPED, bool SPARSE, int KR = 128>
int launch_kv(const void* Q, const void* K, const void* V, const void* dO, const float* LSE2,
             const float* Dv, float* dQacc, void* dK, void* dV, float* dKacc, float* dVacc,
             int BH, const HeadMap& hm, int gsplit, const TileLists& tl, int n, int n_pad,
             float scale, int causal, const KernelCtl& ctl, cudaStream_t st) {
  using C = KvCfgT<DH>;
  const int BHkv = BH / hm.group;
  CUtensorMap tq, tk, tv, tg, tdq;
  if (!make_tmap_bf16(&tq, Q, DH, n, BH, 64, C::BM) ||
      !make_tmap_bf16(&tk, K, DH, n, BHkv, 64, C::BNK) ||
      !make_tmap_bf16(&tv, V, DH, n, BHkv, 64, C::BNK) ||
      !make_tmap_bf16(&tg, dO, DH, n, BH, 64, C::BM))
    return ATTN_ERR_CUDA;
  if (DQ) {
    if (!make_tmap_f32(&tdq, dQacc, DH, n, BH, 32, C::BM / 2, true)) return ATTN_ERR_CUDA;
  } else {
    tdq = tq;   // not read
  }
  auto kern = bwd_kv128_kernel<DH, DQ, GROUPED, SPARSE, KR>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  const int nkt = ceil_div(n, KR);
  dim3 grid = (causal || SPARSE) ? dim3(BHkv * gsplit, nkt) : dim3(nkt, BHkv * gsplit);
  kern<<<grid, DQ ? 512 : 384, C::SMEM, st>>>(tq, tk, tv, tg, tdq, LSE2, Dv, dQacc,
                                              static_cast<__nv_bfloat16*>(dK),
                                              static_cast<__nv_bfloat16*>(dV), dKacc, dVacc, hm,
                                              gsplit, tl, n, n_pad, scale,
                                              scale * 1.4426950408889634f, causal, ctl);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace
}  // namespace attn

// Dispatch over the dQ mode, grouped and block-sparse instances of head dim DH.
#define ATTN_KV_DISPATCH(DH)                                                                     \
  do {                                                                                           \
    if (tl.lists) { /* block-sparse: one key/value head per query head */                        \
      if (hm.group > 1) return ATTN_ERR_UNSUPPORTED;                                             \
      if (dQacc) return ATTN_KV_LAUNCH(DH, true, false, true);                                   \
      return ATTN_KV_LAUNCH(DH, false, false, true);                                             \
    }                                                                                            \
    if (hm.group > 1) {                                                                          \
      if (dQacc) return ATTN_KV_LAUNCH(DH, true, true, false);                                   \
      return ATTN_KV_LAUNCH(DH, false, true, false);                                             \
    }                                                                                            \
    if (dQacc) return ATTN_KV_LAUNCH(DH, true, false, false);                                    \
    return ATTN_KV_LAUNCH(DH, false, false, false);                                              \
  } while (0)
#define ATTN_KV_LAUNCH(DH, DQQ, GRP, SPR)                                                        \
  launch_kv<DH, DQQ, GRP, SPR>(Q, K, V, dO, LSE2, Dv, dQacc, dK, dV, dKacc, dVacc, BH, hm, gsplit, \
                               tl, n, n_pad, scale, causal, ctl, st)
