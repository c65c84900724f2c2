// bwd_tc.cu -- fused exact attention backward on the tcgen05 tensor cores.
//
// The backward pass never stores P: it recomputes it tile by tile from the
// saved logsumexp ("Chapter 3.1 -- The cost of attention", section 5;
// "Flash Attention: Revolutionizing Transformer Efficiency", key idea 2,
// recomputation), with P_ij = 2^(s_ij * scale * log2e - LSE2_i) and
// LSE2 = LSE * log2e, and the exact chain rule
//   dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = scale dS K,
//   dK = scale dS^T Q,   D_i = dO_i . O_i (from the preprocessing kernel).
//
// bwd_kv_kernel -- the key-tile kernel at d = 256 (d = 64 and 128 use the
// pipelined key-tile kernel of bwd_kv.cuh).  dV and dK of a 128-key tile
// would fill the 512 TMEM columns, so two neighbouring CTAs share each key
// tile.  Everything is transposed so that the key index lands on the TMEM
// lanes, and K, the A operand of S^T and constant for the CTA, is copied
// once into tensor memory (which leaves shared memory for three Q and two
// dO slots):
//   both CTAs  S^T  = K Q_i^T    (TS-MMA, M = 128 keys, N = 64 queries)
//              P^T  = 2^(S^T * c - LSE2)
//   dV CTA     dV  += P^T dO_i   (TS-MMA: P^T in bf16 over S^T)
//   dK CTA     dP^T = V dO_i^T   (SS-MMA)
//              dS^T = P^T o (dP^T - D)   -> bf16 over dP^T
//              dK  += dS^T Q_i   (TS-MMA)
// Neither CTA lets its tensor pipe wait for the compute warps of a tile:
// the dV CTA, which has no dP^T, alternates S^T between two column slots and
// issues S^T(i+1) before dV(i); the dK CTA issues S^T(i+1) as soon as its
// compute warps hold P(i) in registers, so the pipe runs dP^T(i), S^T(i+1),
// dK(i) back to back while they form dS^T(i).
// In the dQ mode "spill" the dK CTA also stores its dS^T rows into the
// workspace and dQ = scale dS K is then one GEMM; otherwise dQ comes from
// bwd_q_kernel.
//
// bwd_q_kernel -- one CTA per 128-query tile: S = Q K_j^T, dP = dO V_j^T,
// dS = P o (dP - D) -> bf16 TMEM, dQ += dS K_j (TS-MMA); no atomics.  The dQ
// pass of every head dim (ATTN_DQ_PASS, and at d = 256 wherever the spill mode
// does not apply); at d = 256 Q sits in TMEM as the A operand of S.
#include <cuda_bf16.h>

#include <cstring>

#include "kernels.h"
#include "sm100.cuh"

namespace attn {
namespace {

using namespace sm100;

__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const uint32_t (&r)[32], float mul) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i)
    pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * mul, __uint_as_float(r[2 * i + 1]) * mul);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    reinterpret_cast<uint4*>(dst)[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
}

// ============================================================================ key-tile kernel
template <int D>
struct KvCfg {
  static constexpr int BNK = 128;                    // keys per CTA (TMEM lanes)
  static constexpr int BM = 64;                      // queries per iteration
  static constexpr int DO = D;                       // accumulator columns (all of d)
  // dV and dK of a key tile would take all 512 TMEM columns, so two CTAs
  // share a key tile, one accumulating dV (needs S only) and one dK (needs S
  // and dP); each recomputes S, only the dK CTA computes dP
  static constexpr int NOUT = 2;                     // CTAs per key tile
  // Q and dO tiles in separate rings, each slot released by its last reader:
  // the dK CTA reads Q(i) until dK(i) and dO(i) until dP^T(i), the dV CTA
  // Q(i) until S^T(i) and dO(i) until dV(i).  Three Q slots give the load of
  // Q(i+1) a whole iteration in the dK CTA, where S^T(i+1) runs before dK(i).
  static constexpr int QSL = 3;
  static constexpr int OSL = 2;
  static constexpr int NKB = D / 64;
  static constexpr uint32_t KV_BYTES = BNK * D * 2;
  static constexpr uint32_t QT_BYTES = BM * D * 2;   // one Q or dO tile
  static constexpr uint32_t STAT_BYTES = BM * 4;     // LSE2 or D of the tile
  static constexpr uint32_t V_OFF = 0;
  static constexpr uint32_t QS_OFF = KV_BYTES;                       // Q slots
  static constexpr uint32_t OS_OFF = QS_OFF + QSL * QT_BYTES;        // dO slots
  // the row statistics travel with the slot their last reader releases:
  // LSE2 and D with Q in the dK CTA, LSE2 with dO in the dV CTA
  static constexpr uint32_t QST_OFF = OS_OFF + OSL * QT_BYTES;
  static constexpr uint32_t OST_OFF = QST_OFF + QSL * 2 * STAT_BYTES;
  static constexpr uint32_t BAR_OFF = OST_OFF + OSL * STAT_BYTES;
  static constexpr uint32_t SMEM = BAR_OFF + 256;    // base must be 1024-byte aligned
  // K (the A operand of S^T = K Q^T, constant for the CTA) is copied into
  // tensor memory; its load lands in Q slots 1 and 2 of the dK CTA (which
  // holds V) and in the unused V area of the dV CTA
  static constexpr uint32_t K_LOAD_DK = QS_OFF + QT_BYTES;
  // TMEM columns: the CTA's one accumulator, S^T, dP^T (the dV CTA's second
  // S^T slot), K
  static constexpr int ACC_COL = 0;
  static constexpr int S_COL = DO;
  static constexpr int DP_COL = S_COL + BM;
  static constexpr int K_COL = S_COL + 2 * BM;
  static constexpr int NTHREADS = 384;
  static_assert(D == 256, "head dims 64 and 128 use the key-tile kernel of bwd_kv.cuh");
  static_assert(K_COL + D / 2 <= 512, "tensor memory budget");
  static_assert(2 * QT_BYTES == KV_BYTES, "K's load fills Q slots 1 and 2");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// Barriers (every waiter waits on consecutive phases from phase 0, and the
// phase after the one it waits for cannot complete before its own next
// action):
//   K_KV        K (and, in the dK CTA, V) loaded;  K_CP  K copied into TMEM
//   K_QF/K_OF   Q / dO slot full (TMA, with the slot's row statistics)
//   K_QE        dK CTA: Q slot free (committed after dK)
//   K_PR        dV CTA: P^T in TMEM (one per Q slot, which it also frees)
//   K_OE        dO slot free: dV CTA after dV; dK CTA in the dQ mode "spill"
//               after the dS^T staged there has been stored
//   K_SF/K_SF1  S^T slot full (the dK CTA uses K_SF only)
//   K_SC        dK CTA: the compute warps hold P in registers (S^T slot free)
//   K_DPF       dK CTA: dP^T full (one per dO slot; in the pass mode it also
//               frees the slot)
//   K_DSR       dK CTA: dS^T in TMEM
//   K_DSS       spill: dS^T staged in the dO slot for the TMA store
//   K_ACC/K_DRAIN  all MMAs done (epilogue / abort drain)
enum : int { K_KV = 0, K_QF = 1, K_QE = 4, K_OF = 7, K_OE = 9, K_SF = 11, K_SF1 = 12, K_DPF = 13,
             K_PR = 15, K_SC = 18, K_DSR = 19, K_ACC = 20, K_DRAIN = 21, K_CP = 22, K_DSS = 23 };

// GROUPED: query heads share key/value heads (compiled separately so that the
// one-head-per-head kernel keeps its simple loops).  SPARSE: the CTA walks
// the listed query tiles of a block pattern instead of the dense range.
// KR < 128 (IO study only): the CTA owns the first KR keys of its 128-key
// tile, key tiles start KR keys apart, and the other keys' probabilities are
// set to 0 (less K and V kept on chip, Q and dO streamed 128 / KR times as
// often).
template <int D, bool GROUPED, bool SPARSE, int KR = 128>
__global__ void __launch_bounds__(KvCfg<D>::NTHREADS, 1)
bwd_kv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
              const float* __restrict__ LSE2, const float* __restrict__ Dv,
              __nv_bfloat16* __restrict__ dK,
              __nv_bfloat16* __restrict__ dV, float* __restrict__ dKacc,
              float* __restrict__ dVacc, HeadMap hm, int gsplit, TileLists tl, int n, int n_pad,
              float scale, float scale_log2, int causal, KernelCtl ctl,
              const __grid_constant__ CUtensorMap tmS, int spill_ds) {
  using C = KvCfg<D>;
  static_assert(KR == C::BNK || (KR >= 32 && KR < C::BNK && !SPARSE && !GROUPED),
                "owned key rows: a dense, one-head-per-head study instance");
  extern __shared__ uint8_t smem_raw[];
  // the layout has no room to align itself: it needs the base 1024-byte
  // aligned (the 128-byte swizzle atoms); report and leave before touching
  // anything
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_error(ctl, ATTN_ERR_CUDA, SITE_BWD_SMEM_ALIGN);
    return;
  }
  uint8_t* smem = smem_raw;
  const uint32_t sb = smem_u32(smem);
  const uint32_t bars = sb + C::BAR_OFF;
  auto bar = [&](int i) { return bars + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::BAR_OFF + 240);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + 248);

  const int warp = warp_id_uniform(), lane = threadIdx.x & 31;
  // Causal or block-sparse (tiles of unequal length): heads vary fastest in
  // the grid and tiles slowest, longest first, so the long tiles of every
  // head start early instead of the last heads' long tiles trailing the rest
  // (CTAs start in grid order).  Otherwise tiles vary fastest, which keeps a
  // head's K and V shared in L2 by CTAs that run together.
  // The two CTAs of a key tile are neighbours in the grid: the output index
  // is the fastest part of grid.x, and grid.y stays at most the head count
  // (the grid's y limit).
  const bool heads_fast = causal || SPARSE;
  const int kt = heads_fast ? (int)blockIdx.y : (int)blockIdx.x / C::NOUT;
  const int oh = (int)blockIdx.x % C::NOUT;      // 0 accumulates dV, 1 dK
  const int bh = heads_fast ? (int)blockIdx.x / C::NOUT : (int)blockIdx.y;   // key/value head
  const int part = (int)blockIdx.z;              // part of the group (gsplit > 1)
  const bool want_dk = oh == 1, want_dv = !want_dk;
  const int k0 = kt * KR;
  const int nq = (n + C::BM - 1) / C::BM;
  const int i_start = causal ? (k0 / C::BM) : 0;
  const int* qlist = SPARSE ? tl.lists + (size_t)kt * tl.stride : nullptr;
  const int cnt = SPARSE ? tl.counts[kt] : nq - i_start;   // query tiles per query head
  auto qtile = [&](int ut) { return SPARSE ? (qlist[ut] & 0xFFFF) : i_start + ut; };
  // The query heads of this key/value head's group are split over gsplit
  // CTAs; iteration u visits query tile i_start + u % cnt of query head
  // qbase + u / cnt, so dK and dV accumulate over this CTA's part of the
  // group.  Each role runs an outer loop over its heads and an inner loop
  // over the query tiles.
  const int gper = GROUPED ? hm.group / gsplit : 1;
  const int qbase = GROUPED ? hm.q_of(bh, part * gper) : bh;
  const int total = gper * cnt;
  const uint32_t k_load = want_dk ? C::K_LOAD_DK : C::V_OFF;
  // dQ mode "spill": the dK CTA also writes dS^T ([BH][n keys][n queries]
  // through tmS) for dQ = scale dS K as one GEMM.  Its compute warps stage
  // each tile's dS^T in the dO slot that dP^T has just consumed, and warp 3
  // stores it with TMA and then releases the slot.
  const bool spill = !GROUPED && !SPARSE && KR == C::BNK && spill_ds != 0 && want_dk;
  // S^T of iteration u, its columns and its barriers.  The dK CTA keeps one
  // slot (its dP^T columns receive dS^T); the dV CTA has no dP^T, so its S^T
  // alternates between the S^T and the dP^T columns, with a "full" and a
  // "P ready" barrier per slot (each waited with the parity of u / 2).
  auto s_col = [&](int u) { return (want_dk || !(u & 1)) ? C::S_COL : C::DP_COL; };
  auto sf_bar = [&](int u) { return (want_dk || !(u & 1)) ? bar(K_SF) : bar(K_SF1); };
  auto sf_par = [&](int u) { return want_dk ? (u & 1) : ((u >> 1) & 1); };
  auto pr_bar = [&](int u) { return bar(K_PR + u % C::QSL); };

  if (threadIdx.x == 0) {
    mbar_init(bar(K_KV), 1);
    for (int s = 0; s < C::QSL; ++s) {
      mbar_init(bar(K_QF + s), 1);
      mbar_init(bar(K_QE + s), 1);
    }
    for (int s = 0; s < C::OSL; ++s) {
      mbar_init(bar(K_OF + s), 1);
      mbar_init(bar(K_OE + s), 1);
      mbar_init(bar(K_DSS + s), 256);
    }
    mbar_init(bar(K_SF), 1);
    mbar_init(bar(K_SF1), 1);
    for (int s = 0; s < C::OSL; ++s) mbar_init(bar(K_DPF + s), 1);
    for (int s = 0; s < C::QSL; ++s) mbar_init(bar(K_PR + s), 256);
    mbar_init(bar(K_SC), 256);
    mbar_init(bar(K_DSR), 256);
    mbar_init(bar(K_ACC), 1);
    mbar_init(bar(K_DRAIN), 1);
    mbar_init(bar(K_CP), 128);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    if (spill) tma_prefetch_desc(&tmS);
  }
  if (warp == 2) tmem_alloc<512>(smem_u32(tmem_slot));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------ K, V and Q producer
      mbar_expect_tx(bar(K_KV), (want_dk ? 2 : 1) * C::KV_BYTES);   // V only for dP
#pragma unroll
      for (int kb = 0; kb < C::NKB; ++kb) {
        tma_load_3d(sb + k_load + kb * (C::BNK * 128), &tmK, kb * 64, k0, bh, bar(K_KV));
        if (want_dk)
          tma_load_3d(sb + C::V_OFF + kb * (C::BNK * 128), &tmV, kb * 64, k0, bh, bar(K_KV));
      }
      // Q (with LSE2 and D in the dK CTA); dO has its own producer (warp 2)
      int q_last[C::QSL];
      for (int s = 0; s < C::QSL; ++s) q_last[s] = -1;
      bool go = true;
      for (int gi = 0, u = 0; go && gi < gper; ++gi) {
        const int bq = qbase + gi;
        for (int ut = 0; ut < cnt; ++ut, ++u) {
          const int qs = u % C::QSL;
          const int q0 = qtile(ut) * C::BM;
          // the slot's previous tile is done: after dK in the dK CTA, after
          // the compute warps read S^T ("P ready") in the dV CTA
          if (!mbar_wait(want_dk ? bar(K_QE + qs) : pr_bar(u), ((u / C::QSL) & 1) ^ 1, abort_flag, ctl,
                         SITE_BWD_Q_EMPTY)) {
            go = false;
            break;
          }
          // Q slots 1 and 2 of the dK CTA hold K until it has been copied to tensor memory
          if (want_dk && u == 1 && !mbar_wait(bar(K_CP), 0, abort_flag, ctl, SITE_BWD_KV)) {
            go = false;
            break;
          }
          const uint32_t qd = sb + C::QS_OFF + qs * C::QT_BYTES;
          mbar_expect_tx(bar(K_QF + qs), C::QT_BYTES + (want_dk ? 2 * C::STAT_BYTES : 0));
#pragma unroll
          for (int kb = 0; kb < C::NKB; ++kb)
            tma_load_3d(qd + kb * (C::BM * 128), &tmQ, kb * 64, q0, bq, bar(K_QF + qs));
          if (want_dk) {
            const uint32_t stq = sb + C::QST_OFF + qs * 2 * C::STAT_BYTES;
            bulk_load(stq, LSE2 + (size_t)bq * n_pad + q0, C::STAT_BYTES, bar(K_QF + qs));
            bulk_load(stq + C::STAT_BYTES, Dv + (size_t)bq * n_pad + q0, C::STAT_BYTES,
                      bar(K_QF + qs));
          }
          q_last[qs] = u;
        }
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        mbar_wait(bar(K_KV), 0, &no_abort, ctl, SITE_BWD_KV);
        for (int s = 0; s < C::QSL; ++s)
          if (q_last[s] >= 0)
            mbar_wait(bar(K_QF + s), (q_last[s] / C::QSL) & 1, &no_abort, ctl, SITE_BWD_Q_FULL);
      }
    } else if (warp == 2 && lane == 0) {
      // ------------------------------------------------------------ dO producer
      // (with LSE2 in the dV CTA)
      int o_last[C::OSL];
      for (int s = 0; s < C::OSL; ++s) o_last[s] = -1;
      bool go = true;
      for (int gi = 0, u = 0; go && gi < gper; ++gi) {
        const int bq = qbase + gi;
        for (int ut = 0; ut < cnt; ++ut, ++u) {
          const int os = u % C::OSL;
          const int q0 = qtile(ut) * C::BM;
          // the slot's previous tile is done: after dP^T in the dK CTA (after
          // its dS^T store in the spill mode), after dV in the dV CTA
          const uint32_t free_bar = (want_dk && !spill) ? bar(K_DPF + os) : bar(K_OE + os);
          if (!mbar_wait(free_bar, ((u / C::OSL) & 1) ^ 1, abort_flag, ctl, SITE_BWD_Q_EMPTY)) {
            go = false;
            break;
          }
          const uint32_t od = sb + C::OS_OFF + os * C::QT_BYTES;
          mbar_expect_tx(bar(K_OF + os), C::QT_BYTES + (want_dv ? C::STAT_BYTES : 0));
#pragma unroll
          for (int kb = 0; kb < C::NKB; ++kb)
            tma_load_3d(od + kb * (C::BM * 128), &tmdO, kb * 64, q0, bq, bar(K_OF + os));
          if (want_dv)
            bulk_load(sb + C::OST_OFF + os * C::STAT_BYTES, LSE2 + (size_t)bq * n_pad + q0,
                      C::STAT_BYTES, bar(K_OF + os));
          o_last[os] = u;
        }
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        for (int s = 0; s < C::OSL; ++s)
          if (o_last[s] >= 0)
            mbar_wait(bar(K_OF + s), (o_last[s] / C::OSL) & 1, &no_abort, ctl, SITE_BWD_Q_FULL);
      }
    } else if (warp == 3 && lane == 0) {
      // ------------------------------------------------------------ dS^T store (spill)
      if (spill) {
        for (int u = 0; u < total; ++u) {   // one query head (no group, no tile list)
          const int os = u % C::OSL;
          if (!mbar_wait(bar(K_DSS + os), (u / C::OSL) & 1, abort_flag, ctl, SITE_BWD_DS_READY))
            break;
          tma_store_3d(&tmS, sb + C::OS_OFF + os * C::QT_BYTES, qtile(u) * C::BM, k0, bh);
          bulk_commit_group();
          bulk_wait_read_all();   // the slot has been read: dO(u + 2) may load
          mbar_arrive(bar(K_OE + os));
        }
        bulk_wait_all();
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // (the whole warp runs the loop; one elected lane issues each MMA/commit)
      constexpr uint32_t id_s = idesc_bf16(128, C::BM, false, false);   // K/V K-major, Q/dO K-major
      constexpr uint32_t id_acc = idesc_bf16(128, C::DO, false, true);  // P^T/dS^T TMEM, dO/Q MN-major
      bool ok = mbar_wait_warp(bar(K_KV), 0, abort_flag, ctl, SITE_BWD_KV);
      ok = ok && mbar_wait_warp(bar(K_CP), 0, abort_flag, ctl, SITE_BWD_KV);
      // MMAs in groups of four from one asm block, with the shared-memory
      // descriptors' low halves precomputed (the MMA queue is shallow, so
      // scalar work between MMAs costs tensor time)
      constexpr uint32_t HI = sdesc_hi(1024);
      constexpr uint32_t QT16 = C::QT_BYTES >> 4;
      const uint32_t v_km = sdesc_lo(sb + C::V_OFF, 16);                // V, K-major
      const uint32_t q_km = sdesc_lo(sb + C::QS_OFF, 16);               // Q slot 0, K-major
      const uint32_t q_mn = sdesc_lo(sb + C::QS_OFF, C::BM * 128);      // Q slot 0, MN-major
      const uint32_t g_km = sdesc_lo(sb + C::OS_OFF, 16);               // dO slot 0, K-major
      const uint32_t g_mn = sdesc_lo(sb + C::OS_OFF, C::BM * 128);      // dO slot 0, MN-major
      // K-major operand, 64-wide column box b of a tile with `rows` rows
      auto km4 = [](uint32_t base, int rows, int b, uint32_t (&lo)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) lo[i] = base + b * (rows * 128 / 16) + 2 * i;
      };
      // MN-major operand, K slices 0..3 (16 rows = 2048 bytes each)
      auto mn4 = [](uint32_t base, uint32_t (&lo)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) lo[i] = base + i * (2048 / 16);
      };
      // S^T(u) = K Q_u^T into column col: A = K from tensor memory (16
      // elements = 8 columns per MMA), contraction over d
      auto issue_s = [&](int u, int col) {
        const uint32_t qb = q_km + (u % C::QSL) * QT16;
#pragma unroll
        for (int b = 0; b < C::NKB; ++b) {
          uint32_t blo[4];
          km4(qb, C::BM, b, blo);
          mma_ts_x4(tmem + col, tmem + C::K_COL + 32 * b, blo, HI, id_s, b > 0);
        }
      };
      // S^T of the next tile is issued before this tile's accumulator
      // product: in the dV CTA into the other slot, in the dK CTA as soon as
      // the compute warps hold P in registers (K_SC), so that it runs while
      // they form dS^T.
      if (ok && total > 0) {
        ok = mbar_wait_warp(bar(K_QF), 0, abort_flag, ctl, SITE_BWD_Q_FULL);
        if (ok) {
          tc_fence_after();
          issue_s(0, s_col(0));
          tc_commit(sf_bar(0));
        }
      }
      for (int u = 0; ok && u < total; ++u) {
        const int qs = u % C::QSL, os = u % C::OSL;
        const int qn = (u + 1) % C::QSL, pn = ((u + 1) / C::QSL) & 1;
        const bool more = u + 1 < total;
        if (want_dk) {
          // dP^T = V dO^T; dO is then free
          if (!(ok = mbar_wait_warp(bar(K_OF + os), (u / C::OSL) & 1, abort_flag, ctl, SITE_BWD_Q_FULL)))
            break;
          tc_fence_after();
#pragma unroll
          for (int b = 0; b < C::NKB; ++b) {
            uint32_t alo[4], blo[4];
            km4(v_km, C::BNK, b, alo);
            km4(g_km + os * QT16, C::BM, b, blo);
            mma_ss_x4(tmem + C::DP_COL, alo, HI, blo, HI, id_s, b > 0);
          }
          tc_commit(bar(K_DPF + os));   // also frees the dO slot (spill: after the dS^T store)
          if (more) {
            if (!(ok = mbar_wait_warp(bar(K_SC), u & 1, abort_flag, ctl, SITE_BWD_S_READ))) break;
            if (!(ok = mbar_wait_warp(bar(K_QF + qn), pn, abort_flag, ctl, SITE_BWD_Q_FULL))) break;
            tc_fence_after();
            issue_s(u + 1, C::S_COL);
            tc_commit(bar(K_SF));
          }
          // dK += dS^T Q; Q is then free
          if (!(ok = mbar_wait_warp(bar(K_DSR), u & 1, abort_flag, ctl, SITE_BWD_DS_READY))) break;
          tc_fence_after();
          {   // dS^T half h (queries [32h, 32h+32)) at columns [32h, 32h+16)
            uint32_t blo[4];
            mn4(q_mn + qs * QT16, blo);
            mma_ts_x4_halves<C::BM / 2>(tmem + C::ACC_COL, tmem + C::DP_COL, blo, HI, id_acc, u > 0);
          }
          tc_commit(bar(K_QE + qs));
        } else {
          // dO(u) (loaded long before) is waited for ahead of S^T(u+1), so
          // that only "P ready" stands between S^T(u+1) and dV(u)
          if (!(ok = mbar_wait_warp(bar(K_OF + os), (u / C::OSL) & 1, abort_flag, ctl, SITE_BWD_Q_FULL)))
            break;
          if (more) {
            if (!(ok = mbar_wait_warp(bar(K_QF + qn), pn, abort_flag, ctl, SITE_BWD_Q_FULL))) break;
            tc_fence_after();
            issue_s(u + 1, s_col(u + 1));
            tc_commit(sf_bar(u + 1));
          }
          // dV += P^T dO  (contraction over the BM queries of this tile); dO is then free
          if (!(ok = mbar_wait_warp(pr_bar(u), (u / C::QSL) & 1, abort_flag, ctl, SITE_BWD_P_READY)))
            break;
          tc_fence_after();
          {   // P^T half h (queries [32h, 32h+32)) at columns [32h, 32h+16) of the slot
            uint32_t blo[4];
            mn4(g_mn + os * QT16, blo);
            mma_ts_x4_halves<C::BM / 2>(tmem + C::ACC_COL, tmem + s_col(u), blo, HI, id_acc, u > 0);
          }
          tc_commit(bar(K_OE + os));
        }
      }
      tc_commit(bar(K_ACC));
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        tc_commit(bar(K_DRAIN));
        volatile int no_abort = 0;
        mbar_wait_warp(bar(K_DRAIN), 0, &no_abort, ctl, SITE_BWD_ACC_DONE);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- compute
    const int q = warp & 3, h = (warp - 4) >> 2;
    const int r = q * 32 + lane;          // key row within the tile (TMEM lane)
    const int key = k0 + r;
    constexpr int NC = C::BM / 2;         // query columns of this thread
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint32_t dp_addr = tmem + lane_off + C::DP_COL + h * NC;
    bool ok = true;
    if (h == 0) {   // first warpgroup: K rows into tensor memory
      ok = mbar_wait(bar(K_KV), 0, abort_flag, ctl, SITE_BWD_KV);
      if (__all_sync(0xffffffffu, ok)) {
        tile_to_tmem<D>(smem + k_load, tmem + lane_off + C::K_COL, r);
        tc_fence_before();
        mbar_arrive(bar(K_CP));
      } else {
        ok = false;
      }
    }
    for (int gi = 0, u = 0; ok && gi < gper; ++gi) {
      for (int ut = 0; ut < cnt; ++ut, ++u) {
        const int qs = u % C::QSL, os = u % C::OSL;
        const int q0 = qtile(ut) * C::BM;
        const uint32_t s_addr = tmem + lane_off + s_col(u) + h * NC;
        // LSE2 (and D): with Q in the dK CTA, with dO in the dV CTA
        const float* lse2;
        if (want_dk) {
          lse2 = reinterpret_cast<const float*>(smem + C::QST_OFF + qs * 2 * C::STAT_BYTES) + h * NC;
          ok = mbar_wait(bar(K_QF + qs), (u / C::QSL) & 1, abort_flag, ctl, SITE_BWD_Q_FULL);
        } else {
          lse2 = reinterpret_cast<const float*>(smem + C::OST_OFF + os * C::STAT_BYTES) + h * NC;
          ok = mbar_wait(bar(K_OF + os), (u / C::OSL) & 1, abort_flag, ctl, SITE_BWD_Q_FULL);
        }
        const float* dd = lse2 + C::BM;
        ok = ok && mbar_wait(sf_bar(u), sf_par(u), abort_flag, ctl, SITE_BWD_S_FULL);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const bool masked = causal && (k0 + C::BNK - 1 > q0);
        const int qbase = q0 + h * NC;     // first query column of this thread
        float p[NC];
#pragma unroll
        for (int c0 = 0; c0 < NC; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(s_addr + c0, rr);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float v = ex2(fmaf(__uint_as_float(rr[i]), scale_log2, -lse2[c0 + i]));
            if (masked && key > qbase + c0 + i) v = 0.f;
            p[c0 + i] = v;
          }
        }
        if (want_dk) {   // S^T has been read: its columns take the next tile's S^T
          tc_fence_before();
          mbar_arrive(bar(K_SC));
        }
        if constexpr (KR < C::BNK) {   // keys of the next study tile: no contribution
          if (r >= KR) {
#pragma unroll
            for (int c = 0; c < NC; ++c) p[c] = 0.f;
          }
        }
        if (want_dv) {   // P^T in bf16 over S^T: the A operand of dV
#pragma unroll
          for (int c0 = 0; c0 < NC; c0 += 32) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(p[c0 + 2 * i], p[c0 + 2 * i + 1]);
            tmem_st16(s_addr + c0 / 2, pk);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(pr_bar(u));
          continue;   // the dV CTA forms no dP, no dS
        }
        ok = mbar_wait(bar(K_DPF + os), (u / C::OSL) & 1, abort_flag, ctl, SITE_BWD_DP_FULL);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        uint32_t ds[NC / 2];
#pragma unroll
        for (int c0 = 0; c0 < NC; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(dp_addr + c0, rr);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a = p[c0 + 2 * i] * (__uint_as_float(rr[2 * i]) - dd[c0 + 2 * i]);
            const float b = p[c0 + 2 * i + 1] * (__uint_as_float(rr[2 * i + 1]) - dd[c0 + 2 * i + 1]);
            ds[c0 / 2 + i] = pack_bf16x2(a, b);
          }
        }
#pragma unroll
        for (int c0 = 0; c0 < NC / 2; c0 += 16) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = ds[c0 + i];
          tmem_st16(dp_addr + c0, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(K_DSR));
        if (spill) {
          // dS^T rows of queries [h NC, h NC + NC) into the consumed dO slot
          // as one 128-byte-swizzled [128 keys][64 queries] box
          uint8_t* stg = smem + C::OS_OFF + os * C::QT_BYTES;
#pragma unroll
          for (int j = 0; j < NC / 8; ++j)
            *reinterpret_cast<uint4*>(stg + sw128_offset(r, h * (NC / 8) + j)) =
                make_uint4(ds[4 * j], ds[4 * j + 1], ds[4 * j + 2], ds[4 * j + 3]);
          fence_proxy_async_smem();
          mbar_arrive(bar(K_DSS + os));
        }
      }
    }
    // ---- epilogue: warpgroup h writes columns [h d/2, (h+1) d/2) of this
    // CTA's output (dK scaled)
    if (ok) {
      ok = mbar_wait(bar(K_ACC), 0, abort_flag, ctl, SITE_BWD_ACC_DONE);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      constexpr int W = D / 2;   // columns of this warpgroup
      const int c_first = h * W;
      const uint32_t src = tmem + lane_off + C::ACC_COL + c_first;
      const size_t off = ((size_t)bh * n + key) * D + c_first;
      const float mul = want_dv ? 1.f : scale;
      float* acc = GROUPED ? (want_dv ? dVacc : dKacc) : nullptr;   // set when the group is split
#pragma unroll 1
      for (int c0 = 0; c0 < W; c0 += 32) {
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
              red_add_v4(acc + off + c0 + i, mul * __uint_as_float(rr[i]),
                         mul * __uint_as_float(rr[i + 1]), mul * __uint_as_float(rr[i + 2]),
                         mul * __uint_as_float(rr[i + 3]));
          } else {
            store32_bf16((want_dv ? dV : dK) + off + c0, rr, mul);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc<512>(tmem);
}

// ============================================================================ query-tile kernel
template <int D>
struct QCfg {
  static constexpr int BM = 128;                     // queries per CTA (TMEM lanes)
  static constexpr int BN = (D == 256) ? 64 : 128;   // keys per iteration
  // K_j and V_j in separate rings, each slot released by its last reader
  // (K_j after dQ(j), V_j after dP(j)); three K slots give the load of
  // K_{j+1} a whole iteration, since S(j+1) is issued before dQ(j)
  static constexpr int KSL = 3;
  static constexpr int VSL = 2;
  // d = 256: Q (the A operand of S = Q K^T, constant for the CTA) lives in
  // tensor memory, which frees the shared memory of the rings
  static constexpr bool Q_IN_TMEM = (D == 256);
  static constexpr int NKB = D / 64;
  static constexpr uint32_t QT_BYTES = BM * D * 2;
  static constexpr uint32_t KV_BYTES = BN * D * 2;
  static constexpr uint32_t Q_OFF = 0;                              // unused when Q_IN_TMEM
  static constexpr uint32_t G_OFF = Q_IN_TMEM ? 0 : QT_BYTES;
  static constexpr uint32_t KS_OFF = G_OFF + QT_BYTES;              // K slots
  static constexpr uint32_t VS_OFF = KS_OFF + KSL * KV_BYTES;       // V slots
  // where Q's load lands: K slots 1 and 2, before their first use
  static constexpr uint32_t Q_LOAD_OFF = Q_IN_TMEM ? KS_OFF + KV_BYTES : Q_OFF;
  static constexpr uint32_t BAR_OFF = VS_OFF + VSL * KV_BYTES;
  static constexpr uint32_t SMEM = BAR_OFF + 256;    // base must be 1024-byte aligned
  static constexpr int S_COL = 0;
  static constexpr int DP_COL = BN;                   // dP, then dS in bf16 over it
  static constexpr int DQ_COL = 2 * BN;
  static constexpr int Q_COL = 2 * BN + D;            // Q as A operand (Q_IN_TMEM)
  static constexpr int NTHREADS = 384;
  static_assert(2 * BN + D + (Q_IN_TMEM ? D / 2 : 0) <= 512, "tensor memory budget");
  static_assert(BN == 64 || BN == 128, "dS halves as the dQ product reads them");
  static_assert(!Q_IN_TMEM || QT_BYTES <= 2 * KV_BYTES, "Q's load fits in K slots 1 and 2");
  static_assert(KV_BYTES % 1024 == 0 && QT_BYTES % 1024 == 0, "slots stay 1024-byte aligned");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// Q_SC: the compute warps hold P of the current key tile in registers, so the
// S columns are free for the next tile's S.
enum : int { Q_QF = 0, Q_KF = 1, Q_KE = 4, Q_VF = 7, Q_VE = 9, Q_SF = 11, Q_DPF = 12, Q_DSR = 13,
             Q_ACC = 14, Q_DRAIN = 15, Q_CP = 16, Q_SC = 17 };

template <int D>
__global__ void __launch_bounds__(QCfg<D>::NTHREADS, 1)
bwd_q_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
             const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
             const float* __restrict__ LSE2, const float* __restrict__ Dv,
             __nv_bfloat16* __restrict__ dQ, HeadMap hm, TileLists tl, int n, int n_pad,
             float scale, float scale_log2, int causal, KernelCtl ctl) {
  using C = QCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  // no room to align the layout: it needs the base 1024-byte aligned (the
  // 128-byte swizzle atoms); report and leave before touching anything
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_error(ctl, ATTN_ERR_CUDA, SITE_BWD_SMEM_ALIGN);
    return;
  }
  uint8_t* smem = smem_raw;
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
  // head's K and V shared in L2 by CTAs that run together.
  const bool heads_fast = causal || tl.lists != nullptr;
  const int ntile = heads_fast ? gridDim.y : gridDim.x;
  const int tile_ix = heads_fast ? (int)blockIdx.y : (int)blockIdx.x;
  const int it = causal ? (ntile - 1 - tile_ix) : tile_ix;
  const int bh = heads_fast ? blockIdx.x : blockIdx.y;   // query head (Q, dO, dQ, LSE, D)
  const int bkv = hm.kv_of(bh);       // key/value head (K, V)
  const int q0 = it * C::BM;
  const int nkv = (n + C::BN - 1) / C::BN;
  const int jend = causal ? min(nkv - 1, (q0 + C::BM - 1) / C::BN) : nkv - 1;
  // block-sparse: the key tiles of this query tile's list, in place of 0..jend
  const int* klist = tl.lists ? tl.lists + (size_t)it * tl.stride : nullptr;
  const int cnt = klist ? tl.counts[it] : jend + 1;
  auto ktile = [&](int j) { return klist ? (klist[j] & 0xFFFF) : j; };

  if (threadIdx.x == 0) {
    mbar_init(bar(Q_QF), 1);
    for (int s = 0; s < C::KSL; ++s) {
      mbar_init(bar(Q_KF + s), 1);
      mbar_init(bar(Q_KE + s), 1);
    }
    for (int s = 0; s < C::VSL; ++s) {
      mbar_init(bar(Q_VF + s), 1);
      mbar_init(bar(Q_VE + s), 1);
    }
    mbar_init(bar(Q_SF), 1);
    mbar_init(bar(Q_DPF), 1);
    mbar_init(bar(Q_DSR), 256);
    mbar_init(bar(Q_SC), 256);
    mbar_init(bar(Q_ACC), 1);
    mbar_init(bar(Q_DRAIN), 1);
    mbar_init(bar(Q_CP), 128);
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
      // ------------------------------------------------------------ Q, dO and K producer
      mbar_expect_tx(bar(Q_QF), 2 * C::QT_BYTES);
#pragma unroll
      for (int kb = 0; kb < C::NKB; ++kb) {
        tma_load_3d(sb + C::Q_LOAD_OFF + kb * (C::BM * 128), &tmQ, kb * 64, q0, bh, bar(Q_QF));
        tma_load_3d(sb + C::G_OFF + kb * (C::BM * 128), &tmdO, kb * 64, q0, bh, bar(Q_QF));
      }
      int k_last[C::KSL];
      for (int s = 0; s < C::KSL; ++s) k_last[s] = -1;
      for (int j = 0; j < cnt; ++j) {
        const int s = j % C::KSL;
        if (!mbar_wait(bar(Q_KE + s), ((j / C::KSL) & 1) ^ 1, abort_flag, ctl, SITE_BWD_Q_EMPTY))
          break;
        // K slots 1 and 2 hold Q until it has been copied to tensor memory
        if (C::Q_IN_TMEM && j == 1 && !mbar_wait(bar(Q_CP), 0, abort_flag, ctl, SITE_BWD_Q_FULL))
          break;
        const uint32_t kd = sb + C::KS_OFF + s * C::KV_BYTES;
        mbar_expect_tx(bar(Q_KF + s), C::KV_BYTES);
#pragma unroll
        for (int kb = 0; kb < C::NKB; ++kb)
          tma_load_3d(kd + kb * (C::BN * 128), &tmK, kb * 64, ktile(j) * C::BN, bkv, bar(Q_KF + s));
        k_last[s] = j;
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        mbar_wait(bar(Q_QF), 0, &no_abort, ctl, SITE_BWD_Q_FULL);
        for (int s = 0; s < C::KSL; ++s)
          if (k_last[s] >= 0)
            mbar_wait(bar(Q_KF + s), (k_last[s] / C::KSL) & 1, &no_abort, ctl, SITE_BWD_KV);
      }
    } else if (warp == 2 && lane == 0) {
      // ------------------------------------------------------------ V producer
      int v_last[C::VSL];
      for (int s = 0; s < C::VSL; ++s) v_last[s] = -1;
      for (int j = 0; j < cnt; ++j) {
        const int s = j % C::VSL;
        if (!mbar_wait(bar(Q_VE + s), ((j / C::VSL) & 1) ^ 1, abort_flag, ctl, SITE_BWD_Q_EMPTY))
          break;
        const uint32_t vd = sb + C::VS_OFF + s * C::KV_BYTES;
        mbar_expect_tx(bar(Q_VF + s), C::KV_BYTES);
#pragma unroll
        for (int kb = 0; kb < C::NKB; ++kb)
          tma_load_3d(vd + kb * (C::BN * 128), &tmV, kb * 64, ktile(j) * C::BN, bkv, bar(Q_VF + s));
        v_last[s] = j;
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        for (int s = 0; s < C::VSL; ++s)
          if (v_last[s] >= 0)
            mbar_wait(bar(Q_VF + s), (v_last[s] / C::VSL) & 1, &no_abort, ctl, SITE_BWD_KV);
      }
    } else if (warp == 1) {
      // MMA issuer (the whole warp runs the loop; one elected lane issues)
      constexpr uint32_t id_s = idesc_bf16(128, C::BN, false, false);
      constexpr uint32_t id_dq = idesc_bf16(128, D, false, true);
      bool ok = mbar_wait_warp(bar(Q_QF), 0, abort_flag, ctl, SITE_BWD_Q_FULL);
      if (C::Q_IN_TMEM) ok = ok && mbar_wait_warp(bar(Q_CP), 0, abort_flag, ctl, SITE_BWD_Q_FULL);
      // MMAs in groups of four from one asm block, with the shared-memory
      // descriptors' low halves precomputed
      constexpr uint32_t HI = sdesc_hi(1024);
      constexpr uint32_t KV16 = C::KV_BYTES >> 4;
      const uint32_t q_km = sdesc_lo(sb + C::Q_OFF, 16);              // Q, K-major
      const uint32_t g_km = sdesc_lo(sb + C::G_OFF, 16);              // dO, K-major
      const uint32_t k_km = sdesc_lo(sb + C::KS_OFF, 16);             // K slot 0, K-major
      const uint32_t k_mn = sdesc_lo(sb + C::KS_OFF, C::BN * 128);    // K slot 0, MN-major
      const uint32_t v_km = sdesc_lo(sb + C::VS_OFF, 16);             // V slot 0, K-major
      auto km4 = [](uint32_t base, int rows, int b, uint32_t (&lo)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) lo[i] = base + b * (rows * 128 / 16) + 2 * i;
      };
      auto mn4 = [](uint32_t base, int g, uint32_t (&lo)[4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) lo[i] = base + (4 * g + i) * (2048 / 16);
      };
      // S = Q K_j^T into the S columns  (contraction over d, 64 per group)
      auto issue_s = [&](int j) {
        const uint32_t kb0 = k_km + (j % C::KSL) * KV16;
#pragma unroll
        for (int b = 0; b < C::NKB; ++b) {
          uint32_t blo[4];
          km4(kb0, C::BN, b, blo);
          if (C::Q_IN_TMEM) {   // A = Q from tensor memory, 16 elements = 8 columns per MMA
            mma_ts_x4(tmem + C::S_COL, tmem + C::Q_COL + 32 * b, blo, HI, id_s, b > 0);
          } else {
            uint32_t alo[4];
            km4(q_km, C::BM, b, alo);
            mma_ss_x4(tmem + C::S_COL, alo, HI, blo, HI, id_s, b > 0);
          }
        }
      };
      // dS goes over dP, so S of the next key tile is issued as soon as the
      // compute warps hold P in registers (Q_SC): the pipe runs dP(j),
      // S(j+1), dQ(j) back to back while they form dS(j).
      if (ok && cnt > 0) {
        ok = mbar_wait_warp(bar(Q_KF), 0, abort_flag, ctl, SITE_BWD_KV);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          tc_commit(bar(Q_SF));
        }
      }
      for (int j = 0; ok && j < cnt; ++j) {
        const int ks = j % C::KSL, vs = j % C::VSL;
        // dP = dO V_j^T; V_j is then free
        if (!(ok = mbar_wait_warp(bar(Q_VF + vs), (j / C::VSL) & 1, abort_flag, ctl, SITE_BWD_KV)))
          break;
        tc_fence_after();
#pragma unroll
        for (int b = 0; b < C::NKB; ++b) {
          uint32_t alo[4], blo[4];
          km4(g_km, C::BM, b, alo);
          km4(v_km + vs * KV16, C::BN, b, blo);
          mma_ss_x4(tmem + C::DP_COL, alo, HI, blo, HI, id_s, b > 0);
        }
        tc_commit(bar(Q_DPF));
        tc_commit(bar(Q_VE + vs));
        if (j + 1 < cnt) {
          if (!(ok = mbar_wait_warp(bar(Q_SC), j & 1, abort_flag, ctl, SITE_BWD_S_READ))) break;
          if (!(ok = mbar_wait_warp(bar(Q_KF + (j + 1) % C::KSL), ((j + 1) / C::KSL) & 1, abort_flag,
                                    ctl, SITE_BWD_KV)))
            break;
          tc_fence_after();
          issue_s(j + 1);
          tc_commit(bar(Q_SF));
        }
        // dQ += dS K_j: dS half h (keys [h BN/2, (h+1) BN/2)) at columns
        // [h BN/2, h BN/2 + BN/4) over dP; K_j is then free
        if (!(ok = mbar_wait_warp(bar(Q_DSR), j & 1, abort_flag, ctl, SITE_BWD_DS_READY))) break;
        tc_fence_after();
        if constexpr (C::BN == 64) {
          uint32_t blo[4];
          mn4(k_mn + ks * KV16, 0, blo);
          mma_ts_x4_halves<C::BN / 2>(tmem + C::DQ_COL, tmem + C::DP_COL, blo, HI, id_dq, j > 0);
        } else {
#pragma unroll
          for (int g = 0; g < C::BN / 64; ++g) {
            uint32_t blo[4];
            mn4(k_mn + ks * KV16, g, blo);
            mma_ts_x4(tmem + C::DQ_COL, tmem + C::DP_COL + 64 * g, blo, HI, id_dq, (j > 0 || g > 0));
          }
        }
        tc_commit(bar(Q_KE + ks));
      }
      tc_commit(bar(Q_ACC));
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        tc_commit(bar(Q_DRAIN));
        volatile int no_abort = 0;
        mbar_wait_warp(bar(Q_DRAIN), 0, &no_abort, ctl, SITE_BWD_ACC_DONE);
      }
    }
    __syncwarp();
  } else {
    const int q = warp & 3, h = (warp - 4) >> 2;
    const int r = q * 32 + lane;       // query row (TMEM lane)
    const int qrow = q0 + r;
    constexpr int NC = C::BN / 2;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + C::S_COL + h * NC;
    const uint32_t dp_addr = tmem + lane_off + C::DP_COL + h * NC;
    const float lse2 = LSE2[(size_t)bh * n_pad + qrow];   // +inf on padded rows -> P = 0
    const float dd = Dv[(size_t)bh * n_pad + qrow];
    bool ok = true;
    if (C::Q_IN_TMEM && h == 0) {   // first warpgroup: Q rows into tensor memory
      ok = mbar_wait(bar(Q_QF), 0, abort_flag, ctl, SITE_BWD_Q_FULL);
      if (__all_sync(0xffffffffu, ok)) {
        tile_to_tmem<D>(smem + C::Q_LOAD_OFF, tmem + lane_off + C::Q_COL, r);
        tc_fence_before();
        mbar_arrive(bar(Q_CP));
      } else {
        ok = false;
      }
    }
    for (int j = 0; ok && j < cnt; ++j) {
      const int k0 = ktile(j) * C::BN;
      ok = mbar_wait(bar(Q_SF), j & 1, abort_flag, ctl, SITE_BWD_S_FULL);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const int kbase = k0 + h * NC;
      const bool masked = causal && (k0 + C::BN - 1 > q0);
      float p[NC];
#pragma unroll
      for (int c0 = 0; c0 < NC; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(s_addr + c0, rr);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float v = ex2(fmaf(__uint_as_float(rr[i]), scale_log2, -lse2));
          if (masked && kbase + c0 + i > qrow) v = 0.f;
          p[c0 + i] = v;
        }
      }
      tc_fence_before();   // S has been read: its columns take the next key tile's S
      mbar_arrive(bar(Q_SC));
      ok = mbar_wait(bar(Q_DPF), j & 1, abort_flag, ctl, SITE_BWD_DP_FULL);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < NC; c0 += 32) {
        uint32_t rr[32], pk[16];
        tmem_ld32(dp_addr + c0, rr);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack_bf16x2(p[c0 + 2 * i] * (__uint_as_float(rr[2 * i]) - dd),
                              p[c0 + 2 * i + 1] * (__uint_as_float(rr[2 * i + 1]) - dd));
        tmem_st16(dp_addr + c0 / 2, pk);   // dS over this half's own dP columns
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(Q_DSR));
    }
    if (ok) {
      ok = mbar_wait(bar(Q_ACC), 0, abort_flag, ctl, SITE_BWD_ACC_DONE);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const uint32_t src = tmem + lane_off + C::DQ_COL + h * (D / 2);
      __nv_bfloat16* dst = dQ + ((size_t)bh * n + qrow) * D + h * (D / 2);
#pragma unroll 1
      for (int c0 = 0; c0 < D / 2; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(src + c0, rr);
        tmem_ld_wait();
        if (cnt == 0) {   // block-sparse tile that keeps nothing: dQ = 0, TMEM never written
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = 0u;
        }
        if (qrow < n) store32_bf16(dst + c0, rr, scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc<512>(tmem);
}

template <int D, int KR = 128>
int launch_kv_cfg(const void* Q, const void* K, const void* V, const void* dO, const float* LSE2,
                  const float* Dv, void* dK, void* dV, float* dKacc, float* dVacc,
                  int BH, const HeadMap& hm, int gsplit, const TileLists& tl, int n, int n_pad,
                  float scale, int causal, const KernelCtl& ctl, cudaStream_t st,
                  void* dSt = nullptr, int ld_ds = 0) {
  using C = KvCfg<D>;
  const int BHkv = BH / hm.group;
  CUtensorMap tq, tk, tv, tg;
  if (!make_tmap_bf16(&tq, Q, D, n, BH, 64, C::BM) ||
      !make_tmap_bf16(&tk, K, D, n, BHkv, 64, C::BNK) ||
      !make_tmap_bf16(&tv, V, D, n, BHkv, 64, C::BNK) ||
      !make_tmap_bf16(&tg, dO, D, n, BH, 64, C::BM))
    return ATTN_ERR_CUDA;
  // dS^T for the dQ mode "spill": [BH][n keys][n queries], rows ld_ds apart;
  // stores are clipped at n in both dimensions
  CUtensorMap ts;
  std::memset(&ts, 0, sizeof(ts));
  if (dSt && !make_tmap_bf16(&ts, dSt, n, n, BH, 64, C::BNK, ld_ds)) return ATTN_ERR_CUDA;
  if (tl.lists && hm.group > 1) return ATTN_ERR_UNSUPPORTED;
  if (dSt && (tl.lists || hm.group > 1 || KR != C::BNK)) return ATTN_ERR_UNSUPPORTED;
  auto kern = bwd_kv_kernel<D, false, false, KR>;
  if constexpr (KR == C::BNK) {
    if (tl.lists) kern = bwd_kv_kernel<D, false, true>;
    else if (hm.group > 1) kern = bwd_kv_kernel<D, true, false>;
  } else if (tl.lists || hm.group > 1) {
    return ATTN_ERR_UNSUPPORTED;
  }
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const int nkt = ceil_div(n, KR);
  dim3 grid = (causal || tl.lists) ? dim3(BHkv * C::NOUT, nkt, gsplit)
                                   : dim3(nkt * C::NOUT, BHkv, gsplit);
  kern<<<grid, C::NTHREADS, C::SMEM, st>>>(tq, tk, tv, tg, LSE2, Dv,
                                           static_cast<__nv_bfloat16*>(dK),
                                           static_cast<__nv_bfloat16*>(dV), dKacc, dVacc, hm,
                                           gsplit, tl, n, n_pad, scale,
                                           scale * 1.4426950408889634f, causal, ctl, ts,
                                           dSt != nullptr ? 1 : 0);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D>
int launch_q(const void* Q, const void* K, const void* V, const void* dO, const float* LSE2,
             const float* Dv, void* dQ, int BH, const HeadMap& hm, const TileLists& tl, int n,
             int n_pad, float scale, int causal, const KernelCtl& ctl, cudaStream_t st) {
  using C = QCfg<D>;
  const int BHkv = BH / hm.group;
  CUtensorMap tq, tk, tv, tg;
  if (!make_tmap_bf16(&tq, Q, D, n, BH, 64, C::BM) ||
      !make_tmap_bf16(&tk, K, D, n, BHkv, 64, C::BN) ||
      !make_tmap_bf16(&tv, V, D, n, BHkv, 64, C::BN) ||
      !make_tmap_bf16(&tg, dO, D, n, BH, 64, C::BM))
    return ATTN_ERR_CUDA;
  auto kern = bwd_q_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return ATTN_ERR_CUDA;
  const int ntile = ceil_div(n, C::BM);
  dim3 grid = (causal || tl.lists) ? dim3(BH, ntile) : dim3(ntile, BH);
  kern<<<grid, C::NTHREADS, C::SMEM, st>>>(tq, tk, tv, tg, LSE2, Dv, static_cast<__nv_bfloat16*>(dQ),
                                           hm, tl, n, n_pad, scale, scale * 1.4426950408889634f,
                                           causal, ctl);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

int launch_bwd_kv_tc(const void* Q, const void* K, const void* V, const void* dO,
                     const float* LSE2, const float* Dv, float* dQacc, void* dK, void* dV,
                     float* dKacc, float* dVacc, int BH, const HeadMap& hm, int gsplit,
                     const TileLists& tl, int n, int n_pad, int d, float scale, int causal,
                     const KernelCtl& ctl, cudaStream_t st, void* dSt, int ld_ds) {
  if (gsplit < 1 || hm.group % gsplit != 0 || (gsplit > 1 && (!dKacc || !dVacc)))
    return ATTN_ERR_INVALID_ARG;
  if (dSt && (d != 256 || hm.group != 1 || tl.lists || causal || ld_ds < n || ld_ds % 8 ||
              (reinterpret_cast<uintptr_t>(dSt) & 15u)))
    return ATTN_ERR_UNSUPPORTED;
  const bool dq = dQacc != nullptr;
  switch (d) {
    case 64:
      return launch_bwd_kv64_tc(Q, K, V, dO, LSE2, Dv, dQacc, dK, dV, dKacc, dVacc, BH, hm, gsplit,
                                tl, n, n_pad, scale, causal, ctl, st);
    case 128:
      return launch_bwd_kv128_tc(Q, K, V, dO, LSE2, Dv, dQacc, dK, dV, dKacc, dVacc, BH, hm, gsplit,
                                 tl, n, n_pad, scale, causal, ctl, st);
    case 256:   // dQ from the query-tile pass or the spill GEMM, never from this kernel
      if (dq) return ATTN_ERR_UNSUPPORTED;
      return launch_kv_cfg<256>(Q, K, V, dO, LSE2, Dv, dK, dV, dKacc, dVacc, BH, hm, gsplit, tl, n,
                                n_pad, scale, causal, ctl, st, dSt, ld_ds);
    default: return ATTN_ERR_UNSUPPORTED;
  }
}

int launch_bwd_kv_study(const void* Q, const void* K, const void* V, const void* dO,
                        const float* LSE2, const float* Dv, float* dQacc, void* dK, void* dV,
                        int BH, int key_rows, int n, int n_pad, int d, float scale, int causal,
                        const KernelCtl& ctl, cudaStream_t st) {
  const HeadMap hm{BH, 1};
  if (d != 256)
    return launch_bwd_kv_study_d64_128(Q, K, V, dO, LSE2, Dv, dQacc, dK, dV, BH, key_rows, n,
                                       n_pad, d, scale, causal, ctl, st);
  if (dQacc) return ATTN_ERR_UNSUPPORTED;
#define ATTN_KVS(KRR)                                                                          \
  return launch_kv_cfg<256, KRR>(Q, K, V, dO, LSE2, Dv, dK, dV, nullptr, nullptr,               \
                                        BH, hm, 1, TileLists(), n, n_pad, scale, causal, ctl, st)
  switch (key_rows) {
    case 128: ATTN_KVS(128);
    case 64: ATTN_KVS(64);
    case 32: ATTN_KVS(32);
    default: return ATTN_ERR_INVALID_ARG;
  }
#undef ATTN_KVS
}

int launch_bwd_q_tc(const void* Q, const void* K, const void* V, const void* dO,
                    const float* LSE2, const float* Dv, void* dQ, int BH, const HeadMap& hm,
                    const TileLists& tl, int n, int n_pad, int d, float scale, int causal,
                    const KernelCtl& ctl, cudaStream_t st) {
#define ATTN_Q(DD) \
  return launch_q<DD>(Q, K, V, dO, LSE2, Dv, dQ, BH, hm, tl, n, n_pad, scale, causal, ctl, st)
  switch (d) {
    case 64: ATTN_Q(64);
    case 128: ATTN_Q(128);
    case 256: ATTN_Q(256);
    default: return ATTN_ERR_UNSUPPORTED;
  }
#undef ATTN_Q
}

void bwd_kv_tiling(int d, int* kv_rows, int* query_rows) {
  *kv_rows = 128;
  *query_rows = d == 256 ? 64 : 128;
}

void bwd_q_tiling(int d, int* query_rows, int* kv_rows) {
  *query_rows = 128;
  *kv_rows = d == 256 ? 64 : 128;
}

}  // namespace attn
