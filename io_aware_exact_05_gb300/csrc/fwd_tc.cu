// fwd_tc.cu -- fused exact attention forward on the tcgen05 tensor cores.
//
// Computes O = softmax(scale Q K^T) V and LSE per row without writing the
// n x n score matrix anywhere but tensor memory ("Chapter 3.1 -- The cost of
// attention", section 5: tile Q, K, V into fast on-chip memory and combine
// partial softmax statistics block by block; "Flash Attention:
// Revolutionizing Transformer Efficiency", "The mathematics behind Flash
// Attention", formulas 1-2).
//
// CTA = QT query tiles of 128 rows of one (b, h) head.  Roles:
//   warp 0 (one lane)  TMA producer: Q tiles once, then the K_j tiles into
//                      their shared-memory ring.
//   warp 3 (one lane)  TMA producer of the V_j tiles (a ring of their own).
//   warp 1             MMA issuer (the whole warp runs the loop, an elected
//                      lane issues): S = Q K_j^T (SS-MMA into a TMEM slot;
//                      TS with Q in TMEM at d = 256), O_t += P V_j (TS-MMA:
//                      P read from TMEM).
//   warp 2             allocates / frees tensor memory; in block-sparse
//                      launches with two query tiles, warps 1 and 2 each
//                      issue the MMAs of one tile.
//   warpgroup 1 + t    softmax of query tile t: thread r owns row r (TMEM
//                      lane r).  Loads its S row, applies the causal/ragged
//                      mask, updates the running max m and sum l (log2
//                      domain), writes P = 2^(s*scale*log2e - m) as bf16 over
//                      the S slot, rescales its O row in TMEM when m moved,
//                      and finally writes O / l and LSE.
// Units (t, j) are processed in the order j-major, t-minor; unit number k
// uses S slot k % 2, so the tensor cores compute the next unit's S while the
// current unit's softmax runs (two tiles ping-pong when QT = 2).
//
// The running-max rescale is skipped while the new maximum exceeds the kept
// one by at most 8 (a factor 256 in P); both l and O are accumulated against
// the same kept maximum, so the final O / l is unchanged.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm100.cuh"

namespace attn {
namespace {

using namespace sm100;

template <int D, int BN, int QT>
struct FwdCfg {
  static constexpr int BM = 128;
  static constexpr int NKB = D / 64;            // 64-wide (128 B) column boxes
  static constexpr int KSTK = 3;                 // K ring depth
  static constexpr int KSTV = (D == 64) ? 3 : 2; // V ring depth
  static constexpr uint32_t Q_BYTES = BM * D * 2;
  static constexpr uint32_t KV_BYTES = BN * D * 2;
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = Q_OFF + QT * Q_BYTES;
  static constexpr uint32_t V_OFF = K_OFF + KSTK * KV_BYTES;
  static constexpr uint32_t BAR_OFF = V_OFF + KSTV * KV_BYTES;
  static constexpr uint32_t SMEM = BAR_OFF + 256 + 1024;
  static constexpr int S_COL = 0;               // two S slots of BN columns
  static constexpr int O_COL = 2 * BN;          // QT accumulators of D columns
  // d = 256 (one query tile): Q is the A operand of S = Q K^T from tensor
  // memory, so the S products read only K from shared memory
  static constexpr bool Q_IN_TMEM = (D == 256 && QT == 1);
  static constexpr int Q_COL = 2 * BN + QT * D;
  static constexpr int NTHREADS = 128 * (1 + QT);
  static constexpr int TMEM_NEED = 2 * BN + QT * D + (Q_IN_TMEM ? D / 2 : 0);
  // allocation: a power of two of at least 32 columns; at most 256 columns
  // and half the shared memory let two CTAs share an SM (each with its own
  // producer, MMA issuer and softmax warpgroup)
  static constexpr int TMEM_COLS = TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
  static constexpr int MINB = (TMEM_COLS <= 256 && SMEM <= 232448 / 2) ? 2 : 1;
  static_assert(TMEM_NEED <= 512, "tensor memory budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// Barrier indices inside the barrier block.
enum : int { B_Q = 0, B_KF = 1, B_KE = 4, B_VF = 7, B_VE = 10, B_SF = 13, B_PF = 15, B_OD = 17,
             B_DRAIN = 19, B_QC = 20, B_DRAIN1 = 21, B_COUNT = 22 };
// B_QC: Q copied to tensor memory; B_DRAIN1: the second issuer's drain
// The barrier block holds at most three K and three V ring stages (and 24
// barriers of 8 bytes below the tensor-memory slot at +192).
template <class C>
struct FitsBarrierBlock {
  static constexpr bool value = C::KSTK <= B_KE - B_KF && C::KSTK <= B_VF - B_KE &&
                                C::KSTV <= B_VE - B_VF && C::KSTV <= B_SF - B_VE &&
                                B_COUNT * 8 <= 192;
};

struct TileInfo {
  int last0, last1;   // last KV tile index each query tile needs (-1: none)
};

// Unit k -> (query tile t, KV tile j) in the issue order j-major, t-minor.
// Tile 1 never needs fewer KV tiles than tile 0, so the order is: pairs
// (0, j), (1, j) while both tiles need j, then tile 1 alone.
struct Unit { int t, j; };
template <int QT>
__device__ __forceinline__ Unit unit_at(int k, const TileInfo& ti) {
  if (QT == 1 || ti.last1 < 0) return {0, k};
  const int pairs = ti.last0 + 1;
  if (k < 2 * pairs) return {k & 1, k >> 1};
  return {1, k - pairs};
}

__device__ __forceinline__ int unit_pos(int t, int j, const TileInfo& ti) {
  return min(j, ti.last0 + 1) + min(j, ti.last1 + 1) + ((t == 1 && j <= ti.last0) ? 1 : 0);
}
// The issuer follows PV of unit k with S of unit k + 2.  When that S is the
// same query tile's next KV step, the commit that tells the tile's softmax
// "S ready" also covers the PV before it (a commit tracks every earlier MMA
// of its thread), so that PV needs no commit of its own and the softmax no
// wait for it.  Both sides evaluate this to keep the O-done phases in step.
__device__ __forceinline__ bool pv_implied(int t, int j, const TileInfo& ti) {
  const int last = t == 0 ? ti.last0 : ti.last1;
  return j < last && unit_pos(t, j + 1, ti) == unit_pos(t, j, ti) + 2;
}

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const float* v, float mul) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(v[2 * i] * mul, v[2 * i + 1] * mul);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    reinterpret_cast<uint4*>(dst)[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
}

// GROUPED: query heads share key/value heads (compiled separately so the
// one-head-per-head kernel does no head arithmetic).  SPARSE: a block
// pattern keeps only some KV tiles; the CTA walks its list of them (the
// union over its query tiles, each entry flagging the tiles it is kept for)
// instead of the dense range.
template <int D, int BN, int QT, bool GROUPED, bool SPARSE>
__global__ void __launch_bounds__(FwdCfg<D, BN, QT>::NTHREADS, FwdCfg<D, BN, QT>::MINB)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
              float* __restrict__ LSE, HeadMap hm, TileLists tl, int n, float scale_log2,
              int causal, KernelCtl ctl) {
  using C = FwdCfg<D, BN, QT>;
  static_assert(FitsBarrierBlock<C>::value, "ring deeper than its barrier slots");
  // Block-sparse, two query tiles: one MMA-issuing warp per tile (warps 1
  // and 2), each tile with its own S slot, so a tile whose list entry is not
  // kept never waits behind the other tile's units (A/B on
  // b2h16_n16k_d128_sparse: 0.394 -> 0.346 ms).  Dense launches keep one
  // issuer with S ping-ponging between the tiles in a fixed unit order (one
  // issuer per tile was 10 % slower there: each tile's S then completes
  // later behind the other tile's interleaved MMAs).
  constexpr bool DUAL = (QT == 2) && SPARSE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
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
  // head's K and V shared in L2 by CTAs that run together.  Causal and dense,
  // the heads go in groups of 8 (the last group may be smaller), each
  // group's tiles longest first, group after group: only one group's K and
  // V are in flight, which keeps them in L2 (DRAM reads per launch 545 ->
  // 202 MB on B2 H16 n8192 d128, 0.411 -> 0.406 ms).
  const bool heads_fast = causal || SPARSE;
  int head_ix = heads_fast ? blockIdx.x : blockIdx.y;
  int tile_pos = heads_fast ? (int)blockIdx.y : (int)blockIdx.x;
  if (causal && !SPARSE) {
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
  const int bh = head_ix;                        // query head (Q, O, LSE)
  const int bkv = GROUPED ? hm.kv_of(bh) : bh;   // key/value head (K, V)
  const int ntile = heads_fast ? gridDim.y : gridDim.x;
  const int tile_ix = tile_pos;
  const int cta = causal ? (ntile - 1 - tile_ix) : tile_ix;
  const int row0 = cta * (QT * C::BM);
  const int nkv = (n + BN - 1) / BN;

  // SPARSE: list position j holds KV tile tile_at(j) (both query tiles walk
  // the whole list; a tile masks the entries not kept for it).
  const int* slist = SPARSE ? tl.lists + (size_t)cta * tl.stride : nullptr;
  const int slen = SPARSE ? tl.counts[cta] : 0;
  auto tile_at = [&](int j) { return SPARSE ? (slist[j] & 0xFFFF) : j; };
  TileInfo ti;
  {
    int last[2] = {-1, -1};
    for (int t = 0; t < QT; ++t) {
      const int r0 = row0 + t * C::BM;
      if (r0 < n)
        last[t] = SPARSE ? slen - 1 : causal ? min(nkv - 1, (r0 + C::BM - 1) / BN) : nkv - 1;
    }
    ti.last0 = last[0];
    ti.last1 = last[1];
  }
  const int jmax = max(ti.last0, ti.last1);

  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q), 1);
    for (int s = 0; s < C::KSTK; ++s) {
      mbar_init(bar(B_KF + s), 1);
      mbar_init(bar(B_KE + s), DUAL ? 2 : 1);   // DUAL: released by both issuers
    }
    for (int s = 0; s < C::KSTV; ++s) {
      mbar_init(bar(B_VF + s), 1);
      mbar_init(bar(B_VE + s), DUAL ? 2 : 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_SF + s), 1);
      mbar_init(bar(B_PF + s), 128);
      mbar_init(bar(B_OD + s), 1);
    }
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_DRAIN1), 1);
    mbar_init(bar(B_QC), 128);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 2) tmem_alloc<C::TMEM_COLS>(smem_u32(tmem_slot));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    if (QT == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 88;");
    if (warp == 0 && lane == 0) {
      // --------------------------------------------------- producer: Q, then K tiles
      uint32_t qbytes = 0;
      for (int t = 0; t < QT; ++t)
        if (row0 + t * C::BM < n) qbytes += C::Q_BYTES;
      mbar_expect_tx(bar(B_Q), qbytes);
      for (int t = 0; t < QT; ++t) {
        if (row0 + t * C::BM >= n) continue;
#pragma unroll
        for (int kb = 0; kb < C::NKB; ++kb)
          tma_load_3d(sb + C::Q_OFF + t * C::Q_BYTES + kb * (C::BM * 128), &tmQ, kb * 64,
                      row0 + t * C::BM, bh, bar(B_Q));
      }
      int last_k[C::KSTK];
      for (int s = 0; s < C::KSTK; ++s) last_k[s] = -1;
      for (int j = 0; j <= jmax; ++j) {
        const int s = j % C::KSTK;
        if (!mbar_wait(bar(B_KE + s), ((j / C::KSTK) & 1) ^ 1, abort_flag, ctl, SITE_FWD_KV_EMPTY))
          break;
        mbar_expect_tx(bar(B_KF + s), C::KV_BYTES);
#pragma unroll
        for (int kb = 0; kb < C::NKB; ++kb)
          tma_load_3d(sb + C::K_OFF + s * C::KV_BYTES + kb * (BN * 128), &tmK, kb * 64, tile_at(j) * BN, bkv,
                      bar(B_KF + s));
        last_k[s] = j;
      }
      if (*abort_flag) {   // let issued copies land before the CTA may exit
        volatile int no_abort = 0;
        mbar_wait(bar(B_Q), 0, &no_abort, ctl, SITE_FWD_LOAD_Q);
        for (int s = 0; s < C::KSTK; ++s)
          if (last_k[s] >= 0)
            mbar_wait(bar(B_KF + s), (last_k[s] / C::KSTK) & 1, &no_abort, ctl, SITE_FWD_K_FULL);
      }
    } else if (warp == 3 && lane == 0) {
      // --------------------------------------------------- producer: V tiles
      int last_v[C::KSTV];
      for (int s = 0; s < C::KSTV; ++s) last_v[s] = -1;
      for (int j = 0; j <= jmax; ++j) {
        const int s = j % C::KSTV;
        if (!mbar_wait(bar(B_VE + s), ((j / C::KSTV) & 1) ^ 1, abort_flag, ctl, SITE_FWD_KV_EMPTY))
          break;
        mbar_expect_tx(bar(B_VF + s), C::KV_BYTES);
#pragma unroll
        for (int kb = 0; kb < C::NKB; ++kb)
          tma_load_3d(sb + C::V_OFF + s * C::KV_BYTES + kb * (BN * 128), &tmV, kb * 64, tile_at(j) * BN, bkv,
                      bar(B_VF + s));
        last_v[s] = j;
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        for (int s = 0; s < C::KSTV; ++s)
          if (last_v[s] >= 0)
            mbar_wait(bar(B_VF + s), (last_v[s] / C::KSTV) & 1, &no_abort, ctl, SITE_FWD_V_FULL);
      }
    } else if (DUAL && (warp == 1 || warp == 2)) {
      // ------------------------------------------- MMA issuer of query tile t
      // Tile t's S lives in slot t.  Per KV step j: S(t, j) (after K_j
      // landed), then, once the softmax published P(t, j), PV(t, j) and S(t,
      // j + 1).  The commit after S(t, j + 1) also covers PV(t, j) (a commit
      // tracks every earlier MMA of its thread), so only the tile's last PV
      // is committed on its own.  Each issuer releases a K or V stage once
      // it has read it, twice when the other tile does not use that stage.
      const int t = warp - 1;
      constexpr uint32_t idesc_s = idesc_bf16(C::BM, BN, false, false);   // Q, K both K-major
      constexpr uint32_t idesc_o = idesc_bf16(C::BM, D, false, true);     // P (TMEM), V MN-major
      constexpr uint32_t HI = sdesc_hi(1024);
      const int last = t == 0 ? ti.last0 : ti.last1;
      const int last_other = t == 0 ? ti.last1 : ti.last0;
      const uint32_t qb = sdesc_lo(sb + C::Q_OFF, 16) + t * (C::Q_BYTES >> 4);
      const uint32_t k_lo = sdesc_lo(sb + C::K_OFF, 16);
      const uint32_t v_lo = sdesc_lo(sb + C::V_OFF, BN * 128);
      const uint32_t s_col = tmem + C::S_COL + t * BN;
      bool ok = mbar_wait_warp(bar(B_Q), 0, abort_flag, ctl, SITE_FWD_LOAD_Q);
      bool drop_s = false, o_init = false;
      auto issue_s = [&](int j, int ent) -> bool {   // S(t, j) = Q_t K_j^T into slot t
        const int st = j % C::KSTK;
        if (!mbar_wait_warp(bar(B_KF + st), (j / C::KSTK) & 1, abort_flag, ctl, SITE_FWD_K_FULL))
          return false;
        drop_s = SPARSE && !((ent >> (16 + t)) & 1);
        tc_fence_after();
        const uint32_t kb = k_lo + st * (C::KV_BYTES >> 4);
#pragma unroll
        for (int b = 0; b < C::NKB; ++b) {
          if (drop_s) break;
          uint32_t alo[4], blo[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            alo[i] = qb + b * (C::BM * 128 / 16) + 2 * i;
            blo[i] = kb + b * (BN * 128 / 16) + 2 * i;
          }
          mma_ss_x4(s_col, alo, HI, blo, HI, idesc_s, b > 0);
        }
        tc_commit(bar(B_SF + t));
        tc_commit(bar(B_KE + st));
        if (j > last_other) tc_commit(bar(B_KE + st));
        return true;
      };
      auto entry_of = [&](int j) { return SPARSE ? slist[j] : 0; };
      if (ok && last >= 0) ok = issue_s(0, entry_of(0));
      for (int j = 0; ok && j <= last; ++j) {
        const int sv = j % C::KSTV;
        const uint32_t vb = v_lo + sv * (C::KV_BYTES >> 4);
        const int ent1 = (SPARSE && j + 1 <= last) ? entry_of(j + 1) : 0;   // load before the wait
        if (!mbar_wait_warp(bar(B_PF + t), j & 1, abort_flag, ctl, SITE_FWD_P_FULL)) break;
        if (!mbar_wait_warp(bar(B_VF + sv), (j / C::KSTV) & 1, abort_flag, ctl, SITE_FWD_V_FULL))
          break;
        tc_fence_after();
#pragma unroll
        for (int b = 0; b < BN / 64; ++b) {   // 64 keys (4 MMAs of K = 16) per group
          if (drop_s) break;
          uint32_t blo[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) blo[i] = vb + (4 * b + i) * (2048 / 16);
          const bool acc = SPARSE ? (o_init || b > 0) : (j > 0 || b > 0);
          mma_ts_x4(tmem + C::O_COL + t * D, s_col + 32 * b, blo, HI, idesc_o, acc);
        }
        if (SPARSE && !drop_s) o_init = true;
        if (j == last) tc_commit(bar(B_OD + t));
        tc_commit(bar(B_VE + sv));
        if (j > last_other) tc_commit(bar(B_VE + sv));
        if (j + 1 <= last) ok = issue_s(j + 1, ent1);
      }
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        const int drain = t == 0 ? B_DRAIN : B_DRAIN1;
        tc_commit(bar(drain));
        volatile int no_abort = 0;
        mbar_wait_warp(bar(drain), 0, &no_abort, ctl, SITE_FWD_O_DONE);
      }
    } else if (!DUAL && warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs this loop (one elected lane issues each MMA and
      // commit), so every descriptor stays warp-uniform.  Per-unit
      // bookkeeping is kept to a few integer operations: the MMA queue is
      // shallow, so scalar work between units shows up as idle tensor cycles.
      constexpr uint32_t idesc_s = idesc_bf16(C::BM, BN, false, false);   // Q, K both K-major
      constexpr uint32_t idesc_o = idesc_bf16(C::BM, D, false, true);     // P (TMEM), V MN-major
      constexpr uint32_t HI = sdesc_hi(1024);
      const int total = (ti.last0 + 1) + (ti.last1 + 1);
      const uint32_t q_lo = sdesc_lo(sb + C::Q_OFF, 16), k_lo = sdesc_lo(sb + C::K_OFF, 16);
      const uint32_t v_lo = sdesc_lo(sb + C::V_OFF, BN * 128);
      auto first_user = [&](int t, int j) { return t == 0 || j > ti.last0; };
      auto last_user = [&](int t, int j) { return QT == 1 || t == 1 || j > ti.last1; };
      bool ok = mbar_wait_warp(bar(B_Q), 0, abort_flag, ctl, SITE_FWD_LOAD_Q);
      if (C::Q_IN_TMEM) ok = ok && mbar_wait_warp(bar(B_QC), 0, abort_flag, ctl, SITE_FWD_LOAD_Q);
      // SPARSE: a unit whose list entry is not kept for its tile ("dropped")
      // gets no MMAs; its waits and commits stay, so every barrier phase is
      // the same as with the MMAs (a commit with nothing new completes when
      // the earlier MMAs have).  Bit k & 1 of drop_s remembers S(k)'s flag for
      // PV(k); bit t of o_init says tile t's O holds a first PV already.
      uint32_t drop_s = 0, o_init = 0;
      auto dropped_unit = [&](const Unit& u, int ent) {
        return SPARSE && !((ent >> (16 + u.t)) & 1);
      };
      // S(k) = Q_t K_j^T into S slot k & 1
      auto issue_s = [&](int k, int ent) -> bool {
        const Unit u = unit_at<QT>(k, ti);
        const int s = u.j % C::KSTK;
        const uint32_t qb = q_lo + u.t * (C::Q_BYTES >> 4), kb = k_lo + s * (C::KV_BYTES >> 4);
        if (first_user(u.t, u.j)) {
          if (!mbar_wait_warp(bar(B_KF + s), (u.j / C::KSTK) & 1, abort_flag, ctl, SITE_FWD_K_FULL))
            return false;
        }
        const bool drop = dropped_unit(u, ent);
        drop_s = (drop_s & ~(1u << (k & 1))) | ((uint32_t)drop << (k & 1));
        tc_fence_after();
#pragma unroll
        for (int b = 0; b < C::NKB; ++b) {   // one 64-wide column box of Q and K per group
          if (drop) break;
          uint32_t alo[4], blo[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            alo[i] = qb + b * (C::BM * 128 / 16) + 2 * i;
            blo[i] = kb + b * (BN * 128 / 16) + 2 * i;
          }
          if (C::Q_IN_TMEM)   // A = Q from tensor memory: box b at columns 32b
            mma_ts_x4(tmem + C::S_COL + (k & 1) * BN, tmem + C::Q_COL + 32 * b, blo, HI, idesc_s,
                      b > 0);
          else
            mma_ss_x4(tmem + C::S_COL + (k & 1) * BN, alo, HI, blo, HI, idesc_s, b > 0);
        }
        tc_commit(bar(B_SF + (k & 1)));
        if (last_user(u.t, u.j)) tc_commit(bar(B_KE + s));
        return true;
      };
      auto entry_of = [&](int k) { return SPARSE ? slist[unit_at<QT>(k, ti).j] : 0; };
      if (ok && total > 0) ok = issue_s(0, entry_of(0));
      if (ok && total > 1) ok = issue_s(1, entry_of(1));
      for (int k = 0; ok && k < total; ++k) {
        const Unit u = unit_at<QT>(k, ti);
        const int s = u.j % C::KSTV;
        const uint32_t vb = v_lo + s * (C::KV_BYTES >> 4);
        const uint32_t pa = tmem + C::S_COL + (k & 1) * BN;   // P: bf16 pairs, BN/2 columns
        const int ent2 = (SPARSE && k + 2 < total) ? entry_of(k + 2) : 0;   // load before the wait
        if (!mbar_wait_warp(bar(B_PF + (k & 1)), (k >> 1) & 1, abort_flag, ctl, SITE_FWD_P_FULL)) break;
        if (first_user(u.t, u.j)) {
          if (!mbar_wait_warp(bar(B_VF + s), (u.j / C::KSTV) & 1, abort_flag, ctl, SITE_FWD_V_FULL)) break;
        }
        tc_fence_after();
        const bool drop_pv = SPARSE && ((drop_s >> (k & 1)) & 1);
#pragma unroll
        for (int b = 0; b < BN / 64; ++b) {   // 64 keys (4 MMAs of K = 16) per group
          if (drop_pv) break;
          uint32_t blo[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) blo[i] = vb + (4 * b + i) * (2048 / 16);
          const bool acc = SPARSE ? (((o_init >> u.t) & 1) || b > 0) : (u.j > 0 || b > 0);
          mma_ts_x4(tmem + C::O_COL + u.t * D, pa + 32 * b, blo, HI, idesc_o, acc);
        }
        if (SPARSE && !drop_pv) o_init |= 1u << u.t;
        if (!pv_implied(u.t, u.j, ti)) tc_commit(bar(B_OD + u.t));
        if (last_user(u.t, u.j)) tc_commit(bar(B_VE + s));
        if (k + 2 < total) ok = issue_s(k + 2, ent2);
      }
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        tc_commit(bar(B_DRAIN));
        volatile int no_abort = 0;
        mbar_wait_warp(bar(B_DRAIN), 0, &no_abort, ctl, SITE_FWD_O_DONE);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax
    if (QT == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 208;");
    const int t = (warp >> 2) - 1;
    const int q = warp & 3;                       // TMEM lane quarter
    const int r = q * 32 + lane;
    const int row = row0 + t * C::BM + r;
    const int last = (t == 0) ? ti.last0 : ti.last1;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    float m = -INFINITY, l = 0.f;
    int odc = 0;   // O-done phases consumed (PVs with a commit of their own)
    bool ok = true;
    if (C::Q_IN_TMEM) {   // the (only) softmax warpgroup copies the Q rows into tensor memory
      ok = mbar_wait(bar(B_Q), 0, abort_flag, ctl, SITE_FWD_LOAD_Q);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tile_to_tmem<D>(smem + C::Q_OFF, tmem + lane_off + C::Q_COL, r);
        tc_fence_before();
        mbar_arrive(bar(B_QC));
      }
    }
    for (int j = 0; ok && j <= last; ++j) {
      const int k = DUAL ? 2 * j : unit_pos(t, j, ti);   // DUAL: slot t, phase j
      const int slot = DUAL ? t : (k & 1);
      const int ent = SPARSE ? slist[j] : j;   // read before the wait hides its latency
      ok = mbar_wait(bar(B_SF + slot), (k >> 1) & 1, abort_flag, ctl, SITE_FWD_S_FULL);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // SPARSE: an entry kept only for the other tile of the CTA ("dropped")
      // got no S or PV MMA; its step keeps only the barrier phases
      const bool drop = SPARSE && !((ent >> (16 + t)) & 1);
      float alpha = 1.0f, m_new = m;
      if (!drop) {
        tc_fence_after();
        const uint32_t sa = tmem + lane_off + C::S_COL + slot * BN;
        // all BN columns of this row: issue every TMEM load, then wait once
        uint32_t sr[BN];
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32)
          tmem_ld32(sa + c0, *reinterpret_cast<uint32_t(*)[32]>(&sr[c0]));
        tmem_ld_wait();
        reg_fence<BN>(sr);
        float* s = reinterpret_cast<float*>(sr);
        const int col0 = (SPARSE ? (ent & 0xFFFF) : j) * BN;
        const bool need_mask = (col0 + BN > n) || (causal && col0 + BN - 1 > row0 + t * C::BM);
        if (need_mask) {
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
        m_new = (m_cand > m + 8.0f) ? m_cand : m;
        // SPARSE: a row can have no kept score yet (m_new = -inf); exponents are
        // then taken against 0, so P = 0 and alpha = 0 instead of NaN
        const float m_base = (SPARSE && m_new == -INFINITY) ? 0.f : m_new;
        alpha = ex2(m - m_base);   // 0 on the first tile (m = -inf)
        // exponents and row sum on column pairs (paired fp32 FMA and add)
        const float2 c2 = make_float2(scale_log2, scale_log2);
        const float2 nm2 = make_float2(-m_base, -m_base);
        float2 rs4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        const uint32_t pa = sa;   // P overwrites the first BN/2 columns of the slot
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x = __ffma2_rn(make_float2(s[c0 + 2 * i], s[c0 + 2 * i + 1]), c2, nm2);
            const float2 p = make_float2(ex2(x.x), ex2(x.y));
            rs4[i & 3] = __fadd2_rn(rs4[i & 3], p);
            pk[i] = pack_bf16x2(p.x, p.y);
          }
          tmem_st16(pa + c0 / 2, pk);
        }
        const float2 rs2 = __fadd2_rn(__fadd2_rn(rs4[0], rs4[1]), __fadd2_rn(rs4[2], rs4[3]));
        const float rs = rs2.x + rs2.y;
        tmem_st_wait();
        l = l * alpha + rs;
      }
      // PV of step j-1 must be done before O is rescaled.  It is when its
      // completion was implied by the S wait above; otherwise wait for its
      // own commit (every committed phase is waited for, so a parity wait
      // is never more than one phase behind).
      if (j > 0 && !DUAL && !pv_implied(t, j - 1, ti)) {
        ok = mbar_wait(bar(B_OD + t), odc & 1, abort_flag, ctl, SITE_FWD_O_DONE);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++odc;
      }
      // Rescale this row of O when its kept maximum moved.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {   // dropped: alpha = 1
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
      mbar_arrive(bar(B_PF + slot));
    }
    if (ok && last >= 0) {
      ok = mbar_wait(bar(B_OD + t), odc & 1, abort_flag, ctl, SITE_FWD_O_DONE);   // last PV: committed
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        // SPARSE, no kept score in this row: O = 0 (its TMEM columns may never
        // have been written, when every entry was dropped for this tile)
        const bool zero = SPARSE && l == 0.f;
        const float inv = zero ? 0.f : 1.f / l;
        const uint32_t oa = tmem + lane_off + C::O_COL + t * D;
        const size_t obase = ((size_t)bh * n + row) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t rr[32];
          tmem_ld32(oa + c0, rr);
          tmem_ld_wait();
          if (row < n) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = zero ? 0.f : __uint_as_float(rr[i]);
            store_row_bf16(O + obase + c0, v, inv);
          }
        }
        if (row < n)
          LSE[(size_t)bh * n + row] =
              (SPARSE && l == 0.f) ? -INFINITY : (m + __log2f(l)) * 0.69314718055994531f;
      }
    } else if (SPARSE && ok && last < 0 && row < n) {   // nothing kept for this CTA
      const size_t obase = ((size_t)bh * n + row) * D;
      for (int c = 0; c < D; c += 8)
        *reinterpret_cast<uint4*>(O + obase + c) = make_uint4(0u, 0u, 0u, 0u);
      LSE[(size_t)bh * n + row] = -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc<C::TMEM_COLS>(tmem);
}

template <int D, int BN, int QT>
int launch_cfg(const void* Q, const void* K, const void* V, void* O, float* LSE, int BH,
               const HeadMap& hm, const TileLists& tl, int n, float scale, int causal,
               const KernelCtl& ctl, cudaStream_t st) {
  using C = FwdCfg<D, BN, QT>;
  const int BHkv = BH / hm.group;
  if (tl.lists && hm.group > 1) return ATTN_ERR_UNSUPPORTED;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_bf16(&tq, Q, D, n, BH, 64, C::BM) || !make_tmap_bf16(&tk, K, D, n, BHkv, 64, BN) ||
      !make_tmap_bf16(&tv, V, D, n, BHkv, 64, BN))
    return ATTN_ERR_CUDA;
  auto kern = tl.lists        ? fwd_tc_kernel<D, BN, QT, false, true>
              : hm.group > 1 ? fwd_tc_kernel<D, BN, QT, true, false>
                             : fwd_tc_kernel<D, BN, QT, false, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  const int ntile = ceil_div(n, QT * C::BM);
  dim3 grid = (causal || tl.lists) ? dim3(BH, ntile) : dim3(ntile, BH);
  const float scale_log2 = scale * 1.4426950408889634f;
  kern<<<grid, C::NTHREADS, C::SMEM, st>>>(tq, tk, tv, static_cast<__nv_bfloat16*>(O), LSE, hm, tl,
                                           n, scale_log2, causal, ctl);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

// d = 64: one 128-query tile and 64-key tiles per CTA (192 TMEM columns,
// 66 KB of shared memory), so two CTAs share an SM; d = 128: two query tiles
// that ping-pong on one MMA issuer; d = 256: one query tile, Q in TMEM.
void fwd_tiling(int d, int* query_rows, int* query_tiles, int* kv_rows) {
  *query_rows = 128;
  *query_tiles = d == 128 ? 2 : 1;
  *kv_rows = d == 128 ? 128 : 64;
}

int launch_fwd_tc(const void* Q, const void* K, const void* V, void* O, float* LSE, int BH,
                  const HeadMap& hm, const TileLists& tl, int n, int d, float scale, int causal,
                  const KernelCtl& ctl, cudaStream_t st) {
  switch (d) {
    case 64: return launch_cfg<64, 64, 1>(Q, K, V, O, LSE, BH, hm, tl, n, scale, causal, ctl, st);
    case 128:
      return launch_cfg<128, 128, 2>(Q, K, V, O, LSE, BH, hm, tl, n, scale, causal, ctl, st);
    case 256: return launch_cfg<256, 64, 1>(Q, K, V, O, LSE, BH, hm, tl, n, scale, causal, ctl, st);
    default: return ATTN_ERR_UNSUPPORTED;
  }
}

}  // namespace attn
