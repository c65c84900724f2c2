// gemm_tc.cu -- batched bf16 GEMM on the 5th-generation tensor cores.
//
//   C[b] = alpha * A[b] (M x K) * B[b] (K x N), fp32 accumulation in TMEM.
//
// One CTA computes one 128 x BN tile of C.  Warp 0 (one lane) streams 64-wide
// K blocks of A and B into a 4-stage shared-memory ring with TMA; warp 1
// (one lane) issues tcgen05.mma (M=128, N=BN, K=16) per K block and releases
// each stage with tcgen05.commit; then all four warps read the accumulator
// back with tcgen05.ld (thread t <-> row t) and store C: through a ring of
// 128-byte-swizzled 16 KB shared-memory boxes (the drained stage ring) and
// TMA tile stores when C's rows are 16-byte multiples, else directly from
// registers.  A and B may each be
// K-major or MN-major in global memory: the shared-memory descriptors and the
// transpose bits of the instruction descriptor absorb the difference, so no
// operand is ever transposed in memory.  This GEMM carries every n x n and
// n x d product of the materialise-P comparison path.
#include <cuda_bf16.h>

#include "kernels.h"
#include "sm100.cuh"

namespace attn {
namespace {

using namespace sm100;

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kStages = 4;
static_assert(kBK == 64, "four K slices of 16 per staged block");

// MT: 128-row M tiles per CTA, each with its own BN-column accumulator, all
// fed by the same staged B block (MT = 2 halves B's reads through L2 for the
// long n x d-output contractions, where every M tile reads all of B).
template <int BN, int STG = kStages, int MT = 1>
struct GemmLayout {
  static constexpr uint32_t A_TILE = kBM * kBK * 2;
  static constexpr uint32_t A_BYTES = MT * A_TILE;
  static constexpr uint32_t B_BYTES = BN * kBK * 2;
  static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
  static constexpr uint32_t BAR_OFF = STG * STAGE;
  static constexpr uint32_t TOTAL = BAR_OFF + 256 + 1024;  // barriers + slack for 1 KB alignment
  // two CTAs per SM when their shared and tensor memory fit (the epilogue of
  // one then overlaps the loads and MMAs of the other)
  static constexpr int MINB = (TOTAL <= 232448 / 2 && BN <= 256) ? 2 : 1;
  static_assert(2 * STG + 2 <= 16, "barriers below the tensor-memory slot");
  static_assert(MT * BN <= 512, "accumulators within the tensor memory");
};

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Descriptor of one 16-deep K slice `kk` of a 64-deep staged K block.
//  K-major: rows of 64 K elements (128 B); the slice starts 32 B further.
//  MN-major: rows of 64 M/N elements, one per k; the slice starts 16 rows
//  (2048 B) further; 64-wide M/N blocks are `mn_block_bytes` apart.
// (Low half; the high half is sdesc_hi(1024) in both cases.)
__device__ __forceinline__ uint32_t operand_lo(uint32_t base, bool kmajor, int kk,
                                               uint32_t mn_block_bytes) {
  return kmajor ? sdesc_lo(base + kk * 32, 16) : sdesc_lo(base + kk * 2048, mn_block_bytes);
}

template <int BN, bool A_K, bool B_K, bool C_F32, int STG = kStages, bool TMA_C = true, int MT = 1>
__global__ void __launch_bounds__(128, GemmLayout<BN, STG, MT>::MINB)
gemm_bf16_kernel(const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tB,
                 const __grid_constant__ CUtensorMap tC, void* __restrict__ C, int M, int N, int K,
                 float alpha, KernelCtl ctl) {
  using L = GemmLayout<BN, STG, MT>;
  constexpr int kStages = STG;   // ring depth of this instance
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1k(smem_raw);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::BAR_OFF;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t acc_bar = bar0 + 8u * (2 * kStages);
  const uint32_t drain_bar = acc_bar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::BAR_OFF + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::BAR_OFF + 136);

  const int warp = warp_id_uniform(), lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * (kBM * MT), n0 = blockIdx.x * BN, b = blockIdx.z;
  const int nkb = (K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(acc_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tA);
    tma_prefetch_desc(&tB);
  }
  if (warp == 2) tmem_alloc<BN * MT>(smem_u32(tmem_slot));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    int issued_last[kStages];
    for (int s = 0; s < kStages; ++s) issued_last[s] = -1;
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % kStages;
      if (!mbar_wait(empty(s), ((kb / kStages) & 1) ^ 1, abort_flag, ctl, SITE_GEMM_EMPTY)) break;
      const uint32_t sa = sbase + s * L::STAGE, sb = sa + L::A_BYTES;
      mbar_expect_tx(full(s), L::STAGE);
#pragma unroll
      for (int t = 0; t < MT; ++t) {   // rows beyond M read the fill value
        const uint32_t sat = sa + t * L::A_TILE;
        const int mt = m0 + t * kBM;
        if (A_K) {
          tma_load_3d(sat, &tA, kb * kBK, mt, b, full(s));
        } else {
          tma_load_3d(sat, &tA, mt, kb * kBK, b, full(s));
          tma_load_3d(sat + 8192, &tA, mt + 64, kb * kBK, b, full(s));
        }
      }
      if (B_K) {
        tma_load_3d(sb, &tB, kb * kBK, n0, b, full(s));
      } else {
#pragma unroll
        for (int nb = 0; nb < BN / 64; ++nb) tma_load_3d(sb + nb * 8192, &tB, n0 + nb * 64, kb * kBK, b, full(s));
      }
      issued_last[s] = kb;
    }
    if (*abort_flag) {
      // Let every copy already issued land before the CTA can exit.
      for (int s = 0; s < kStages; ++s)
        if (issued_last[s] >= 0) {
          KernelCtl c2 = ctl;
          volatile int no_abort = 0;
          mbar_wait(full(s), (issued_last[s] / kStages) & 1, &no_abort, c2, SITE_GEMM_FULL);
        }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (the whole warp runs the loop; one elected lane issues)
    constexpr uint32_t idesc = idesc_bf16(kBM, BN, !A_K, !B_K);
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % kStages;
      if (!mbar_wait_warp(full(s), (kb / kStages) & 1, abort_flag, ctl, SITE_GEMM_FULL)) break;
      tc_fence_after();
      const uint32_t sa = sbase + s * L::STAGE, sb = sa + L::A_BYTES;
      // the block's four K slices from one asm block per M tile
      uint32_t blo[4];
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) blo[kk] = operand_lo(sb, B_K, kk, 8192);
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        uint32_t alo[4];
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) alo[kk] = operand_lo(sa + t * L::A_TILE, A_K, kk, 8192);
        mma_ss_x4(tmem + t * BN, alo, sdesc_hi(1024), blo, sdesc_hi(1024), idesc, kb != 0);
      }
      tc_commit(empty(s));
    }
    tc_commit(acc_bar);
    if (__any_sync(0xffffffffu, *abort_flag != 0)) {
      tc_commit(drain_bar);
      volatile int no_abort = 0;
      mbar_wait_warp(drain_bar, 0, &no_abort, ctl, SITE_GEMM_ACC);
    }
  }
  __syncwarp();

  // ---------------- epilogue: TMEM -> registers -> global
  // one verdict for the whole CTA: the TMA epilogue's named barriers need
  // every thread, so no thread may leave on its own
  const bool ok = __syncthreads_and(mbar_wait(acc_bar, 0, abort_flag, ctl, SITE_GEMM_ACC)) != 0;
  tc_fence_after();
  if (TMA_C && ok) {
    // Every MMA has completed, so the stage ring is free: it holds NBOX boxes
    // of [128 rows][128 bytes] (32 fp32 or 64 bf16 columns), thread r writing
    // row r; one thread stores each box with TMA and keeps NBOX - 1 stores
    // reading shared memory while the next box is written.
    constexpr uint32_t BOX = kBM * 128;
    constexpr int COLS = C_F32 ? 32 : 64;
    constexpr int NBOX = (int)((L::BAR_OFF / BOX) < 4 ? (L::BAR_OFF / BOX) : 4);
    static_assert(NBOX >= 2, "two staging boxes at least");
    const int r = warp * 32 + lane;
    int slot = 0;
#pragma unroll 1
    for (int t = 0; t < MT && m0 + t * kBM < M; ++t) {
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16) + t * BN;
#pragma unroll 1
    for (int c0 = 0; c0 < BN && n0 + c0 < N; c0 += COLS) {
      uint32_t w[32];
      if (C_F32) {
        tmem_ld32(taddr + c0, w);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(alpha * __uint_as_float(w[i]));
      } else {
        uint32_t a[32], bb[32];
        tmem_ld32(taddr + c0, a);
        tmem_ld32(taddr + c0 + 32, bb);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          w[i] = pack_bf16x2(alpha * __uint_as_float(a[2 * i]), alpha * __uint_as_float(a[2 * i + 1]));
          w[16 + i] = pack_bf16x2(alpha * __uint_as_float(bb[2 * i]),
                                  alpha * __uint_as_float(bb[2 * i + 1]));
        }
      }
      uint8_t* box = smem + slot * BOX;
      if (threadIdx.x == 0) bulk_wait_read<NBOX - 1>();   // this box's last store has read it
      named_bar_sync(1, 128);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(box + sw128_offset(r, j)) =
            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (threadIdx.x == 0) {
        tma_store_3d(&tC, smem_u32(box), n0 + c0, m0 + t * kBM, b);
        bulk_commit_group();
      }
      slot = (slot + 1 == NBOX) ? 0 : slot + 1;
    }
    }
    if (threadIdx.x == 0) bulk_wait_all();   // the stores are complete before the CTA exits
  }
  if (!TMA_C && ok) {
#pragma unroll 1
    for (int t = 0; t < MT; ++t) {
    const int row = m0 + t * kBM + warp * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16) + t * BN;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(taddr + c0, r);
      tmem_ld_wait();
      const int col = n0 + c0;
      if (row < M && col < N) {
        if (C_F32) {
          float* dst = static_cast<float*>(C) + ((size_t)b * M + row) * N + col;
          if (col + 32 <= N && (N & 3) == 0) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(dst + i) =
                  make_float4(alpha * __uint_as_float(r[i]), alpha * __uint_as_float(r[i + 1]),
                              alpha * __uint_as_float(r[i + 2]), alpha * __uint_as_float(r[i + 3]));
          } else {
            for (int i = 0; i < 32 && col + i < N; ++i) dst[i] = alpha * __uint_as_float(r[i]);
          }
        } else {
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(C) + ((size_t)b * M + row) * N + col;
          if (col + 32 <= N && (N & 7) == 0) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[i] = pack_bf16x2(alpha * __uint_as_float(r[2 * i]),
                                  alpha * __uint_as_float(r[2 * i + 1]));
#pragma unroll
            for (int i = 0; i < 4; ++i)
              *reinterpret_cast<uint4*>(dst + 8 * i) =
                  make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          } else {
            for (int i = 0; i < 32 && col + i < N; ++i)
              dst[i] = __float2bfloat16_rn(alpha * __uint_as_float(r[i]));
          }
        }
      }
    }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) tmem_dealloc<BN * MT>(tmem);
}

template <int BN, bool A_K, bool B_K, bool C_F32, int STG = kStages, int MT = 1>
int launch_variant(const CUtensorMap& ta, const CUtensorMap& tb, void* C, int batch, int M,
                   int N, int K, float alpha, const KernelCtl& ctl, cudaStream_t st) {
  // long contractions with n x d bf16 outputs (dQ = dS K and the other
  // products against an n x n operand): two M tiles per CTA share each
  // staged B block, which halves B's reads through L2 (every M tile reads
  // all of B); three stages of 64 KB
  if constexpr (STG == kStages && MT == 1 && BN == 256 && !C_F32) {
    if (K > 4 * kBK && M > kBM)
      return launch_variant<BN, A_K, B_K, C_F32, 3, 2>(ta, tb, C, batch, M, N, K, alpha, ctl, st);
  }
  // short contractions (the n x n score products, K = d <= 256: four K blocks
  // or fewer) need no deep ring; two stages let two CTAs share an SM so that
  // one CTA's stores of its fp32 tile overlap the other's MMAs
  if constexpr (STG == kStages && C_F32 && A_K && B_K) {
    if (K <= 4 * kBK) return launch_variant<BN, A_K, B_K, C_F32, 2>(ta, tb, C, batch, M, N, K, alpha, ctl, st);
  }
  // C through TMA tile stores when its rows are 16-byte multiples (the
  // tensor map's stride rule) and its base is 16-byte aligned
  CUtensorMap tc;
  const bool tma_c =
      (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && (N * (C_F32 ? 4 : 2)) % 16 == 0 &&
      (C_F32 ? make_tmap_f32(&tc, C, N, M, batch, 32, kBM, true)
             : make_tmap_bf16(&tc, C, N, M, batch, 64, kBM));
  if (!tma_c) tc = ta;   // not read
  auto kern = tma_c ? gemm_bf16_kernel<BN, A_K, B_K, C_F32, STG, true, MT>
                    : gemm_bf16_kernel<BN, A_K, B_K, C_F32, STG, false, MT>;
  constexpr int smem = GemmLayout<BN, STG, MT>::TOTAL;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return ATTN_ERR_CUDA;
  dim3 grid(ceil_div(N, BN), ceil_div(M, kBM * MT), batch);
  kern<<<grid, 128, smem, st>>>(ta, tb, tc, C, M, N, K, alpha, ctl);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int BN>
int dispatch_bn(const CUtensorMap& ta, const CUtensorMap& tb, void* C, int batch, int M, int N,
                int K, bool ak, bool bk, bool cf, float alpha, const KernelCtl& ctl,
                cudaStream_t st) {
#define ATTN_GEMM_CASE(AK, BK, CF)                                                    \
  if (ak == AK && bk == BK && cf == CF)                                               \
    return launch_variant<BN, AK, BK, CF>(ta, tb, C, batch, M, N, K, alpha, ctl, st);
  ATTN_GEMM_CASE(true, true, true)
  ATTN_GEMM_CASE(true, false, true)
  ATTN_GEMM_CASE(false, true, true)
  ATTN_GEMM_CASE(false, false, true)
  ATTN_GEMM_CASE(true, true, false)
  ATTN_GEMM_CASE(true, false, false)
  ATTN_GEMM_CASE(false, true, false)
  ATTN_GEMM_CASE(false, false, false)
#undef ATTN_GEMM_CASE
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace

int launch_gemm_bf16(const void* A, const void* B, void* C, int batch, int M, int N, int K,
                     bool a_kmajor, bool b_kmajor, bool c_f32, float alpha, const KernelCtl& ctl,
                     cudaStream_t st, int lda) {
  const int BN = N > 128 ? 256 : 128;
  CUtensorMap ta, tb;
  // A: K-major [b][M][K] (x = K) or MN-major [b][K][M] (x = M)
  bool ok = a_kmajor ? make_tmap_bf16(&ta, A, K, M, batch, 64, kBM, lda)
                     : make_tmap_bf16(&ta, A, M, K, batch, 64, kBK, lda);
  // B: K-major [b][N][K] (x = K) or MN-major [b][K][N] (x = N)
  ok = ok && (b_kmajor ? make_tmap_bf16(&tb, B, K, N, batch, 64, BN)
                       : make_tmap_bf16(&tb, B, N, K, batch, 64, kBK));
  if (!ok) return ATTN_ERR_CUDA;
  return BN == 256 ? dispatch_bn<256>(ta, tb, C, batch, M, N, K, a_kmajor, b_kmajor, c_f32, alpha,
                                      ctl, st)
                   : dispatch_bn<128>(ta, tb, C, batch, M, N, K, a_kmajor, b_kmajor, c_f32, alpha,
                                      ctl, st);
}

}  // namespace attn
