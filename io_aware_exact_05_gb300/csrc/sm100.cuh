// sm100.cuh -- inline-PTX building blocks for Blackwell (sm_100a/sm_103a):
// mbarriers with bounded waits, TMA tile loads, tcgen05 tensor-memory
// allocation, MMA issue/commit, and tensor-memory loads/stores.
//
// Operand layouts used throughout: bf16 tiles are staged by TMA with the
// 128-byte swizzle.  A "K-major" operand keeps the contraction index
// contiguous (rows of 64 elements = 128 B, eight rows = one 1024 B swizzle
// atom, atoms 1024 B apart); an "MN-major" operand keeps the M/N index
// contiguous (64 M/N elements per 128 B row, one row per k, atoms of eight
// k rows 1024 B apart, 64-wide M/N blocks `lbo` bytes apart).
#pragma once

#include <cstdint>
#include <cuda.h>

#include "common.cuh"

namespace attn {
namespace sm100 {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Warp index, broadcast from lane 0 so the compiler treats it (and what is
// derived from it) as warp-uniform: an MMA issuer whose loop runs on the whole
// warp keeps its descriptors in uniform registers.
__device__ __forceinline__ int warp_id_uniform() {
  return __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait.  Returns true when the phase with `parity` completed.  After
// `timeout_ns` of polling, or as soon as another thread of the CTA raised
// `*abort`, it records ATTN_ERR_DEVICE_TIMEOUT (first error wins) with the
// wait site, raises `*abort` and returns false: callers then leave their loop.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          const KernelCtl& ctl, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer();
  for (uint32_t spin = 1;; ++spin) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((spin & 255u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > ctl.timeout_ns) {
        record_error(ctl, ATTN_ERR_DEVICE_TIMEOUT, site);
        *abort = 1;
        return false;
      }
    }
  }
}

// Whole-warp forms (every lane waits; the result is the same on all lanes):
// for loops that a whole warp runs, such as an MMA issuer.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort,
                                               const KernelCtl& ctl, int site) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, ctl, site));
}

// ------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// 3-D tiled load (x innermost) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
// Plain bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 3-D tiled reduce-add of a shared-memory tile into global memory (the
// element type and the add come from the tensor map), tracked by the issuing
// thread's bulk async-group.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* m, uint32_t src, int x, int y,
                                                  int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%1, %2, %3}], [%4];" ::"l"(reinterpret_cast<uint64_t>(m)),
      "r"(x), "r"(y), "r"(z), "r"(src)
      : "memory");
}
// 3-D tiled store of a shared-memory tile to global memory (rows and columns
// outside the tensor are not written), tracked by the issuing thread's bulk
// async-group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int x, int y,
                                             int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group"
      " [%0, {%1, %2, %3}], [%4];" ::"l"(reinterpret_cast<uint64_t>(m)),
      "r"(x), "r"(y), "r"(z), "r"(src)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every committed bulk group of this thread has finished reading
// its shared-memory source.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until at most N of this thread's most recently committed bulk groups
// are still reading their shared-memory sources.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Named barrier over `count` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also ANDs `pred` over its `count` threads: threads that
// meet at later named barriers take the same branch after a bounded wait.
__device__ __forceinline__ bool named_bar_and(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
template <int NCOLS>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem) {
  static_assert(NCOLS >= 32 && NCOLS <= 512 && (NCOLS & (NCOLS - 1)) == 0, "tmem cols");
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(NCOLS)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <int NCOLS>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(NCOLS)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// MMA issue and commit helpers below are called by a whole converged warp;
// one lane, chosen by elect.sync, issues.  (Running the issue loop on the
// whole warp keeps its values warp-uniform; a loop under `lane == 0` pays a
// register-to-uniform move per descriptor and halves the MMA issue rate.)
//
// Arrive on `bar` once every tcgen05.mma issued so far by the elected lane is
// done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 accumulation.
// Bits: [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B
// format, 15 A MN-major, 16 B MN-major, [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::f8f6f4 with e4m3 A and B (format 0 at bits
// [7,10) and [10,13)), fp32 accumulation, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.  Start address, leading
// byte offset and stride byte offset are stored >> 4; bit 46 is the fixed
// descriptor version; bits [61,64) = 2 select the 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Four MMAs of one K-block group, issued back to back from one asm block so
// no other instruction lands between them.  Descriptors are passed as 32-bit
// halves: lo[i] (start address and leading offset, which vary per MMA) and hi
// (stride offset, version and swizzle, shared).  The first MMA accumulates
// iff acc != 0; the other three always accumulate.
#define ATTN_MMA_SS_X4(NAME, CG, KIND)                                                           \
  __device__ __forceinline__ void NAME(uint32_t d, const uint32_t(&alo)[4], uint32_t ahi,       \
                                       const uint32_t(&blo)[4], uint32_t bhi, uint32_t idesc,   \
                                       uint32_t acc) {                                          \
    asm volatile(                                                                               \
        "{\n\t.reg .pred p, t, e;\n\t.reg .b64 a0, a1, a2, a3, b0, b1, b2, b3;\n\t"             \
        "elect.sync _|e, 0xffffffff;\n\t"                                                        \
        "setp.ne.b32 p, %12, 0;\n\tsetp.eq.b32 t, %12, %12;\n\t"                                \
        "mov.b64 a0, {%1, %9};\n\tmov.b64 a1, {%2, %9};\n\t"                                    \
        "mov.b64 a2, {%3, %9};\n\tmov.b64 a3, {%4, %9};\n\t"                                    \
        "mov.b64 b0, {%5, %10};\n\tmov.b64 b1, {%6, %10};\n\t"                                  \
        "mov.b64 b2, {%7, %10};\n\tmov.b64 b3, {%8, %10};\n\t"                                  \
        "@e tcgen05.mma.cta_group::" CG ".kind::" KIND " [%0], a0, b0, %11, p;\n\t"                     \
        "@e tcgen05.mma.cta_group::" CG ".kind::" KIND " [%0], a1, b1, %11, t;\n\t"                     \
        "@e tcgen05.mma.cta_group::" CG ".kind::" KIND " [%0], a2, b2, %11, t;\n\t"                     \
        "@e tcgen05.mma.cta_group::" CG ".kind::" KIND " [%0], a3, b3, %11, t;\n\t}\n" ::"r"(d),        \
        "r"(alo[0]), "r"(alo[1]), "r"(alo[2]), "r"(alo[3]), "r"(blo[0]), "r"(blo[1]),           \
        "r"(blo[2]), "r"(blo[3]), "r"(ahi), "r"(bhi), "r"(idesc), "r"(acc)                      \
        : "memory");                                                                            \
  }
ATTN_MMA_SS_X4(mma_ss_x4, "1", "f16")
ATTN_MMA_SS_X4(mma_ss_x4_f8, "1", "f8f6f4")   // e4m3 operands: 32 per MMA along K
#undef ATTN_MMA_SS_X4

// Same with A read from tensor memory: A of MMA i starts at column a_tmem + 8 i
// (sixteen bf16 values of K per MMA, two per 32-bit column).
#define ATTN_MMA_TS_X4(NAME, CG, KIND)                                                           \
  __device__ __forceinline__ void NAME(uint32_t d, uint32_t a_tmem, const uint32_t(&blo)[4],    \
                                       uint32_t bhi, uint32_t idesc, uint32_t acc) {            \
    asm volatile(                                                                               \
        "{\n\t.reg .pred p, t, e;\n\t.reg .b64 b0, b1, b2, b3;\n\t.reg .b32 x1, x2, x3;\n\t"    \
        "elect.sync _|e, 0xffffffff;\n\t"                                                        \
        "setp.ne.b32 p, %7, 0;\n\tsetp.eq.b32 t, %7, %7;\n\t"                                   \
        "mov.b64 b0, {%2, %6};\n\tmov.b64 b1, {%3, %6};\n\t"                                    \
        "mov.b64 b2, {%4, %6};\n\tmov.b64 b3, {%5, %6};\n\t"                                    \
        "add.u32 x1, %1, 8;\n\tadd.u32 x2, %1, 16;\n\tadd.u32 x3, %1, 24;\n\t"                  \
        "@e tcgen05.mma.cta_group::" CG ".kind::" KIND " [%0], [%1], b0, %8, p;\n\t"                    \
        "@e tcgen05.mma.cta_group::" CG ".kind::" KIND " [%0], [x1], b1, %8, t;\n\t"                    \
        "@e tcgen05.mma.cta_group::" CG ".kind::" KIND " [%0], [x2], b2, %8, t;\n\t"                    \
        "@e tcgen05.mma.cta_group::" CG ".kind::" KIND " [%0], [x3], b3, %8, t;\n\t}\n" ::"r"(d),       \
        "r"(a_tmem), "r"(blo[0]), "r"(blo[1]), "r"(blo[2]), "r"(blo[3]), "r"(bhi), "r"(acc),    \
        "r"(idesc)                                                                              \
        : "memory");                                                                            \
  }
ATTN_MMA_TS_X4(mma_ts_x4, "1", "f16")
// e4m3 A from tensor memory: four values per 32-bit column, so the eight
// columns per MMA again hold its 32 values of K
ATTN_MMA_TS_X4(mma_ts_x4_f8, "1", "f8f6f4")
#undef ATTN_MMA_TS_X4

// Four bf16 MMAs with A from tensor memory at columns a, a + 8, a + H and
// a + H + 8: a 64-wide K range held as two 16-column halves H columns apart
// (P^T or dS^T of a 64-query tile, each half written by its own warpgroup).
template <int H>
__device__ __forceinline__ void mma_ts_x4_halves(uint32_t d, uint32_t a_tmem,
                                                 const uint32_t (&blo)[4], uint32_t bhi,
                                                 uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, t, e;\n\t.reg .b64 b0, b1, b2, b3;\n\t.reg .b32 x1, x2, x3;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %7, 0;\n\tsetp.eq.b32 t, %7, %7;\n\t"
      "mov.b64 b0, {%2, %6};\n\tmov.b64 b1, {%3, %6};\n\t"
      "mov.b64 b2, {%4, %6};\n\tmov.b64 b3, {%5, %6};\n\t"
      "add.u32 x1, %1, 8;\n\tadd.u32 x2, %1, %9;\n\tadd.u32 x3, %1, %10;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], b0, %8, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [x1], b1, %8, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [x2], b2, %8, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [x3], b3, %8, t;\n\t}\n" ::"r"(d),
      "r"(a_tmem), "r"(blo[0]), "r"(blo[1]), "r"(blo[2]), "r"(blo[3]), "r"(bhi), "r"(acc),
      "r"(idesc), "n"(H), "n"(H + 8)
      : "memory");
}

// Low and high 32-bit halves of the 128-byte-swizzle shared-memory descriptor
// (same fields as sdesc_sw128).
__host__ __device__ constexpr uint32_t sdesc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t sdesc_hi(uint32_t sbo) {
  return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}

// Tensor memory <-> registers, shape 32x32b: thread t of the warp moves lane
// (base lane + t), N consecutive 32-bit columns.
#define ATTN_R8(a, o) "=r"(a[o + 0]), "=r"(a[o + 1]), "=r"(a[o + 2]), "=r"(a[o + 3]), \
    "=r"(a[o + 4]), "=r"(a[o + 5]), "=r"(a[o + 6]), "=r"(a[o + 7])
#define ATTN_W8(a, o) "r"(a[o + 0]), "r"(a[o + 1]), "r"(a[o + 2]), "r"(a[o + 3]), \
    "r"(a[o + 4]), "r"(a[o + 5]), "r"(a[o + 6]), "r"(a[o + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : ATTN_R8(r, 0), ATTN_R8(r, 8), ATTN_R8(r, 16), ATTN_R8(r, 24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      ATTN_W8(r, 0), ATTN_W8(r, 8)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      ATTN_W8(r, 0), ATTN_W8(r, 8), ATTN_W8(r, 16), ATTN_W8(r, 24)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// After tcgen05.wait::ld: make every later use of these registers depend on
// an instruction that follows the wait, so no use is scheduled before it.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}

// ----------------------------------------------------------- small helpers
// Four floats to e4m3 (round to nearest, saturating), byte i = value i.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  unsigned short lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ void red_add_v4(float* gptr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(gptr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// Byte offset of the 16-byte chunk `chunk` (0..7) of row `row` inside a
// 128-byte-swizzled region whose rows are 128 bytes apart.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// Copies a 128-row bf16 tile held in shared memory as D/64 128-byte-swizzled
// boxes of [128 rows][64 columns] into tensor memory as an MMA A operand
// (lane = row, two consecutive elements per 32-bit column, D/2 columns from
// `tcol`).  Run by one warpgroup: thread r copies row r.
template <int D>
__device__ __forceinline__ void tile_to_tmem(const uint8_t* tile, uint32_t tcol, int r) {
#pragma unroll
  for (int kb = 0; kb < D / 64; ++kb) {
    const uint8_t* box = tile + kb * (128 * 128);
    uint32_t w[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(box + sw128_offset(r, c));
      w[4 * c] = v.x;
      w[4 * c + 1] = v.y;
      w[4 * c + 2] = v.z;
      w[4 * c + 3] = v.w;
    }
    tmem_st32(tcol + 32 * kb, w);
  }
  tmem_st_wait();
}

}  // namespace sm100
}  // namespace attn
