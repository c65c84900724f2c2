// sparse.cu -- tile lists of a block-sparse attention pattern.
//
// A block pattern keeps or drops 128 x 128 blocks of the score matrix
// (sparse attention over a block pattern: "Chapter 3.1 -- The cost of
// attention", section 3, Longformer's local windows and global tokens and
// BigBird's random links; "On the fine-grained I/O complexity of attention
// backward passes", item 2, sparse attention with Z_QK kept entries).  The
// tiled kernels walk, for each of their outer units (a CTA's query tiles, or
// a key tile), only the inner tiles that meet a kept block.  This kernel
// writes those lists: for outer unit u, lists[u * stride + p] for p < counts[u]
// are the inner tile indices in increasing order (low 16 bits), each with one
// bit per member tile of the unit (bit 16 + m) saying whether member m's
// rows meet a kept block of that inner tile and, when causal, a key at or
// below a row.  A unit is `members` consecutive tiles of `osz` rows; inner
// tiles have `isz` rows.  outer_is_query selects which side is the query.
// One block per outer unit builds its list in parallel over the inner tiles.
#include "kernels.h"

namespace attn {
namespace {

__device__ __forceinline__ bool range_kept(const uint8_t* __restrict__ mask, int nb, int q_lo,
                                           int q_hi, int k_lo, int k_hi, int causal) {
  // rows [q_lo, q_hi) x keys [k_lo, k_hi), both non-empty
  if (causal && q_hi - 1 < k_lo) return false;
  for (int bq = q_lo / 128; bq <= (q_hi - 1) / 128; ++bq)
    for (int bk = k_lo / 128; bk <= (k_hi - 1) / 128; ++bk)
      if (mask[(size_t)bq * nb + bk]) return true;
  return false;
}

// One block per outer unit; its threads take the inner tiles in chunks of
// kListThreads and write the kept ones in increasing order (ballot within a
// warp, warp totals through shared memory for the order across warps).
constexpr int kListThreads = 128;

__global__ void __launch_bounds__(kListThreads)
tile_lists_kernel(const uint8_t* __restrict__ mask, int n, int causal, int outer_is_query,
                  int osz, int members, int isz, int* __restrict__ lists,
                  int* __restrict__ counts, int stride) {
  __shared__ int warp_tot[kListThreads / 32];
  const int u = blockIdx.x;
  const int nb = (n + 127) / 128;
  const int ninner = (n + isz - 1) / isz;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int base = 0;
  for (int t0 = 0; t0 < ninner; t0 += kListThreads) {
    const int t = t0 + (int)threadIdx.x;
    int bits = 0;
    if (t < ninner) {
      const int i_lo = t * isz, i_hi = min(n, i_lo + isz);
      for (int m = 0; m < members; ++m) {
        const int o_lo = (u * members + m) * osz;
        if (o_lo >= n) break;
        const int o_hi = min(n, o_lo + osz);
        const bool kept = outer_is_query ? range_kept(mask, nb, o_lo, o_hi, i_lo, i_hi, causal)
                                         : range_kept(mask, nb, i_lo, i_hi, o_lo, o_hi, causal);
        if (kept) bits |= 1 << m;
      }
    }
    const unsigned kept_lanes = __ballot_sync(0xffffffffu, bits != 0);
    if (lane == 0) warp_tot[warp] = __popc(kept_lanes);
    __syncthreads();
    int off = base, chunk = 0;
#pragma unroll
    for (int w = 0; w < kListThreads / 32; ++w) {
      if (w < warp) off += warp_tot[w];
      chunk += warp_tot[w];
    }
    if (bits) lists[(size_t)u * stride + off + __popc(kept_lanes & ((1u << lane) - 1u))] =
        t | (bits << 16);
    __syncthreads();   // warp_tot is rewritten by the next chunk
    base += chunk;
  }
  if (threadIdx.x == 0) counts[u] = base;
}

}  // namespace

size_t tile_lists_bytes(int n, int osz, int members, int isz) {
  const size_t nouter = (n + (size_t)osz * members - 1) / ((size_t)osz * members);
  const size_t ninner = (n + (size_t)isz - 1) / isz;
  return (nouter * ninner + nouter) * sizeof(int);
}

cudaError_t launch_tile_lists(const uint8_t* mask, int n, int causal, bool outer_is_query, int osz,
                              int members, int isz, int* buf, cudaStream_t st) {
  const int nouter = (n + osz * members - 1) / (osz * members);
  const int ninner = (n + isz - 1) / isz;
  int* lists = buf;
  int* counts = buf + (size_t)nouter * ninner;
  tile_lists_kernel<<<nouter, kListThreads, 0, st>>>(mask, n, causal, outer_is_query ? 1 : 0, osz,
                                                     members, isz, lists, counts, ninner);
  note_launch();
  return cudaGetLastError();
}

}  // namespace attn
