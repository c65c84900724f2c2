// common.cuh -- shared host/device definitions for libattn.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/attn.h"

namespace attn {

// Query heads -> key/value heads (grouped-query attention, "Flash Attention:
// Revolutionizing Transformer Efficiency", section FlashAttention-2, item 3):
// query head h of batch b reads key/value head h / group of the same batch;
// there are H / group key/value heads per batch (group = 1: one per query
// head, group = H: a single shared one).  Indices are flat b * heads + h.
struct HeadMap {
  int H;       // query heads per batch
  int group;   // query heads per key/value head (divides H)
  __host__ __device__ int hkv() const { return H / group; }
  __host__ __device__ int kv_of(int bh) const { return (bh / H) * (H / group) + (bh % H) / group; }
  __host__ __device__ int q_of(int bkv, int i) const {
    return (bkv / (H / group)) * H + (bkv % (H / group)) * group + i;
  }
};

// Passed by value to every kernel that waits on a barrier.
struct KernelCtl {
  int* err;              // device status word: [0] = first error code, [1] = site
  uint64_t timeout_ns;   // limit for any single barrier wait
};

__device__ __forceinline__ void record_error(const KernelCtl& c, int code, int site) {
  if (atomicCAS(c.err, 0, code) == 0) c.err[1] = site;
}

// Wait-site identifiers reported with ATTN_ERR_DEVICE_TIMEOUT (status word [1]).
enum WaitSite : int {
  SITE_FWD_LOAD_Q = 101,
  SITE_FWD_KV_EMPTY = 102,
  SITE_FWD_K_FULL = 103,
  SITE_FWD_V_FULL = 104,
  SITE_FWD_S_FULL = 105,
  SITE_FWD_P_FULL = 106,
  SITE_FWD_O_DONE = 107,
  SITE_FWD_S_FREE = 108,
  SITE_BWD_KV = 201,
  SITE_BWD_Q_EMPTY = 202,
  SITE_BWD_Q_FULL = 203,
  SITE_BWD_S_FULL = 204,
  SITE_BWD_DP_FULL = 205,
  SITE_BWD_P_READY = 206,
  SITE_BWD_DS_READY = 207,
  SITE_BWD_DQ_FULL = 208,
  SITE_BWD_DQ_FREE = 209,
  SITE_BWD_ACC_DONE = 210,
  SITE_BWD_DS_FREE = 211,
  SITE_BWD_SMEM_ALIGN = 212,   // shared-memory base not 1024-byte aligned (not a wait)
  SITE_BWD_S_READ = 213,       // the compute warps have taken S into registers
  SITE_GEMM_FULL = 301,
  SITE_GEMM_EMPTY = 302,
  SITE_GEMM_ACC = 303,
  SITE_SELFTEST = 901,
};

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace attn
