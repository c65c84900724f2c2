// bwd_noalloc.cu -- attn_bwd_noalloc: the backward pass without a workspace.
//
// Some callers cannot hand the library a workspace.  A host program may own
// only the tensors it passes in and have no device allocator to draw extra
// memory from.  A runtime may fix its device-memory budget at start-up and
// forbid any allocation afterwards.  Other callers must not call cudaMalloc
// where they call the backward, because cudaMalloc can block the host thread
// or synchronise the device.  For them this entry point keeps the backward's
// scratch (the log2-scaled LSE and D = rowsum(dO o O) row statistics) in a
// file-scope device array that exists as soon as the library is loaded, and it
// allocates nothing itself.
//
// Limits and sharing rules:
//   * The array holds kScratchBytes = 16 MiB on every GPU that loads the
//     library, for the life of the process.
//   * bf16 needs 8 * B*H*n_pad bytes (n_pad = n rounded up to 128), i.e.
//     B*H*n_pad <= 2,097,152; fp32 needs 4 * B*H*n bytes.  Larger problems are
//     rejected with ATTN_ERR_WORKSPACE before anything is launched.
//   * Every call uses the same array and leaves its contents behind.  Each
//     call writes all of the scratch it reads before reading it (the
//     preprocessing kernel fills every row, padding included), so nothing has
//     to start at zero.
//   * Calls whose work overlaps on the GPU (two streams, or two host threads
//     without ordering between them) race on the array: issue them on one
//     stream, or synchronise in between.
//   * The first call on each device looks up the array's device address with
//     that device current.  Make that first call before capturing any stream.
//     The address is cached under the id of the current CUDA context, so
//     after cudaDeviceReset, or with another context made current on the
//     device, the next call looks the address up again instead of using a
//     stale one.
//
// The computation is the dQ-pass backward: preprocessing kernel, key-tile
// kernel (dK, dV), query-tile kernel (dQ); bf16 results equal those of attn_bwd
// with ATTN_DQ_PASS.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "kernels.h"

namespace attn {
namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;

// Host code must never pass this name to a kernel: on the host it denotes a
// host-side stand-in, not the device address.  Use noalloc_scratch().
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};

// Device address of the scratch array in the current context: looked up once
// per device, and again when the device's current context is not the one the
// cached address belongs to.  nullptr if the lookup fails.
void* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return nullptr;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = current_context_id();   // the lookup made the context current
  }
  return g_scratch_ptr[dev];
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool ok_ptr(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                                const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                                int B, int H, int n, int d, attn_dtype dtype, float scale,
                                int causal, void* stream) {
  const void* ptrs[] = {Q, K, V, O, dO, LSE, dQ, dK, dV};
  for (const void* p : ptrs)
    if (!ok_ptr(p)) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || n < 1 || d < 1) return ATTN_ERR_INVALID_ARG;
  if ((long long)B * H > 65535) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || (causal != 0 && causal != 1)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_BF16 && dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (dtype == ATTN_BF16 && d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (dtype == ATTN_F32 && d > 256) return ATTN_ERR_UNSUPPORTED;

  const size_t BH = (size_t)B * H;
  const size_t n_pad = round_up((size_t)n, 128);
  const size_t stat_bytes = round_up(BH * (dtype == ATTN_BF16 ? n_pad : (size_t)n) * 4, 256);
  const size_t need = dtype == ATTN_BF16 ? 2 * stat_bytes : stat_bytes;
  if (need > kScratchBytes) return ATTN_ERR_WORKSPACE;

  const HeadMap hm{H, 1};
  uint8_t* base = static_cast<uint8_t*>(noalloc_scratch());
  if (!base) return ATTN_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  if (dtype == ATTN_F32) {
    float* delta = reinterpret_cast<float*>(base);
    const float *q = static_cast<const float*>(Q), *k = static_cast<const float*>(K),
                *v = static_cast<const float*>(V), *g = static_cast<const float*>(dO);
    if (launch_delta_f32(static_cast<const float*>(O), g, delta, (int)BH, n, d, st) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (launch_bwd_dkdv_f32(q, k, v, g, LSE, delta, static_cast<float*>(dK),
                            static_cast<float*>(dV), (int)BH, hm, nullptr, n, d, scale, causal,
                            st) != cudaSuccess)
      return ATTN_ERR_CUDA;
    return launch_bwd_dq_f32(q, k, v, g, LSE, delta, static_cast<float*>(dQ), (int)BH, hm, nullptr,
                             n, d, scale, causal, st) == cudaSuccess
               ? ATTN_OK
               : ATTN_ERR_CUDA;
  }

  float* lse2 = reinterpret_cast<float*>(base);
  float* delta = reinterpret_cast<float*>(base + stat_bytes);
  const KernelCtl ctl = default_ctl();
  if (launch_delta_bf16(O, dO, LSE, delta, lse2, nullptr, (int)BH, n, (int)n_pad, d, st) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  int rc = launch_bwd_kv_tc(Q, K, V, dO, lse2, delta, nullptr, dK, dV, nullptr, nullptr, (int)BH,
                            hm, 1, TileLists(), n, (int)n_pad, d, scale, causal, ctl, st);
  if (rc) return rc;
  return launch_bwd_q_tc(Q, K, V, dO, lse2, delta, dQ, (int)BH, hm, TileLists(), n, (int)n_pad, d,
                         scale, causal, ctl, st);
}
