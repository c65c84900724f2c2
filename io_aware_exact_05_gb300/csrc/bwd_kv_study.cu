// bwd_kv_study.cu -- instances of the key-tile backward (bwd_kv.cuh) whose
// CTAs own 64 or 32 of their 128 key rows, for the IO study of the backward
// ("On the fine-grained I/O complexity of attention backward passes",
// Theorem 1.1: with a cache of M words the tiled backward moves
// Theta((n^2 d^2 + n d^3) / M); here M is set by the keys a CTA keeps).
#include "bwd_kv.cuh"

namespace attn {

int launch_bwd_kv_study_d64_128(const void* Q, const void* K, const void* V, const void* dO,
                                const float* LSE2, const float* Dv, float* dQacc, void* dK,
                                void* dV, int BH, int key_rows, int n, int n_pad, int d,
                                float scale, int causal, const KernelCtl& ctl, cudaStream_t st) {
  if (!dQacc) return ATTN_ERR_INVALID_ARG;
  const HeadMap hm{BH, 1};
#define ATTN_KVS(DD, KRR)                                                                      \
  return launch_kv<DD, true, false, false, KRR>(Q, K, V, dO, LSE2, Dv, dQacc, dK, dV, nullptr,  \
                                                nullptr, BH, hm, 1, TileLists(), n, n_pad,      \
                                                scale, causal, ctl, st)
  if (d == 64) {
    switch (key_rows) {
      case 128:   // the product instance
        return launch_bwd_kv64_tc(Q, K, V, dO, LSE2, Dv, dQacc, dK, dV, nullptr, nullptr, BH, hm,
                                  1, TileLists(), n, n_pad, scale, causal, ctl, st);
      case 64: ATTN_KVS(64, 64);
      case 32: ATTN_KVS(64, 32);
      default: return ATTN_ERR_INVALID_ARG;
    }
  }
  if (d == 128) {
    switch (key_rows) {
      case 128:
        return launch_bwd_kv128_tc(Q, K, V, dO, LSE2, Dv, dQacc, dK, dV, nullptr, nullptr, BH,
                                   hm, 1, TileLists(), n, n_pad, scale, causal, ctl, st);
      case 64: ATTN_KVS(128, 64);
      case 32: ATTN_KVS(128, 32);
      default: return ATTN_ERR_INVALID_ARG;
    }
  }
#undef ATTN_KVS
  return ATTN_ERR_UNSUPPORTED;
}

}  // namespace attn
