// bwd_kv128.cu -- the key-tile backward (bwd_kv.cuh) for head dim 128.
#include "bwd_kv.cuh"

namespace attn {

int launch_bwd_kv128_tc(const void* Q, const void* K, const void* V, const void* dO,
                        const float* LSE2, const float* Dv, float* dQacc, void* dK, void* dV,
                        float* dKacc, float* dVacc, int BH, const HeadMap& hm, int gsplit,
                        const TileLists& tl, int n, int n_pad, float scale, int causal,
                        const KernelCtl& ctl, cudaStream_t st) {
  ATTN_KV_DISPATCH(128);
}

}  // namespace attn
