// selftest.cu -- checks that device-side failure detection reaches the host.
//
// Every barrier wait of the library's kernels is bounded (mbar_wait): after
// KernelCtl::timeout_ns it records ATTN_ERR_DEVICE_TIMEOUT and the wait site
// in the device status word, raises the CTA's abort flag and returns, so a
// kernel whose partner never arrives ends instead of hanging, and the host
// reads the code with attn_status().  This kernel exercises exactly that
// path: one thread waits on an mbarrier that nothing arrives at.  There is no
// fault and no hang: the wait ends after timeout_ns and the kernel returns.
#include "kernels.h"
#include "sm100.cuh"

namespace attn {
namespace {

using namespace sm100;

__global__ void wait_selftest_kernel(KernelCtl ctl) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  volatile int abort_flag = 0;
  mbar_wait(b, 0, &abort_flag, ctl, SITE_SELFTEST);   // phase 0 never completes
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t st) {
  KernelCtl c = default_ctl();
  c.timeout_ns = timeout_ns;
  wait_selftest_kernel<<<1, 32, 0, st>>>(c);
  note_launch();
  return cudaGetLastError();
}

}  // namespace attn
