// host.cu -- host-side helpers: TMA tensor-map encoding and the device status
// word shared by every kernel of the library.
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "kernels.h"

namespace attn {

// Kernels the library has launched in this process.
static std::atomic<unsigned long long> g_launches{0};

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

unsigned long long launch_count() { return g_launches.load(std::memory_order_relaxed); }

// First device-side error: [0] = attn_status_t code, [1] = wait site.
__device__ int g_status_word[2];

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

using PFN_ctx_get_current = CUresult (*)(CUcontext*);
using PFN_ctx_get_id = CUresult (*)(CUcontext, unsigned long long*);

template <class F>
F driver_fn(const char* name, int version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<F>(p);
  return nullptr;
}

}  // namespace

unsigned long long current_context_id() {
  static PFN_ctx_get_current get_current = nullptr;
  static PFN_ctx_get_id get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_current = driver_fn<PFN_ctx_get_current>("cuCtxGetCurrent", 4000);
    get_id = driver_fn<PFN_ctx_get_id>("cuCtxGetId", 12000);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;   // none yet: the runtime binds its context at its first real call
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t x, uint64_t y, uint64_t z,
                    uint32_t box_x, uint32_t box_y, uint64_t ld) {
  auto fn = encode_fn();
  if (!fn) return false;
  if (ld == 0) ld = x;
  const cuuint64_t dims[3] = {x, y, z};
  const cuuint64_t strides[2] = {ld * 2, ld * y * 2};   // bytes, dims 1..2
  const cuuint32_t box[3] = {box_x, box_y, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_u8(CUtensorMap* map, const void* base, uint64_t x, uint64_t y, uint64_t z,
                  uint32_t box_x, uint32_t box_y) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {x, y, z};
  const cuuint64_t strides[2] = {x, x * y};   // bytes, dims 1..2
  const cuuint32_t box[3] = {box_x, box_y, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_f32(CUtensorMap* map, const void* base, uint64_t x, uint64_t y, uint64_t z,
                   uint32_t box_x, uint32_t box_y, bool sw128) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {x, y, z};
  const cuuint64_t strides[2] = {x * 4, x * y * 4};
  const cuuint32_t box[3] = {box_x, box_y, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Address of the status word in the current context, looked up once per
// device and again whenever that device's current context changes (after a
// device reset the module is loaded again, possibly at another address).
static int* status_word_ptr() {
  static int* ptrs[64] = {nullptr};
  static unsigned long long ctx_ids[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev] || ctx == 0 || ctx != ctx_ids[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
    ctx_ids[dev] = current_context_id();   // the lookup made the context current
  }
  return ptrs[dev];
}

static uint64_t g_timeout_ns = 2000000000ull;   // 2 s per barrier wait

KernelCtl default_ctl() {
  KernelCtl c;
  c.err = status_word_ptr();
  c.timeout_ns = g_timeout_ns;
  return c;
}

int read_and_clear_status(cudaStream_t st) {
  if (cudaStreamSynchronize(st) != cudaSuccess) return ATTN_ERR_CUDA;
  int* p = status_word_ptr();
  if (!p) return ATTN_ERR_CUDA;
  int h[2] = {0, 0};
  if (cudaMemcpy(h, p, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (h[0] != 0) {
    const int z[2] = {0, 0};
    if (cudaMemcpy(p, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return h[0];
}

}  // namespace attn
