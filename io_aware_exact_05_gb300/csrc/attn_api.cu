// attn_api.cu -- the extern "C" entry points of libattn (declared in
// include/attn.h): argument checks, workspace carving and kernel dispatch.
#include <cmath>
#include <cstdint>
#include <initializer_list>

#include "kernels.h"

namespace attn {
int read_and_clear_status(cudaStream_t st);
}

using namespace attn;

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int H, int n, int d, float scale, int causal) {
  if (B < 1 || H < 1 || n < 1 || d < 1) return ATTN_ERR_INVALID_ARG;
  if ((long long)B * H > 65535) return ATTN_ERR_UNSUPPORTED;   // heads map to a grid dimension
  if (n > 65535 * 128) return ATTN_ERR_UNSUPPORTED;            // 128-row tiles map to grid.y
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

bool bf16_head_dim(int d) { return d == 64 || d == 128 || d == 256; }

// The automatic dQ mode spills dS^T only while that buffer stays below this.
constexpr size_t kSpillAutoMaxBytes = size_t(4) << 30;

// dQ mode actually used for a bf16 shape (measured choices).  d <= 128: the
// key-tile kernel's reduce-adds (1.21-1.38 x faster than the pass).  d = 256:
// the key-tile kernel has no tensor-memory columns for a dQ tile; the spill
// mode (dS^T through the workspace, one GEMM) takes 21 % less time than the pass
// where it applies (non-causal, dense, one key/value head per query head)
// and while its n x n buffer stays under kSpillAutoMaxBytes; else the pass.
attn_dq_mode resolve_mode(int B, int H, int H_kv, int n, int d, int causal, bool masked,
                          attn_dq_mode mode) {
  if (mode != ATTN_DQ_AUTO) return mode;
  if (d <= 128) return ATTN_DQ_ATOMIC;
  const size_t spill = (size_t)B * H * n * round_up(n, 8) * 2;
  if (d == 256 && !causal && !masked && H_kv == H && spill <= kSpillAutoMaxBytes)
    return ATTN_DQ_SPILL;
  return ATTN_DQ_PASS;
}

// CTAs per key/value head for the bf16 key-tile kernel.  A group of query
// heads shares one key/value head, so with few key/value heads the grid of
// (key tiles x key/value heads) CTAs can be smaller than the GPU; the group is
// then split over the smallest divisor of its size that brings the grid to
// two CTAs per SM (152 SMs), each part adding into fp32 dK/dV accumulators.
int group_split(int B, int H, int H_kv, int n, int d, attn_dtype dtype) {
  const int group = H / H_kv;
  if (dtype != ATTN_BF16 || group <= 1) return 1;
  const long long ctas = (long long)((n + 127) / 128) * B * H_kv * (d == 256 ? 2 : 1);
  int split = 1;
  for (int c = 2; c <= group && ctas * split < 2 * 152; ++c)
    if (group % c == 0) split = c;
  return split;
}

struct BwdWorkspace {
  float* lse2;
  float* delta;
  float* dq_acc;
  void* ds_t;      // bf16 [B*H][n][ld_ds] dS^T (ATTN_DQ_SPILL)
  int ld_ds;
  float* dk_acc;   // fp32 [B][H_kv][n][d] when gsplit > 1
  float* dv_acc;
  int gsplit;
  size_t bytes;
};

BwdWorkspace carve_bwd(void* base, int B, int H, int H_kv, int n, int d, attn_dtype dtype,
                       attn_dq_mode mode) {
  const int BH = B * H;
  BwdWorkspace w{};
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  if (dtype == ATTN_F32) {
    w.delta = reinterpret_cast<float*>(p);
    off = round_up((size_t)BH * n * 4, kAlign);
  } else {
    const size_t n_pad = round_up(n, 128);
    w.lse2 = reinterpret_cast<float*>(p + off);
    off += round_up((size_t)BH * n_pad * 4, kAlign);
    w.delta = reinterpret_cast<float*>(p + off);
    off += round_up((size_t)BH * n_pad * 4, kAlign);
    if (mode == ATTN_DQ_ATOMIC) {
      w.dq_acc = reinterpret_cast<float*>(p + off);
      off += round_up((size_t)BH * n * d * 4, kAlign);
    }
    if (mode == ATTN_DQ_SPILL) {
      w.ld_ds = (int)round_up(n, 8);
      w.ds_t = p + off;
      off += round_up((size_t)BH * n * w.ld_ds * 2, kAlign);
    }
    w.gsplit = group_split(B, H, H_kv, n, d, dtype);
    if (w.gsplit > 1) {
      const size_t kv_bytes = round_up((size_t)B * H_kv * n * d * 4, kAlign);
      w.dk_acc = reinterpret_cast<float*>(p + off);
      w.dv_acc = reinterpret_cast<float*>(p + off + kv_bytes);
      off += 2 * kv_bytes;
    }
  }
  if (w.gsplit < 1) w.gsplit = 1;
  w.bytes = off;
  return w;
}

struct MatWorkspace {
  float* s;        // S, later dP: fp32 [BH][n][n]
  void* p;         // P, later dS: bf16 [BH][n][n]
  float* delta;    // [BH][n]
  float* lse2;     // [BH][n]
  size_t bytes;
};

MatWorkspace carve_mat(void* base, int BH, int n) {
  MatWorkspace w{};
  uint8_t* p = static_cast<uint8_t*>(base);
  const size_t nn = (size_t)BH * n * n;
  size_t off = 0;
  w.s = reinterpret_cast<float*>(p + off);
  off += round_up(nn * 4, kAlign);
  w.p = p + off;
  off += round_up(nn * 2, kAlign);
  w.delta = reinterpret_cast<float*>(p + off);
  off += round_up((size_t)BH * n * 4, kAlign);
  w.lse2 = reinterpret_cast<float*>(p + off);
  off += round_up((size_t)BH * n * 4, kAlign);
  w.bytes = off;
  return w;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

}  // namespace

extern "C" {

// Tile lists of a block pattern for the forward's tiling (carved at `buf`).
static size_t fwd_lists_bytes(int n, int d) {
  int qr, qt, kvr;
  fwd_tiling(d, &qr, &qt, &kvr);
  return round_up(tile_lists_bytes(n, qr, qt, kvr), kAlign);
}
static TileLists build_lists(const uint8_t* mask, int n, int causal, bool outer_is_query, int osz,
                             int members, int isz, void* buf, cudaStream_t st, int* rc) {
  TileLists tl;
  const int nouter = ceil_div(n, osz * members), ninner = ceil_div(n, isz);
  int* lists = static_cast<int*>(buf);
  *rc = cuda_rc(launch_tile_lists(mask, n, causal, outer_is_query, osz, members, isz, lists, st));
  tl.lists = lists;
  tl.counts = lists + (size_t)nouter * ninner;
  tl.stride = ninner;
  return tl;
}

// Forward for H query heads sharing H_kv key/value heads; with `mask` a
// block-sparse pattern (bf16 lists carved from `lws`).
static int fwd_impl(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                    int H_kv, int n, int d, attn_dtype dtype, float scale, int causal,
                    const uint8_t* mask, void* lws, size_t lws_bytes, void* stream) {
  if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
    return ATTN_ERR_INVALID_ARG;
  int rc = check_common(B, H, n, d, scale, causal);
  if (rc) return rc;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  const HeadMap hm{H, H / H_kv};
  if (mask && H_kv != H) return ATTN_ERR_UNSUPPORTED;   // block-sparse: one K/V head per head
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  if (dtype == ATTN_F32) {
    if (d > 256) return ATTN_ERR_UNSUPPORTED;
    return cuda_rc(launch_fwd_f32(static_cast<const float*>(Q), static_cast<const float*>(K),
                                  static_cast<const float*>(V), static_cast<float*>(O), LSE, BH, hm,
                                  mask, n, d, scale, causal, st));
  }
  if (dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (!bf16_head_dim(d)) return ATTN_ERR_UNSUPPORTED;
  TileLists tl;
  if (mask) {
    if (!lws || (reinterpret_cast<uintptr_t>(lws) % kAlign) || lws_bytes < fwd_lists_bytes(n, d))
      return ATTN_ERR_WORKSPACE;
    int qr, qt, kvr;
    fwd_tiling(d, &qr, &qt, &kvr);
    tl = build_lists(mask, n, causal, true, qr, qt, kvr, lws, st, &rc);
    if (rc) return rc;
  }
  return launch_fwd_tc(Q, K, V, O, LSE, BH, hm, tl, n, d, scale, causal, default_ctl(), st);
}

int attn_fwd_gqa(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                 int H_kv, int n, int d, attn_dtype dtype, float scale, int causal, void* stream) {
  return fwd_impl(Q, K, V, O, LSE, B, H, H_kv, n, d, dtype, scale, causal, nullptr, nullptr, 0,
                  stream);
}

int attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
             int n, int d, attn_dtype dtype, float scale, int causal, void* stream) {
  return fwd_impl(Q, K, V, O, LSE, B, H, H, n, d, dtype, scale, causal, nullptr, nullptr, 0,
                  stream);
}

size_t attn_fwd_sparse_workspace_size(int n, int d) {
  if (n < 1 || d < 1 || d > 256) return 0;
  return fwd_lists_bytes(n, bf16_head_dim(d) ? d : 128);
}

int attn_fwd_sparse(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                    int H, int n, int d, attn_dtype dtype, float scale, int causal,
                    const unsigned char* block_mask, void* workspace, size_t workspace_bytes,
                    void* stream) {
  if (!block_mask) return ATTN_ERR_INVALID_ARG;
  return fwd_impl(Q, K, V, O, LSE, B, H, H, n, d, dtype, scale, causal, block_mask, workspace,
                  workspace_bytes, stream);
}

size_t attn_bwd_workspace_size(int B, int H, int n, int d, attn_dtype dtype, int causal,
                               attn_dq_mode mode) {
  if (check_common(B, H, n, d, 1.0f, causal) != ATTN_OK) return 0;
  if (dtype == ATTN_F32) {
    if (d > 256 || mode == ATTN_DQ_SPILL) return 0;
    return carve_bwd(nullptr, B, H, H, n, d, dtype, mode).bytes;
  }
  if (dtype != ATTN_BF16 || !bf16_head_dim(d)) return 0;
  const attn_dq_mode m = resolve_mode(B, H, H, n, d, causal, false, mode);
  if (m == ATTN_DQ_ATOMIC && d > 128) return 0;
  if (m == ATTN_DQ_SPILL && (d != 256 || causal)) return 0;
  return carve_bwd(nullptr, B, H, H, n, d, dtype, m).bytes;
}

size_t attn_bwd_gqa_workspace_size(int B, int H, int H_kv, int n, int d, attn_dtype dtype,
                                   int causal, attn_dq_mode mode) {
  if (H_kv < 1 || H % H_kv != 0) return 0;
  if (mode == ATTN_DQ_SPILL && H_kv != H) return 0;
  // the sizes of the grouped call's own mode (the automatic choice depends on H_kv)
  const attn_dq_mode m =
      dtype == ATTN_BF16 ? resolve_mode(B, H, H_kv, n, d, causal, false, mode) : mode;
  const size_t mha = attn_bwd_workspace_size(B, H, n, d, dtype, causal, m);
  if (mha == 0) return 0;
  return carve_bwd(nullptr, B, H, H_kv, n, d, dtype, m).bytes;
}

// Shared checks of the backward stages.  On success fills the resolved mode
// and the carved workspace.
static int bwd_setup(int B, int H, int H_kv, int n, int d, attn_dtype dtype, float scale,
                     int causal, attn_dq_mode mode, void* workspace, size_t workspace_bytes,
                     attn_dq_mode* resolved, BwdWorkspace* w) {
  int rc = check_common(B, H, n, d, scale, causal);
  if (rc) return rc;
  if (H_kv < 1 || H % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (mode != ATTN_DQ_AUTO && mode != ATTN_DQ_ATOMIC && mode != ATTN_DQ_PASS &&
      mode != ATTN_DQ_SPILL)
    return ATTN_ERR_INVALID_ARG;
  if (dtype == ATTN_F32) {
    if (d > 256) return ATTN_ERR_UNSUPPORTED;
    if (mode == ATTN_DQ_SPILL) return ATTN_ERR_UNSUPPORTED;
    *resolved = mode;
  } else if (dtype == ATTN_BF16) {
    if (!bf16_head_dim(d)) return ATTN_ERR_UNSUPPORTED;
    *resolved = resolve_mode(B, H, H_kv, n, d, causal, false, mode);
    if (*resolved == ATTN_DQ_ATOMIC && d > 128) return ATTN_ERR_UNSUPPORTED;
    if (*resolved == ATTN_DQ_SPILL && (d != 256 || causal || H_kv != H))
      return ATTN_ERR_UNSUPPORTED;
  } else {
    return ATTN_ERR_INVALID_ARG;
  }
  *w = carve_bwd(workspace, B, H, H_kv, n, d, dtype, *resolved);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) || workspace_bytes < w->bytes)
    return ATTN_ERR_WORKSPACE;
  return ATTN_OK;
}

static bool ptrs_ok(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (!p || !aligned16(p)) return false;
  return true;
}

int attn_fwd_fp8(const void* Q8, const void* K8, const void* Vt8, void* O, float* LSE, int B,
                 int H, int n, int d, float scale, const float* descale_q,
                 const float* descale_k, const float* descale_v, int causal, void* stream) {
  if (!ptrs_ok({Q8, K8, Vt8, O, LSE})) return ATTN_ERR_INVALID_ARG;
  for (const float* p : {descale_q, descale_k, descale_v})
    if (p && (reinterpret_cast<uintptr_t>(p) & 3u)) return ATTN_ERR_INVALID_ARG;
  int rc = check_common(B, H, n, d, scale, causal);
  if (rc) return rc;
  if (d != 128 || n % 16 != 0) return ATTN_ERR_UNSUPPORTED;
  return launch_fwd_fp8(Q8, K8, Vt8, O, LSE, B * H, n, scale, descale_q, descale_k, descale_v,
                        causal, default_ctl(), static_cast<cudaStream_t>(stream));
}

size_t attn_quantize_fp8_workspace_size(int BH, int n, int d) {
  if (BH < 1 || n < 1 || d != 128) return 0;
  return quant_fp8_workspace_bytes(BH, n);
}

int attn_quantize_fp8(const void* X, void* X8, float* descale, int BH, int n, int d,
                      int transpose, const float* signs, void* workspace, size_t workspace_bytes,
                      void* stream) {
  if (!ptrs_ok({X, X8}) || !descale || (reinterpret_cast<uintptr_t>(descale) & 3u))
    return ATTN_ERR_INVALID_ARG;
  if (signs && (reinterpret_cast<uintptr_t>(signs) & 3u)) return ATTN_ERR_INVALID_ARG;
  if (BH < 1 || n < 1 || d < 1 || (transpose != 0 && transpose != 1)) return ATTN_ERR_INVALID_ARG;
  if (transpose && signs) return ATTN_ERR_INVALID_ARG;   // V is never rotated
  if (BH > 65535) return ATTN_ERR_UNSUPPORTED;
  if (d != 128 || (transpose && n % 16 != 0)) return ATTN_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 3u) ||
      workspace_bytes < quant_fp8_workspace_bytes(BH, n))
    return ATTN_ERR_WORKSPACE;
  return cuda_rc(launch_quant_fp8(X, X8, descale, BH, n, transpose != 0, signs,
                                  static_cast<float*>(workspace),
                                  static_cast<cudaStream_t>(stream)));
}

int attn_bwd_preprocess(const void* O, const void* dO, const float* LSE, int B, int H, int n,
                        int d, attn_dtype dtype, int causal, attn_dq_mode mode, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (!ptrs_ok({O, dO, LSE})) return ATTN_ERR_INVALID_ARG;
  attn_dq_mode m;
  BwdWorkspace w;
  int rc = bwd_setup(B, H, H, n, d, dtype, 1.0f, causal, mode, workspace, workspace_bytes, &m, &w);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == ATTN_F32)
    return cuda_rc(launch_delta_f32(static_cast<const float*>(O), static_cast<const float*>(dO),
                                    w.delta, B * H, n, d, st));
  return cuda_rc(launch_delta_bf16(O, dO, LSE, w.delta, w.lse2,
                                   m == ATTN_DQ_ATOMIC ? w.dq_acc : nullptr, B * H, n,
                                   (int)round_up(n, 128), d, st));
}

// dK, dV stage (and the atomic dQ shares) for H query heads sharing H_kv
// key/value heads.
static int bwd_dkdv_impl(const void* Q, const void* K, const void* V, const void* dO, void* dK,
                         void* dV, int B, int H, int H_kv, int n, int d, attn_dtype dtype,
                         float scale, int causal, attn_dq_mode mode, void* workspace,
                         size_t workspace_bytes, void* stream, const TileLists& tl = TileLists()) {
  if (!ptrs_ok({Q, K, V, dO, dK, dV})) return ATTN_ERR_INVALID_ARG;
  attn_dq_mode m;
  BwdWorkspace w;
  int rc = bwd_setup(B, H, H_kv, n, d, dtype, scale, causal, mode, workspace, workspace_bytes, &m,
                     &w);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == ATTN_F32)
    return ATTN_ERR_INVALID_ARG;   // the fp32 dK/dV kernel needs LSE: use attn_bwd
  const size_t kv_elems = (size_t)B * H_kv * n * d;
  if (w.gsplit > 1) {   // split group: zero the fp32 dK/dV accumulators first
    if (cudaMemsetAsync(w.dk_acc, 0, kv_elems * 4, st) != cudaSuccess ||
        cudaMemsetAsync(w.dv_acc, 0, kv_elems * 4, st) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  if (m == ATTN_DQ_SPILL && tl.lists) return ATTN_ERR_UNSUPPORTED;
  rc = launch_bwd_kv_tc(Q, K, V, dO, w.lse2, w.delta, m == ATTN_DQ_ATOMIC ? w.dq_acc : nullptr, dK,
                        dV, w.dk_acc, w.dv_acc, B * H, HeadMap{H, H / H_kv}, w.gsplit, tl, n,
                        (int)round_up(n, 128), d, scale, causal, default_ctl(), st,
                        m == ATTN_DQ_SPILL ? w.ds_t : nullptr, w.ld_ds);
  if (rc || w.gsplit == 1) return rc;
  rc = cuda_rc(launch_dq_convert(w.dk_acc, dK, kv_elems, st));
  if (rc) return rc;
  return cuda_rc(launch_dq_convert(w.dv_acc, dV, kv_elems, st));
}

static int bwd_dq_impl(const void* Q, const void* K, const void* V, const void* dO, void* dQ, int B,
                       int H, int H_kv, int n, int d, attn_dtype dtype, float scale, int causal,
                       attn_dq_mode mode, void* workspace, size_t workspace_bytes, void* stream,
                       const TileLists& tl = TileLists()) {
  if (!ptrs_ok({dQ})) return ATTN_ERR_INVALID_ARG;
  attn_dq_mode m;
  BwdWorkspace w;
  int rc = bwd_setup(B, H, H_kv, n, d, dtype, scale, causal, mode, workspace, workspace_bytes, &m,
                     &w);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == ATTN_F32) return ATTN_ERR_INVALID_ARG;   // use attn_bwd
  if (m == ATTN_DQ_ATOMIC) return cuda_rc(launch_dq_convert(w.dq_acc, dQ, (size_t)B * H * n * d, st));
  if (m == ATTN_DQ_SPILL) {   // dQ = scale dS K: A = dS stored as dS^T rows (MN-major), B = K
    if (tl.lists) return ATTN_ERR_UNSUPPORTED;
    if (!ptrs_ok({K})) return ATTN_ERR_INVALID_ARG;
    return launch_gemm_bf16(w.ds_t, K, dQ, B * H, n, d, n, false, false, false, scale,
                            default_ctl(), st, w.ld_ds);
  }
  if (!ptrs_ok({Q, K, V, dO})) return ATTN_ERR_INVALID_ARG;
  return launch_bwd_q_tc(Q, K, V, dO, w.lse2, w.delta, dQ, B * H, HeadMap{H, H / H_kv}, tl, n,
                         (int)round_up(n, 128), d, scale, causal, default_ctl(), st);
}

int attn_bwd_dkdv(const void* Q, const void* K, const void* V, const void* dO, void* dK, void* dV,
                  int B, int H, int n, int d, attn_dtype dtype, float scale, int causal,
                  attn_dq_mode mode, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_dkdv_impl(Q, K, V, dO, dK, dV, B, H, H, n, d, dtype, scale, causal, mode, workspace,
                       workspace_bytes, stream);
}

int attn_bwd_dkdv_keys(const void* Q, const void* K, const void* V, const void* dO, void* dK,
                       void* dV, int B, int H, int n, int d, attn_dtype dtype, float scale,
                       int causal, attn_dq_mode mode, int key_rows, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (key_rows != 32 && key_rows != 64 && key_rows != 128) return ATTN_ERR_INVALID_ARG;
  if (!ptrs_ok({Q, K, V, dO, dK, dV})) return ATTN_ERR_INVALID_ARG;
  attn_dq_mode m;
  BwdWorkspace w;
  int rc = bwd_setup(B, H, H, n, d, dtype, scale, causal, mode, workspace, workspace_bytes, &m, &w);
  if (rc) return rc;
  if (dtype == ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (d <= 128 && m != ATTN_DQ_ATOMIC) return ATTN_ERR_UNSUPPORTED;
  if (m == ATTN_DQ_SPILL) return ATTN_ERR_UNSUPPORTED;   // study instances: dQ by the pass
  return launch_bwd_kv_study(Q, K, V, dO, w.lse2, w.delta, m == ATTN_DQ_ATOMIC ? w.dq_acc : nullptr,
                             dK, dV, B * H, key_rows, n, (int)round_up(n, 128), d, scale, causal,
                             default_ctl(), static_cast<cudaStream_t>(stream));
}

int attn_bwd_dq(const void* Q, const void* K, const void* V, const void* dO, void* dQ, int B,
                int H, int n, int d, attn_dtype dtype, float scale, int causal, attn_dq_mode mode,
                void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_dq_impl(Q, K, V, dO, dQ, B, H, H, n, d, dtype, scale, causal, mode, workspace,
                     workspace_bytes, stream);
}

// Bytes of the key-tile and query-tile lists of a block pattern (bf16).
static size_t bwd_lists_bytes(int n, int d) {
  int kr, qr, qr2, kr2;
  bwd_kv_tiling(d, &kr, &qr);
  bwd_q_tiling(d, &qr2, &kr2);
  return round_up(tile_lists_bytes(n, kr, 1, qr), kAlign) +
         round_up(tile_lists_bytes(n, qr2, 1, kr2), kAlign);
}

// Backward for H query heads sharing H_kv key/value heads; with `mask` a
// block-sparse pattern whose lists are carved from the workspace after the
// dense part.
static int bwd_impl(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                    const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int H_kv, int n,
                    int d, attn_dtype dtype, float scale, int causal, attn_dq_mode mode,
                    const uint8_t* mask, void* workspace, size_t workspace_bytes, void* stream) {
  if (!ptrs_ok({Q, K, V, O, dO, LSE, dQ, dK, dV})) return ATTN_ERR_INVALID_ARG;
  if (mask && H_kv != H) return ATTN_ERR_UNSUPPORTED;
  if (mask && mode == ATTN_DQ_SPILL) return ATTN_ERR_UNSUPPORTED;
  // one resolution for every stage below (the stage entry points resolve for
  // a dense, one-head-per-head call, which is not this call's shape)
  if (dtype == ATTN_BF16 && H_kv >= 1 && H % H_kv == 0)
    mode = resolve_mode(B, H, H_kv, n, d, causal, mask != nullptr, mode);
  attn_dq_mode m;
  BwdWorkspace w;
  int rc = bwd_setup(B, H, H_kv, n, d, dtype, scale, causal, mode, workspace, workspace_bytes, &m,
                     &w);
  if (rc) return rc;
  const HeadMap hm{H, H / H_kv};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  if (dtype == ATTN_F32) {
    const float *q = static_cast<const float*>(Q), *k = static_cast<const float*>(K),
                *v = static_cast<const float*>(V), *g = static_cast<const float*>(dO);
    rc = cuda_rc(launch_delta_f32(static_cast<const float*>(O), g, w.delta, BH, n, d, st));
    if (rc) return rc;
    rc = cuda_rc(launch_bwd_dkdv_f32(q, k, v, g, LSE, w.delta, static_cast<float*>(dK),
                                     static_cast<float*>(dV), BH, hm, mask, n, d, scale, causal,
                                     st));
    if (rc) return rc;
    return cuda_rc(launch_bwd_dq_f32(q, k, v, g, LSE, w.delta, static_cast<float*>(dQ), BH, hm,
                                     mask, n, d, scale, causal, st));
  }
  TileLists tl_kv, tl_q;
  if (mask) {
    if (workspace_bytes < w.bytes + bwd_lists_bytes(n, d)) return ATTN_ERR_WORKSPACE;
    uint8_t* lbase = static_cast<uint8_t*>(workspace) + w.bytes;
    int kr, qr;
    bwd_kv_tiling(d, &kr, &qr);
    tl_kv = build_lists(mask, n, causal, false, kr, 1, qr, lbase, st, &rc);
    if (rc) return rc;
    int qr2, kr2;
    bwd_q_tiling(d, &qr2, &kr2);
    tl_q = build_lists(mask, n, causal, true, qr2, 1, kr2,
                       lbase + round_up(tile_lists_bytes(n, kr, 1, qr), kAlign), st, &rc);
    if (rc) return rc;
  }
  rc = attn_bwd_preprocess(O, dO, LSE, B, H, n, d, dtype, causal, mode, workspace,
                           workspace_bytes, stream);
  if (rc) return rc;
  rc = bwd_dkdv_impl(Q, K, V, dO, dK, dV, B, H, H_kv, n, d, dtype, scale, causal, mode, workspace,
                     workspace_bytes, stream, tl_kv);
  if (rc) return rc;
  return bwd_dq_impl(Q, K, V, dO, dQ, B, H, H_kv, n, d, dtype, scale, causal, mode, workspace,
                     workspace_bytes, stream, tl_q);
}

int attn_bwd_gqa(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int H_kv, int n,
                 int d, attn_dtype dtype, float scale, int causal, attn_dq_mode mode,
                 void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, H_kv, n, d, dtype, scale, causal, mode,
                  nullptr, workspace, workspace_bytes, stream);
}

size_t attn_bwd_sparse_workspace_size(int B, int H, int n, int d, attn_dtype dtype, int causal,
                                      attn_dq_mode mode) {
  if (mode == ATTN_DQ_SPILL) return 0;
  if (dtype == ATTN_BF16) mode = resolve_mode(B, H, H, n, d, causal, true, mode);
  const size_t dense = attn_bwd_workspace_size(B, H, n, d, dtype, causal, mode);
  if (dense == 0) return 0;
  return dense + (dtype == ATTN_BF16 ? bwd_lists_bytes(n, d) : 0);
}

int attn_bwd_sparse(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                    const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int n, int d,
                    attn_dtype dtype, float scale, int causal, attn_dq_mode mode,
                    const unsigned char* block_mask, void* workspace, size_t workspace_bytes,
                    void* stream) {
  if (!block_mask) return ATTN_ERR_INVALID_ARG;
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, H, n, d, dtype, scale, causal, mode,
                  block_mask, workspace, workspace_bytes, stream);
}

int attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
             const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int n, int d,
             attn_dtype dtype, float scale, int causal, attn_dq_mode mode, void* workspace,
             size_t workspace_bytes, void* stream) {
  return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, H, n, d, dtype, scale, causal, mode,
                  nullptr, workspace, workspace_bytes, stream);
}

size_t attn_mat_workspace_size(int B, int H, int n, int d) {
  if (check_common(B, H, n, d, 1.0f, 0) != ATTN_OK) return 0;
  if (!bf16_head_dim(d) || (n % 8) != 0) return 0;
  return carve_mat(nullptr, B * H, n).bytes;
}

int attn_mat_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                 int n, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                 void* stream) {
  const void* ptrs[] = {Q, K, V, O, LSE};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return ATTN_ERR_INVALID_ARG;
  int rc = check_common(B, H, n, d, scale, causal);
  if (rc) return rc;
  if (!bf16_head_dim(d) || (n % 8) != 0) return ATTN_ERR_UNSUPPORTED;
  const int BH = B * H;
  MatWorkspace w = carve_mat(workspace, BH, n);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) || workspace_bytes < w.bytes)
    return ATTN_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const KernelCtl ctl = default_ctl();
  // S = scale * Q K^T            (A = Q K-major, B = K stored [n][d]: K-major)
  rc = launch_gemm_bf16(Q, K, w.s, BH, n, n, d, true, true, true, scale, ctl, st);
  if (rc) return rc;
  // P = softmax(S), LSE
  rc = cuda_rc(launch_mat_softmax(w.s, w.p, LSE, BH, n, scale, causal, st));
  if (rc) return rc;
  // O = P V                      (A = P K-major, B = V stored [K=n][N=d]: MN-major)
  return launch_gemm_bf16(w.p, V, O, BH, n, d, n, true, false, false, 1.0f, ctl, st);
}

int attn_mat_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int n, int d,
                 float scale, int causal, void* workspace, size_t workspace_bytes, void* stream) {
  const void* ptrs[] = {Q, K, V, O, dO, LSE, dQ, dK, dV};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return ATTN_ERR_INVALID_ARG;
  int rc = check_common(B, H, n, d, scale, causal);
  if (rc) return rc;
  if (!bf16_head_dim(d) || (n % 8) != 0) return ATTN_ERR_UNSUPPORTED;
  const int BH = B * H;
  MatWorkspace w = carve_mat(workspace, BH, n);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) || workspace_bytes < w.bytes)
    return ATTN_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const KernelCtl ctl = default_ctl();
  // dV = P^T dO                  (A = P^T: P stored [K=q][M=k], MN-major; B = dO MN-major)
  rc = launch_gemm_bf16(w.p, dO, dV, BH, n, d, n, false, false, false, 1.0f, ctl, st);
  if (rc) return rc;
  // dP = dO V^T                  (A = dO K-major, B = V stored [N=k][K=d]: K-major)
  rc = launch_gemm_bf16(dO, V, w.s, BH, n, n, d, true, true, true, 1.0f, ctl, st);
  if (rc) return rc;
  // D = rowsum(dO o O)
  rc = cuda_rc(launch_delta_bf16(O, dO, LSE, w.delta, w.lse2, nullptr, BH, n, n, d, st));
  if (rc) return rc;
  // dS = P o (dP - D), written over P
  rc = cuda_rc(launch_mat_dsoftmax(w.p, w.s, w.delta, w.p, BH, n, st));
  if (rc) return rc;
  // dQ = scale dS K              (A = dS K-major, B = K stored [K=k][N=d]: MN-major)
  rc = launch_gemm_bf16(w.p, K, dQ, BH, n, d, n, true, false, false, scale, ctl, st);
  if (rc) return rc;
  // dK = scale dS^T Q            (A = dS^T: MN-major, B = Q stored [K=q][N=d]: MN-major)
  return launch_gemm_bf16(w.p, Q, dK, BH, n, d, n, false, false, false, scale, ctl, st);
}

int attn_gemm_bf16(const void* A, const void* Bm, void* C, int batch, int M, int N, int K,
                   int a_kmajor, int b_kmajor, int c_f32, float alpha, void* stream) {
  if (!A || !Bm || !C || !aligned16(A) || !aligned16(Bm) || !aligned16(C))
    return ATTN_ERR_INVALID_ARG;
  if (batch < 1 || M < 1 || N < 1 || K < 1 || batch > 65535) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(alpha)) return ATTN_ERR_INVALID_ARG;
  if (K % 8) return ATTN_ERR_UNSUPPORTED;
  if (!a_kmajor && (M % 8)) return ATTN_ERR_UNSUPPORTED;
  if (!b_kmajor && (N % 8)) return ATTN_ERR_UNSUPPORTED;
  return launch_gemm_bf16(A, Bm, C, batch, M, N, K, a_kmajor != 0, b_kmajor != 0, c_f32 != 0,
                          alpha, default_ctl(), static_cast<cudaStream_t>(stream));
}

int attn_status(void* stream) { return read_and_clear_status(static_cast<cudaStream_t>(stream)); }

const char* attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "success";
    case ATTN_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, size, scale)";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape or head dimension for this path";
    case ATTN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case ATTN_ERR_CUDA: return "CUDA runtime or driver call failed";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a device-side barrier wait ran out of time";
    default: return "unknown status code";
  }
}

unsigned long long attn_launch_count(void) { return attn::launch_count(); }

int attn_selftest_wait_timeout(unsigned long long timeout_ns, void* stream) {
  if (timeout_ns < 1000ull || timeout_ns > 10000000000ull) return ATTN_ERR_INVALID_ARG;
  return cuda_rc(launch_wait_selftest(timeout_ns, static_cast<cudaStream_t>(stream)));
}

const char* attn_version(void) { return "libattn 0.1 (sm_103a)"; }

}  // extern "C"
