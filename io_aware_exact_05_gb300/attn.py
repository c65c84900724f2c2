"""ctypes binding of libattn (include/attn.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libattn.so``.  Functions keep the C names and take torch tensors
(device memory, contiguous [B, H, n, d]) plus the current CUDA stream.  If the
library is missing, every call raises: there is no fallback implementation.
"""

import ctypes
import os
import threading

import torch

__all__ = [
    "ATTN_BF16", "ATTN_F32", "ATTN_DQ_AUTO", "ATTN_DQ_ATOMIC", "ATTN_DQ_PASS", "ATTN_DQ_SPILL",
    "AttnError", "lib", "lib_path",
    "attn_fwd", "attn_bwd", "attn_bwd_workspace_size",
    "attn_bwd_preprocess", "attn_bwd_dkdv", "attn_bwd_dq", "attn_bwd_dkdv_keys",
    "attn_fwd_gqa", "attn_bwd_gqa", "attn_bwd_gqa_workspace_size",
    "attn_fwd_sparse", "attn_bwd_sparse", "attn_fwd_sparse_workspace_size", "attn_fwd_fp8",
    "forward_fp8", "attn_quantize_fp8", "attn_quantize_fp8_workspace_size", "quantize_fp8",
    "attn_bwd_sparse_workspace_size",
    "attn_mat_fwd", "attn_mat_bwd", "attn_mat_workspace_size",
    "attn_gemm_bf16", "attn_status", "attn_strerror", "attn_version", "attn_launch_count",
    "attn_selftest_wait_timeout",
    "forward", "backward",
]

ATTN_BF16, ATTN_F32 = 0, 1
(ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_WORKSPACE, ATTN_ERR_CUDA,
 ATTN_ERR_DEVICE_TIMEOUT) = range(6)
ATTN_DQ_AUTO, ATTN_DQ_ATOMIC, ATTN_DQ_PASS, ATTN_DQ_SPILL = 0, 1, 2, 3

_LIB = None
_LOCK = threading.Lock()


def lib_path():
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn.so")


class AttnError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s failed: %s (code %d)" % (where, attn_strerror(code), code))


def lib():
    """Load libattn.so (built in-tree by __graft_entry__.build())."""
    global _LIB
    if _LIB is not None:
        return _LIB
    with _LOCK:
        if _LIB is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    "libattn.so is not built (%s); run __graft_entry__.build()" % path)
            L = ctypes.CDLL(path)
            vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
            L.attn_fwd.restype = i
            L.attn_bwd_workspace_size.argtypes = [i, i, i, i, i, i, i]
            L.attn_bwd_workspace_size.restype = sz
            L.attn_bwd.argtypes = [vp] * 9 + [i, i, i, i, i, f, i, i, vp, sz, vp]
            L.attn_bwd.restype = i
            L.attn_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
            L.attn_fwd_gqa.restype = i
            L.attn_bwd_gqa.argtypes = [vp] * 9 + [i, i, i, i, i, i, f, i, i, vp, sz, vp]
            L.attn_bwd_gqa.restype = i
            L.attn_bwd_gqa_workspace_size.argtypes = [i, i, i, i, i, i, i, i]
            L.attn_bwd_gqa_workspace_size.restype = sz
            L.attn_fwd_fp8.argtypes = [vp] * 5 + [i, i, i, i, f, vp, vp, vp, i, vp]
            L.attn_fwd_fp8.restype = i
            L.attn_quantize_fp8_workspace_size.argtypes = [i, i, i]
            L.attn_quantize_fp8_workspace_size.restype = sz
            L.attn_quantize_fp8.argtypes = [vp, vp, vp, i, i, i, i, vp, vp, sz, vp]
            L.attn_quantize_fp8.restype = i
            L.attn_fwd_sparse_workspace_size.argtypes = [i, i]
            L.attn_fwd_sparse_workspace_size.restype = sz
            L.attn_fwd_sparse.argtypes = [vp] * 5 + [i, i, i, i, i, f, i, vp, vp, sz, vp]
            L.attn_fwd_sparse.restype = i
            L.attn_bwd_sparse_workspace_size.argtypes = [i, i, i, i, i, i, i]
            L.attn_bwd_sparse_workspace_size.restype = sz
            L.attn_bwd_sparse.argtypes = [vp] * 9 + [i, i, i, i, i, f, i, i, vp, vp, sz, vp]
            L.attn_bwd_sparse.restype = i
            L.attn_bwd_preprocess.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, vp, sz, vp]
            L.attn_bwd_preprocess.restype = i
            L.attn_bwd_dkdv.argtypes = [vp] * 6 + [i, i, i, i, i, f, i, i, vp, sz, vp]
            L.attn_bwd_dkdv.restype = i
            L.attn_bwd_dq.argtypes = [vp] * 5 + [i, i, i, i, i, f, i, i, vp, sz, vp]
            L.attn_bwd_dq.restype = i
            L.attn_bwd_dkdv_keys.argtypes = [vp] * 6 + [i, i, i, i, i, f, i, i, i, vp, sz, vp]
            L.attn_bwd_dkdv_keys.restype = i
            L.attn_bwd_noalloc.argtypes = [vp] * 9 + [i, i, i, i, i, f, i, vp]
            L.attn_bwd_noalloc.restype = i
            L.attn_mat_workspace_size.argtypes = [i, i, i, i]
            L.attn_mat_workspace_size.restype = sz
            L.attn_mat_fwd.argtypes = [vp] * 5 + [i, i, i, i, f, i, vp, sz, vp]
            L.attn_mat_fwd.restype = i
            L.attn_mat_bwd.argtypes = [vp] * 9 + [i, i, i, i, f, i, vp, sz, vp]
            L.attn_mat_bwd.restype = i
            L.attn_gemm_bf16.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, f, vp]
            L.attn_gemm_bf16.restype = i
            L.attn_status.argtypes = [vp]
            L.attn_status.restype = i
            L.attn_strerror.argtypes = [i]
            L.attn_strerror.restype = ctypes.c_char_p
            L.attn_version.argtypes = []
            L.attn_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, vp]
            L.attn_selftest_wait_timeout.restype = i
            L.attn_launch_count.argtypes = []
            L.attn_launch_count.restype = ctypes.c_ulonglong
            L.attn_version.restype = ctypes.c_char_p
            _LIB = L
    return _LIB


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float32:
        return ATTN_F32
    raise TypeError("unsupported dtype %s" % t.dtype)


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected [B, H, n, d], got %s" % (tuple(q.shape),))
    return tuple(int(x) for x in q.shape)


def _check(rc, where):
    if rc != 0:
        raise AttnError(rc, where)


def attn_strerror(code):
    return lib().attn_strerror(int(code)).decode()


def attn_version():
    return lib().attn_version().decode()


def attn_status(stream=None):
    """Synchronise the stream; return and clear the first device-side error."""
    return lib().attn_status(_stream(stream))


def attn_selftest_wait_timeout(timeout_ns, stream=None):
    """Launch the bounded-wait self-test: one wait with no arrival runs out
    after timeout_ns, so the next attn_status() returns ATTN_ERR_DEVICE_TIMEOUT."""
    _check(lib().attn_selftest_wait_timeout(int(timeout_ns), _stream(stream)),
           "attn_selftest_wait_timeout")


def attn_launch_count():
    """Kernels the library has enqueued in this process so far."""
    return int(lib().attn_launch_count())


def attn_fwd(Q, K, V, O, LSE, scale, causal, stream=None):
    B, H, n, d = _shape(Q)
    rc = lib().attn_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, n, d,
                        _dtype_code(Q), float(scale), int(bool(causal)), _stream(stream))
    _check(rc, "attn_fwd")


def attn_bwd_workspace_size(B, H, n, d, dtype, causal, mode=ATTN_DQ_AUTO):
    return int(lib().attn_bwd_workspace_size(B, H, n, d, dtype, int(bool(causal)), int(mode)))


def attn_bwd_gqa_workspace_size(B, H, Hkv, n, d, dtype, causal, mode=ATTN_DQ_AUTO):
    return int(lib().attn_bwd_gqa_workspace_size(B, H, Hkv, n, d, dtype, int(bool(causal)),
                                                 int(mode)))


def attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, scale, causal, mode=ATTN_DQ_AUTO,
             workspace=None, stream=None):
    B, H, n, d = _shape(Q)
    dt = _dtype_code(Q)
    need = attn_bwd_workspace_size(B, H, n, d, dt, causal, mode)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=Q.device)
    rc = lib().attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ),
                        _ptr(dK), _ptr(dV), B, H, n, d, dt, float(scale),
                        int(bool(causal)), int(mode), _ptr(workspace),
                        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_bwd")


def attn_bwd_noalloc(Q, K, V, O, dO, LSE, dQ, dK, dV, scale, causal, stream=None):
    """The backward without a workspace: its row statistics live in a fixed
    device array inside the library (dQ by the query-tile pass).  Calls that
    overlap on the GPU share that array, so keep them on one stream."""
    B, H, n, d = _shape(Q)
    rc = lib().attn_bwd_noalloc(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE),
                                _ptr(dQ), _ptr(dK), _ptr(dV), B, H, n, d, _dtype_code(Q),
                                float(scale), int(bool(causal)), _stream(stream))
    _check(rc, "attn_bwd_noalloc")


def _kv_heads(Q, K):
    B, H, n, d = _shape(Q)
    Bk, Hkv, nk, dk = _shape(K)
    if (Bk, nk, dk) != (B, n, d):
        raise ValueError("K shape %s does not match Q shape %s" % (tuple(K.shape), tuple(Q.shape)))
    return Hkv


def attn_fwd_gqa(Q, K, V, O, LSE, scale, causal, stream=None):
    """Grouped-query forward: K, V hold K.shape[1] heads shared by Q's heads."""
    B, H, n, d = _shape(Q)
    Hkv = _kv_heads(Q, K)
    rc = lib().attn_fwd_gqa(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, Hkv, n, d,
                            _dtype_code(Q), float(scale), int(bool(causal)), _stream(stream))
    _check(rc, "attn_fwd_gqa")


def attn_bwd_gqa(Q, K, V, O, dO, LSE, dQ, dK, dV, scale, causal, mode=ATTN_DQ_AUTO,
                 workspace=None, stream=None):
    """Grouped-query backward: dK, dV ([B, H_kv, n, d]) sum over each group."""
    B, H, n, d = _shape(Q)
    Hkv = _kv_heads(Q, K)
    dt = _dtype_code(Q)
    need = attn_bwd_gqa_workspace_size(B, H, Hkv, n, d, dt, causal, mode)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=Q.device)
    rc = lib().attn_bwd_gqa(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ),
                            _ptr(dK), _ptr(dV), B, H, Hkv, n, d, dt, float(scale),
                            int(bool(causal)), int(mode), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_bwd_gqa")


def attn_fwd_fp8(Q8, K8, Vt8, O, LSE, scale, causal, descale_q=None, descale_k=None,
                 descale_v=None, stream=None):
    """FP8 forward: Q8, K8 [B, H, n, 128] and Vt8 [B, H, 128, n] e4m3 tensors,
    per-head fp32 descales [B, H] on the device (None = 1), O bf16, LSE fp32."""
    B, H, n, d = _shape(Q8)
    rc = lib().attn_fwd_fp8(_ptr(Q8), _ptr(K8), _ptr(Vt8), _ptr(O), _ptr(LSE), B, H, n, d,
                            float(scale), _ptr(descale_q), _ptr(descale_k), _ptr(descale_v),
                            int(bool(causal)), _stream(stream))
    _check(rc, "attn_fwd_fp8")


def attn_quantize_fp8_workspace_size(BH, n, d):
    return int(lib().attn_quantize_fp8_workspace_size(int(BH), int(n), int(d)))


def attn_quantize_fp8(X, X8, descale, transpose=False, signs=None, workspace=None, stream=None):
    """Per-head e4m3 encoding of X bf16 [B, H, n, 128] into X8 (same shape, or
    [B, H, 128, n] when transposed) and descale [B, H]; signs (128 floats of
    +-1) selects the Hadamard rotation of incoherent processing."""
    B, H, n, d = _shape(X)
    if workspace is None:
        workspace = torch.empty(max(attn_quantize_fp8_workspace_size(B * H, n, d), 4),
                                dtype=torch.uint8, device=X.device)
    rc = lib().attn_quantize_fp8(_ptr(X), _ptr(X8), _ptr(descale), B * H, n, d,
                                 int(bool(transpose)), _ptr(signs), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_quantize_fp8")


def quantize_fp8(x, transpose=False, signs=None, stream=None):
    """Allocate and run attn_quantize_fp8.  Returns (x8, descale)."""
    B, H, n, d = _shape(x)
    shape = (B, H, d, n) if transpose else (B, H, n, d)
    x8 = torch.empty(shape, dtype=torch.float8_e4m3fn, device=x.device)
    descale = torch.empty((B, H), dtype=torch.float32, device=x.device)
    attn_quantize_fp8(x, x8, descale, transpose, signs, None, stream)
    return x8, descale


def forward_fp8(q8, k8, vt8, descales=(None, None, None), causal=False, scale=None,
                stream=None):
    """Allocate O (bf16) and LSE and run attn_fwd_fp8.  Returns (O, LSE)."""
    B, H, n, d = _shape(q8)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    o = torch.empty((B, H, n, d), dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((B, H, n), dtype=torch.float32, device=q8.device)
    attn_fwd_fp8(q8, k8, vt8, o, lse, scale, causal, *descales, stream=stream)
    return o, lse


def attn_fwd_sparse_workspace_size(n, d):
    return int(lib().attn_fwd_sparse_workspace_size(n, d))


def attn_bwd_sparse_workspace_size(B, H, n, d, dtype, causal, mode=ATTN_DQ_AUTO):
    return int(lib().attn_bwd_sparse_workspace_size(B, H, n, d, dtype, int(bool(causal)),
                                                    int(mode)))


def attn_fwd_sparse(Q, K, V, O, LSE, scale, causal, block_mask, workspace=None, stream=None):
    """Block-sparse forward; block_mask: uint8 device tensor [ceil(n/128)]^2."""
    B, H, n, d = _shape(Q)
    if workspace is None:
        need = attn_fwd_sparse_workspace_size(n, d)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=Q.device)
    rc = lib().attn_fwd_sparse(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, n, d,
                               _dtype_code(Q), float(scale), int(bool(causal)), _ptr(block_mask),
                               _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream))
    _check(rc, "attn_fwd_sparse")


def attn_bwd_sparse(Q, K, V, O, dO, LSE, dQ, dK, dV, scale, causal, block_mask,
                    mode=ATTN_DQ_AUTO, workspace=None, stream=None):
    """Block-sparse backward (same pattern as the forward)."""
    B, H, n, d = _shape(Q)
    dt = _dtype_code(Q)
    if workspace is None:
        need = attn_bwd_sparse_workspace_size(B, H, n, d, dt, causal, mode)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=Q.device)
    rc = lib().attn_bwd_sparse(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE), _ptr(dQ),
                               _ptr(dK), _ptr(dV), B, H, n, d, dt, float(scale),
                               int(bool(causal)), int(mode), _ptr(block_mask), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_bwd_sparse")


def _ws(workspace):
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def attn_bwd_preprocess(O, dO, LSE, causal, mode, workspace, stream=None):
    B, H, n, d = _shape(O)
    wp, wb = _ws(workspace)
    rc = lib().attn_bwd_preprocess(_ptr(O), _ptr(dO), _ptr(LSE), B, H, n, d, _dtype_code(O),
                                   int(bool(causal)), int(mode), wp, wb, _stream(stream))
    _check(rc, "attn_bwd_preprocess")


def attn_bwd_dkdv(Q, K, V, dO, dK, dV, scale, causal, mode, workspace, stream=None):
    B, H, n, d = _shape(Q)
    wp, wb = _ws(workspace)
    rc = lib().attn_bwd_dkdv(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(dK), _ptr(dV), B, H, n, d,
                             _dtype_code(Q), float(scale), int(bool(causal)), int(mode), wp, wb,
                             _stream(stream))
    _check(rc, "attn_bwd_dkdv")


def attn_bwd_dkdv_keys(Q, K, V, dO, dK, dV, scale, causal, mode, key_rows, workspace,
                       stream=None):
    """attn_bwd_dkdv with key tiles of key_rows keys (128, 64, 32): the IO
    study's way of changing the on-chip memory of the key-tile kernel."""
    B, H, n, d = _shape(Q)
    wp, wb = _ws(workspace)
    rc = lib().attn_bwd_dkdv_keys(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(dK), _ptr(dV), B, H,
                                  n, d, _dtype_code(Q), float(scale), int(bool(causal)),
                                  int(mode), int(key_rows), wp, wb, _stream(stream))
    _check(rc, "attn_bwd_dkdv_keys")


def attn_bwd_dq(Q, K, V, dO, dQ, scale, causal, mode, workspace, stream=None):
    B, H, n, d = _shape(dQ)
    wp, wb = _ws(workspace)
    rc = lib().attn_bwd_dq(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(dQ), B, H, n, d,
                           _dtype_code(dQ), float(scale), int(bool(causal)), int(mode), wp, wb,
                           _stream(stream))
    _check(rc, "attn_bwd_dq")


def attn_mat_workspace_size(B, H, n, d):
    return int(lib().attn_mat_workspace_size(B, H, n, d))


def attn_mat_fwd(Q, K, V, O, LSE, scale, causal, workspace, stream=None):
    B, H, n, d = _shape(Q)
    rc = lib().attn_mat_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, n, d,
                            float(scale), int(bool(causal)), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_mat_fwd")


def attn_mat_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, scale, causal, workspace, stream=None):
    B, H, n, d = _shape(Q)
    rc = lib().attn_mat_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE),
                            _ptr(dQ), _ptr(dK), _ptr(dV), B, H, n, d, float(scale),
                            int(bool(causal)), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_mat_bwd")


def attn_gemm_bf16(A, Bm, C, batch, M, N, K, a_kmajor, b_kmajor, alpha=1.0, stream=None):
    c_f32 = C.dtype == torch.float32
    rc = lib().attn_gemm_bf16(_ptr(A), _ptr(Bm), _ptr(C), batch, M, N, K, int(bool(a_kmajor)),
                              int(bool(b_kmajor)), int(c_f32), float(alpha), _stream(stream))
    _check(rc, "attn_gemm_bf16")


# ---------------------------------------------------------------- conveniences

def forward(q, k, v, causal=False, scale=None, stream=None, block_mask=None):
    """Allocate O and LSE with torch and run attn_fwd (attn_fwd_gqa when K
    has fewer heads, attn_fwd_sparse with a block mask).  Returns (O, LSE)."""
    B, H, n, d = _shape(q)
    scale = (1.0 / d ** 0.5) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, n), dtype=torch.float32, device=q.device)
    if block_mask is not None:
        attn_fwd_sparse(q, k, v, o, lse, scale, causal, block_mask, None, stream)
    elif k.shape[1] != H:   # grouped-query: fewer key/value heads than query heads
        attn_fwd_gqa(q, k, v, o, lse, scale, causal, stream)
    else:
        attn_fwd(q, k, v, o, lse, scale, causal, stream)
    return o, lse


def backward(q, k, v, o, do, lse, causal=False, scale=None, mode=ATTN_DQ_AUTO,
             workspace=None, stream=None, block_mask=None):
    """Allocate dQ, dK, dV with torch and run attn_bwd.  Returns (dQ, dK, dV)."""
    d = q.shape[-1]
    scale = (1.0 / d ** 0.5) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if block_mask is not None:
        attn_bwd_sparse(q, k, v, o, do, lse, dq, dk, dv, scale, causal, block_mask, mode,
                        workspace, stream)
    elif k.shape[1] != q.shape[1]:
        attn_bwd_gqa(q, k, v, o, do, lse, dq, dk, dv, scale, causal, mode, workspace, stream)
    else:
        attn_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, causal, mode, workspace, stream)
    return dq, dk, dv
