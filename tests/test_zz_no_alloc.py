"""attn_bwd_noalloc: the backward pass for callers that cannot allocate.

Some callers cannot give the library a workspace (no device allocator of
their own, a memory budget fixed at start-up, or no cudaMalloc allowed where
they run the backward).  attn_bwd_noalloc keeps its scratch in a fixed device
array inside the library instead.  These tests call it through the C ABI and
compare it with attn_bwd, the workspace entry point, and with the float64
oracle, on consecutive calls that reuse the same array (one call's leftovers
must not leak into the next).  This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

import oracle
from io_aware_exact_05_gb300.inputs import Workload, make_inputs
from parity_util import TOL, relerr

FAKE = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced


def _noalloc():
    from io_aware_exact_05_gb300 import attn
    from io_aware_exact_05_gb300.build import build
    import os

    if not os.path.exists(attn.lib_path()):
        build()
    return attn.lib().attn_bwd_noalloc   # argument types set by the binding


def test_noalloc_rejects_problems_beyond_its_scratch():
    f = _noalloc()
    args = [FAKE] * 9
    # bf16: B*H*n_pad = 64 * 32768 fills the 16 MiB array exactly; one more head does not fit
    assert f(*args, 1, 65, 32768, 128, 0, 0.1, 1, None) == 3          # ATTN_ERR_WORKSPACE
    assert f(*args, 1, 1, 4194304 + 128, 64, 1, 0.1, 0, None) == 3    # fp32 limit
    assert f(*args, 1, 1, 128, 96, 0, 0.1, 0, None) == 2              # unsupported head dim
    assert f(ctypes.c_void_p(0), *args[1:], 1, 1, 128, 64, 0, 0.1, 0, None) == 1


def _check_oracle(w, x, got, scale):
    """dQ, dK, dV of attn_bwd_noalloc against the float64 oracle, every head."""
    rdq, rdk, rdv, _ = oracle.attention_backward(x["q"], x["k"], x["v"], x["do"], scale,
                                                 w.causal)
    for g, r, name in zip(got, (rdq, rdk, rdv), ("dQ", "dK", "dV")):
        e = relerr(g, r)
        assert e <= TOL[w.dtype], (w.name, name, "vs oracle", e)


def _run_pair(f, w, dev, scale=None):
    """attn_bwd_noalloc and attn_bwd on the same inputs; returns their outputs
    after checking the noalloc outputs against the oracle."""
    from io_aware_exact_05_gb300 import attn

    scale = w.scale if scale is None else scale
    x = make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = attn.forward(q, k, v, causal=w.causal, scale=scale)
    ref = attn.backward(q, k, v, o, do, lse, causal=w.causal, scale=scale)
    got = [torch.full_like(q, float("nan")) for _ in range(3)]
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())   # noqa: E731
    rc = f(ptr(q), ptr(k), ptr(v), ptr(o), ptr(do), ptr(lse), ptr(got[0]), ptr(got[1]),
           ptr(got[2]), w.B, w.H, w.n, w.d, 0 if w.dtype == "bf16" else 1, scale,
           int(w.causal), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    assert attn.attn_status() == 0
    _check_oracle(w, x, got, scale)
    return got, ref


@pytest.mark.gpu
def test_noalloc_matches_attn_bwd_on_two_calls_in_a_row(cuda_dev):
    f = _noalloc()
    # the second call reuses the array the first one left behind, with a
    # different shape, head dim and mask
    for w in (Workload("na1", 1, 3, 1000, 128, "bf16", True, 1.0, 901),
              Workload("na2", 2, 2, 517, 64, "bf16", False, 1.0, 902)):
        got, ref = _run_pair(f, w, cuda_dev)
        for g, r, name in zip(got, ref, ("dQ", "dK", "dV")):
            e = relerr(g, r)
            assert e <= TOL["bf16"], (w.name, name, e)


@pytest.mark.gpu
def test_noalloc_fp32_and_d256(cuda_dev):
    f = _noalloc()
    for w in (Workload("na3", 1, 2, 300, 256, "bf16", True, 1.0, 903),
              Workload("na4", 1, 2, 130, 100, "f32", True, 1.0, 904)):
        got, ref = _run_pair(f, w, cuda_dev)
        for g, r, name in zip(got, ref, ("dQ", "dK", "dV")):
            e = relerr(g, r)
            assert e <= TOL[w.dtype], (w.name, name, e)


@pytest.mark.gpu
def test_noalloc_scale_argument(cuda_dev):
    # a score scale other than 1/sqrt(d) reaches the kernels
    f = _noalloc()
    for w, scale in ((Workload("na5", 1, 2, 260, 128, "bf16", True, 1.0, 905), 0.2),
                     (Workload("na6", 1, 2, 140, 64, "f32", False, 1.0, 906), 0.05)):
        got, ref = _run_pair(f, w, cuda_dev, scale)
        for g, r, name in zip(got, ref, ("dQ", "dK", "dV")):
            e = relerr(g, r)
            assert e <= TOL[w.dtype], (w.name, name, e)
