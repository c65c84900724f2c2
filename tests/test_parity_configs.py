"""Parity at the five workloads' full sizes, in the launch configuration the
benchmark times: the CUDA path runs every head; the float64 oracle checks
every element of O, LSE, dQ, dK and dV (max|err| / max|ref| per output tensor
of a head) of every head of the fp32, d = 64 and d = 256 workloads, and of the
first, the last and seeded middle heads of the two long causal workloads
(their heads cost the oracle 1.5 s and 24 s each).  Causal grids put heads in
the fastest grid dimension, so middle heads check that mapping too."""

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_05_gb300.inputs import WORKLOADS, make_inputs
from parity_util import TOL, relerr

pytestmark = pytest.mark.gpu

# seeded middle heads checked besides the first and the last
MIDDLE_HEADS = {"b2h16_n8k_d128": 4, "b1h8_n32k_d128": 1}


def _heads(w):
    BH = w.B * w.H
    if w.name not in MIDDLE_HEADS:
        return list(range(BH))
    rng = np.random.default_rng(w.seed)
    mid = rng.choice(np.arange(1, BH - 1), size=MIDDLE_HEADS[w.name], replace=False)
    return sorted({0, BH - 1, *(int(h) for h in mid)})


def _check_heads(w, x, outs, tol):
    o, lse, dq, dk, dv = (t.float().cpu() for t in outs)
    q, k, v, do = (x[n].reshape(w.B * w.H, w.n, w.d) for n in ("q", "k", "v", "do"))
    o, dq, dk, dv = (t.reshape(w.B * w.H, w.n, w.d) for t in (o, dq, dk, dv))
    lse = lse.reshape(w.B * w.H, w.n)
    errs = {}
    for hh in _heads(w):
        ro, rl = oracle.attention_forward_head(q[hh], k[hh], v[hh], w.scale, w.causal)
        rdq, rdk, rdv, _ = oracle.attention_backward_head(q[hh], k[hh], v[hh], do[hh], w.scale,
                                                          w.causal)
        for name, got, ref in (("O", o[hh], ro), ("LSE", lse[hh], rl), ("dQ", dq[hh], rdq),
                               ("dK", dk[hh], rdk), ("dV", dv[hh], rdv)):
            errs["%s[h%d]" % (name, hh)] = relerr(got, ref)
    bad = {k_: e for k_, e in errs.items() if not e <= tol}
    assert not bad, errs
    return errs


@pytest.mark.parametrize("w", WORKLOADS, ids=[w.name for w in WORKLOADS])
def test_workload_fused(cuda_dev, w):
    from io_aware_exact_05_gb300 import attn

    x = make_inputs(w)
    q, k, v, do = (x[n].to(cuda_dev) for n in ("q", "k", "v", "do"))
    o, lse = attn.forward(q, k, v, causal=w.causal)
    dq, dk, dv = attn.backward(q, k, v, o, do, lse, causal=w.causal)
    assert attn.attn_status() == 0
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t).all()
    _check_heads(w, x, (o, lse, dq, dk, dv), TOL[w.dtype])


@pytest.mark.parametrize("name", ["b4h16_n2k_d64", "b2h16_n8k_d128"])
def test_workload_dq_pass(cuda_dev, name):
    from io_aware_exact_05_gb300 import attn
    from io_aware_exact_05_gb300.inputs import workload

    w = workload(name)
    x = make_inputs(w)
    q, k, v, do = (x[n].to(cuda_dev) for n in ("q", "k", "v", "do"))
    o, lse = attn.forward(q, k, v, causal=w.causal)
    dq, dk, dv = attn.backward(q, k, v, o, do, lse, causal=w.causal, mode=attn.ATTN_DQ_PASS)
    assert attn.attn_status() == 0
    _check_heads(w, x, (o, lse, dq, dk, dv), TOL[w.dtype])


@pytest.mark.parametrize("name", ["b2h8_n4k_d256", "b4h16_n2k_d64"])
def test_workload_materialise(cuda_dev, name):
    from io_aware_exact_05_gb300 import attn
    from io_aware_exact_05_gb300.inputs import workload

    w = workload(name)
    x = make_inputs(w)
    q, k, v, do = (x[n].to(cuda_dev) for n in ("q", "k", "v", "do"))
    ws = torch.empty(attn.attn_mat_workspace_size(w.B, w.H, w.n, w.d), dtype=torch.uint8,
                     device=cuda_dev)
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.n, device=cuda_dev)
    attn.attn_mat_fwd(q, k, v, o, lse, w.scale, w.causal, ws)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    attn.attn_mat_bwd(q, k, v, o, do, lse, dq, dk, dv, w.scale, w.causal, ws)
    assert attn.attn_status() == 0
    del ws
    _check_heads(w, x, (o, lse, dq, dk, dv), TOL[w.dtype])


def test_sum_invariants_full_size(cuda_dev):
    # properties that hold at any size, on every head of the headline workload:
    # sum_j dV_j = sum_i dO_i (rows of P sum to 1) and sum_j dK_j = 0 (rowsum dS = 0)
    from io_aware_exact_05_gb300 import attn
    from io_aware_exact_05_gb300.inputs import workload

    w = workload("b2h16_n8k_d128")
    x = make_inputs(w)
    q, k, v, do = (x[n].to(cuda_dev) for n in ("q", "k", "v", "do"))
    o, lse = attn.forward(q, k, v, causal=True)
    dq, dk, dv = attn.backward(q, k, v, o, do, lse, causal=True)
    sv = dv.double().sum(2)
    sd = do.double().sum(2)
    assert float((sv - sd).abs().max() / sd.abs().max()) <= 1e-2
    sk = dk.double().sum(2).abs().max()
    assert float(sk / dk.double().abs().sum(2).max()) <= 1e-2
