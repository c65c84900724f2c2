"""The dQ mode "spill" (d = 256): the key-tile kernel also writes dS^T to the
workspace and dQ = scale dS K is one tensor-core GEMM.  Every element of dQ,
dK and dV against the float64 oracle on ragged shapes and scales, through
attn_bwd and through the three stages; and, since the automatic mode now
spills on the full d = 256 workload, the query-tile pass on every head of it."""

import pytest
import torch

import oracle
from io_aware_exact_05_gb300.inputs import Workload, make_inputs, workload
from parity_util import TOL, relerr

pytestmark = pytest.mark.gpu


def _check(w, x, outs, scale, heads=None):
    q, k, v, do = (x[n] for n in ("q", "k", "v", "do"))
    if heads is None:
        rdq, rdk, rdv, _ = oracle.attention_backward(q, k, v, do, scale, w.causal)
        got = outs
    else:
        BH = w.B * w.H
        flat = [t.reshape(BH, w.n, w.d) for t in (q, k, v, do)]
        got = [t.float().cpu().reshape(BH, w.n, w.d) for t in outs]
        errs = {}
        for hh in heads:
            r = oracle.attention_backward_head(*(t[hh] for t in flat), scale, w.causal)[:3]
            for name, g, rr in zip(("dQ", "dK", "dV"), got, r):
                errs["%s[h%d]" % (name, hh)] = relerr(g[hh], rr)
        assert all(e <= TOL["bf16"] for e in errs.values()), errs
        return
    floor = 1.0 if w.n == 1 else 0.0     # n = 1: dQ = dK = 0 exactly
    errs = {"dQ": relerr(got[0], rdq, floor), "dK": relerr(got[1], rdk, floor),
            "dV": relerr(got[2], rdv)}
    assert all(e <= TOL["bf16"] for e in errs.values()), errs


@pytest.mark.parametrize("n", [1, 7, 129, 300, 520])
def test_spill_small(cuda_dev, n):
    from io_aware_exact_05_gb300 import attn

    w = Workload("spill", 1, 2, n, 256, "bf16", False, 1.0, 2800 + n)
    x = make_inputs(w)
    q, k, v, do = (x[t].to(cuda_dev) for t in ("q", "k", "v", "do"))
    o, lse = attn.forward(q, k, v)
    outs = attn.backward(q, k, v, o, do, lse, mode=attn.ATTN_DQ_SPILL)
    assert attn.attn_status() == 0
    _check(w, x, outs, w.scale)


@pytest.mark.parametrize("scale", [0.05, 0.2])
def test_spill_stages_and_scale(cuda_dev, scale):
    # the three exported stages in spill mode, with a scale other than 1/sqrt(d)
    from io_aware_exact_05_gb300 import attn

    w = Workload("spill_st", 2, 1, 260, 256, "bf16", False, 1.0, 2900)
    x = make_inputs(w)
    q, k, v, do = (x[t].to(cuda_dev) for t in ("q", "k", "v", "do"))
    o, lse = attn.forward(q, k, v, scale=scale)
    mode = attn.ATTN_DQ_SPILL
    ws = torch.empty(attn.attn_bwd_workspace_size(2, 1, w.n, 256, attn.ATTN_BF16, False, mode),
                     dtype=torch.uint8, device=cuda_dev)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    attn.attn_bwd_preprocess(o, do, lse, False, mode, ws)
    attn.attn_bwd_dkdv(q, k, v, do, dk, dv, scale, False, mode, ws)
    attn.attn_bwd_dq(q, k, v, do, dq, scale, False, mode, ws)
    assert attn.attn_status() == 0
    _check(w, x, (dq, dk, dv), scale)


def test_pass_full_workload_every_head(cuda_dev):
    # the automatic mode spills on this workload (test_parity_configs checks
    # it on every head); the query-tile pass, every head, at full size
    from io_aware_exact_05_gb300 import attn

    w = workload("b2h8_n4k_d256")
    x = make_inputs(w)
    q, k, v, do = (x[t].to(cuda_dev) for t in ("q", "k", "v", "do"))
    o, lse = attn.forward(q, k, v)
    outs = attn.backward(q, k, v, o, do, lse, mode=attn.ATTN_DQ_PASS)
    assert attn.attn_status() == 0
    _check(w, x, outs, w.scale, heads=range(w.B * w.H))
