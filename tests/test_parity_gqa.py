"""Grouped-query and multi-query attention (H query heads sharing H_kv
key/value heads) through the C ABI against the float64 oracle: every element
of O, LSE, dQ and of the group-summed dK, dV, on small and ragged shapes for
every dtype / head dim / dQ mode, and at full size on a grouped workload."""

import pytest
import torch

import oracle
from io_aware_exact_05_gb300.inputs import Workload, make_inputs, workload
from parity_util import TOL, relerr

pytestmark = pytest.mark.gpu


def _run(w, dev, mode=0):
    from io_aware_exact_05_gb300 import attn

    x = make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = attn.forward(q, k, v, causal=w.causal)
    dq, dk, dv = attn.backward(q, k, v, o, do, lse, causal=w.causal, mode=mode)
    assert attn.attn_status() == 0
    assert dk.shape == k.shape and dv.shape == v.shape
    return x, (o, lse, dq, dk, dv)


def _check(w, x, outs, tol):
    ro, rl = oracle.attention_forward(x["q"], x["k"], x["v"], w.scale, w.causal)
    rdq, rdk, rdv, _ = oracle.attention_backward(x["q"], x["k"], x["v"], x["do"], w.scale,
                                                 w.causal)
    o, lse, dq, dk, dv = outs
    floor = 1.0 if w.n == 1 else 0.0     # n = 1: dQ = dK = 0 exactly
    errs = {"O": relerr(o, ro), "LSE": relerr(lse, rl), "dQ": relerr(dq, rdq, floor),
            "dK": relerr(dk, rdk, floor), "dV": relerr(dv, rdv)}
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, errs


HEADS = [(4, 2), (4, 1), (6, 3)]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [129, 520])
@pytest.mark.parametrize("H,Hkv", HEADS)
def test_bf16(cuda_dev, d, causal, n, H, Hkv):
    w = Workload("gqa", 1, H, n, d, "bf16", causal, 1.0, 700 + n + d + H + Hkv, H_kv=Hkv)
    x, outs = _run(w, cuda_dev)
    _check(w, x, outs, TOL["bf16"])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (3, 1)])
def test_bf16_dq_pass_mode(cuda_dev, d, H, Hkv):
    from io_aware_exact_05_gb300 import attn

    w = Workload("gqa_pass", 2, H, 300, d, "bf16", True, 1.0, 800 + d + H, H_kv=Hkv)
    x, outs = _run(w, cuda_dev, attn.ATTN_DQ_PASS)
    _check(w, x, outs, TOL["bf16"])


@pytest.mark.parametrize("d,n,causal", [(32, 77, True), (100, 130, False), (64, 1, True)])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (3, 1)])
def test_f32(cuda_dev, d, n, causal, H, Hkv):
    w = Workload("gqa_f32", 2, H, n, d, "f32", causal, 1.0, 900 + n + d + H, H_kv=Hkv)
    x, outs = _run(w, cuda_dev)
    _check(w, x, outs, TOL["f32"])


def test_full_size_grouped_workload(cuda_dev):
    # b2h16kv4_n8k_d128: every element of the first key/value head's dK, dV
    # (the sum over its four query heads) and of those query heads' O, LSE, dQ
    from io_aware_exact_05_gb300 import attn

    w = workload("b2h16kv4_n8k_d128")
    x = make_inputs(w)
    q, k, v, do = (x[n].to(cuda_dev) for n in ("q", "k", "v", "do"))
    o, lse = attn.forward(q, k, v, causal=True)
    dq, dk, dv = attn.backward(q, k, v, o, do, lse, causal=True)
    assert attn.attn_status() == 0
    g = w.H // w.kv_heads
    sub = {n: x[n][:1, :g] for n in ("q", "do")}
    ro, rl = oracle.attention_forward(sub["q"], x["k"][:1, :1], x["v"][:1, :1], w.scale, True)
    rdq, rdk, rdv, _ = oracle.attention_backward(sub["q"], x["k"][:1, :1], x["v"][:1, :1],
                                                 sub["do"], w.scale, True)
    errs = {"O": relerr(o[:1, :g].cpu(), ro), "LSE": relerr(lse[:1, :g].cpu(), rl),
            "dQ": relerr(dq[:1, :g].cpu(), rdq), "dK": relerr(dk[:1, :1].cpu(), rdk),
            "dV": relerr(dv[:1, :1].cpu(), rdv)}
    assert all(e <= TOL["bf16"] for e in errs.values()), errs


def test_bad_group_is_rejected(cuda_dev):
    from io_aware_exact_05_gb300 import attn

    q = torch.zeros(1, 4, 64, 128, dtype=torch.bfloat16, device=cuda_dev)
    k = torch.zeros(1, 3, 64, 128, dtype=torch.bfloat16, device=cuda_dev)
    with pytest.raises(attn.AttnError) as e:
        attn.forward(q, k, k.clone())
    assert e.value.code == 1    # ATTN_ERR_INVALID_ARG: H_kv does not divide H
