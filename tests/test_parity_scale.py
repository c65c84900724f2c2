"""Parity with a score scale other than 1/sqrt(d).

`scale` is an argument of every entry point ("Chapter 3.1 -- The cost of
attention", section 2, and "Flash Attention: Revolutionizing Transformer
Efficiency", "Standard attention": the scores are the dot products times a
factor, 1/sqrt(d) in the pages' formula).  Every other parity test passes
1/sqrt(d), so a kernel that ignored the argument, or derived it from d,
would pass them; these cases pass 0.05 (flatter than 1/sqrt(d) for every d
here) and 0.2 (sharper) through the C ABI and compare every element of O,
LSE, dQ, dK and dV with the float64 oracle given the same scale, for the
bf16 kernels at each head dim, both masks and both dQ modes, the fp32
kernels, grouped-query and block-sparse attention, the materialise-P path
and the FP8 forward.
"""

import pytest
import torch

import oracle
from io_aware_exact_05_gb300.inputs import Workload, make_block_mask, make_inputs
from parity_util import TOL, relerr

pytestmark = pytest.mark.gpu

SCALES = [0.05, 0.2]


def _run(w, scale, dev, mode=0, block_mask=None):
    from io_aware_exact_05_gb300 import attn

    x = make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    bm = None if block_mask is None else block_mask.to(dev)
    o, lse = attn.forward(q, k, v, causal=w.causal, scale=scale, block_mask=bm)
    dq, dk, dv = attn.backward(q, k, v, o, do, lse, causal=w.causal, scale=scale, mode=mode,
                               block_mask=bm)
    assert attn.attn_status() == 0
    return x, (o, lse, dq, dk, dv)


def _check(w, scale, x, outs, tol, block_mask=None):
    bm = None if block_mask is None else block_mask.numpy().astype(bool)
    ro, rl = oracle.attention_forward(x["q"], x["k"], x["v"], scale, w.causal, bm)
    rdq, rdk, rdv, _ = oracle.attention_backward(x["q"], x["k"], x["v"], x["do"], scale,
                                                 w.causal, bm)
    o, lse, dq, dk, dv = outs
    errs = {"O": relerr(o, ro), "LSE": relerr(lse, rl), "dQ": relerr(dq, rdq),
            "dK": relerr(dk, rdk), "dV": relerr(dv, rdv)}
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, (scale, errs)


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("mode", [1, 2], ids=["atomic", "pass"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_bf16(cuda_dev, d, causal, mode, scale):
    if d == 256 and mode == 1:
        pytest.skip("d = 256 computes dQ by the query-tile pass only")
    w = Workload("scale", 1, 2, 300, d, "bf16", causal, 1.0, 2100 + d + int(causal))
    x, outs = _run(w, scale, cuda_dev, mode)
    _check(w, scale, x, outs, TOL["bf16"])


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [32, 100])
def test_f32(cuda_dev, d, causal, scale):
    w = Workload("scale_f32", 2, 1, 150, d, "f32", causal, 1.0, 2200 + d)
    x, outs = _run(w, scale, cuda_dev)
    _check(w, scale, x, outs, TOL["f32"])


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("d,H,Hkv", [(64, 4, 1), (128, 4, 2)])
def test_grouped(cuda_dev, d, H, Hkv, scale):
    w = Workload("scale_gqa", 1, H, 260, d, "bf16", True, 1.0, 2300 + d + H, H_kv=Hkv)
    x, outs = _run(w, scale, cuda_dev)
    _check(w, scale, x, outs, TOL["bf16"])


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("d", [128, 256])
def test_block_sparse(cuda_dev, d, scale):
    w = Workload("scale_sparse", 1, 2, 520, d, "bf16", False, 1.0, 2400 + d)
    mask = make_block_mask(520, 1, 1, 1, 2400 + d)
    x, outs = _run(w, scale, cuda_dev, block_mask=mask)
    _check(w, scale, x, outs, TOL["bf16"], mask)


@pytest.mark.parametrize("scale", SCALES)
def test_materialise_path(cuda_dev, scale):
    from io_aware_exact_05_gb300 import attn

    w = Workload("scale_mat", 1, 2, 264, 128, "bf16", True, 1.0, 2500)
    x = make_inputs(w)
    q, k, v, do = (x[n].to(cuda_dev) for n in ("q", "k", "v", "do"))
    ws = torch.empty(attn.attn_mat_workspace_size(1, 2, w.n, w.d), dtype=torch.uint8,
                     device=cuda_dev)
    o, lse = torch.empty_like(q), torch.empty(1, 2, w.n, device=cuda_dev)
    attn.attn_mat_fwd(q, k, v, o, lse, scale, w.causal, ws)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    attn.attn_mat_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, w.causal, ws)
    assert attn.attn_status() == 0
    _check(w, scale, x, (o, lse, dq, dk, dv), TOL["bf16"])


@pytest.mark.parametrize("scale", SCALES)
def test_fp8_forward(cuda_dev, scale):
    from io_aware_exact_05_gb300 import attn
    from test_parity_fp8 import _check_forward, _oracle_operands

    w = Workload("scale_fp8", 1, 2, 400, 128, "bf16", True, 1.0, 2600)
    ops = _oracle_operands(make_inputs(w))
    o, lse = attn.forward_fp8(ops["q8"].to(cuda_dev), ops["k8"].to(cuda_dev),
                              ops["v8"].to(cuda_dev),
                              (ops["ds_q"].to(cuda_dev), ops["ds_k"].to(cuda_dev),
                               ops["ds_v"].to(cuda_dev)), causal=True, scale=scale)
    assert attn.attn_status() == 0
    ro, rl = oracle.attention_forward(ops["q"], ops["k"], ops["v"], scale, True)
    _check_forward(o, lse, ro, rl)
