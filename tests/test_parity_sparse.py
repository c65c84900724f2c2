"""Block-sparse exact attention through the C ABI against the float64 oracle:
a 128 x 128-block pattern (local window, global blocks, random blocks, and
block rows / columns that keep nothing) on small and ragged shapes for every
dtype, head dim and dQ mode, the all-kept pattern against the dense path, and
one full head of a 16k-token sparse workload."""

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_05_gb300.inputs import Workload, make_block_mask, make_inputs, workload
from parity_util import TOL, relerr, to64

pytestmark = pytest.mark.gpu


def _pattern(n, seed, empty_row=None, empty_col=None):
    m = make_block_mask(n, 1, 1, 1, seed).clone()
    nb = m.shape[0]
    if empty_row is not None and empty_row < nb:
        m[empty_row] = 0
    if empty_col is not None and empty_col < nb:
        m[:, empty_col] = 0
    return m


def _lse_err(got, ref):
    # rows that keep nothing: -inf on both sides; elsewhere max|err| / max|ref|
    g, r = to64(got), to64(ref)
    gi, ri = np.isneginf(g), np.isneginf(r)
    if not np.array_equal(gi, ri) or not np.isfinite(g[~gi]).all():
        return float("inf")
    return relerr(g[~gi], r[~ri]) if (~gi).any() else 0.0


def _run(w, mask, dev, mode=0):
    from io_aware_exact_05_gb300 import attn

    x = make_inputs(w)
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    bm = mask.to(dev)
    o, lse = attn.forward(q, k, v, causal=w.causal, block_mask=bm)
    dq, dk, dv = attn.backward(q, k, v, o, do, lse, causal=w.causal, mode=mode, block_mask=bm)
    assert attn.attn_status() == 0
    return x, (o, lse, dq, dk, dv)


def _check(w, x, mask, outs, tol):
    bm = mask.numpy().astype(bool)
    ro, rl = oracle.attention_forward(x["q"], x["k"], x["v"], w.scale, w.causal, bm)
    rdq, rdk, rdv, _ = oracle.attention_backward(x["q"], x["k"], x["v"], x["do"], w.scale,
                                                 w.causal, bm)
    o, lse, dq, dk, dv = outs
    errs = {"O": relerr(o, ro), "LSE": _lse_err(lse, rl), "dQ": relerr(dq, rdq, 1e-30),
            "dK": relerr(dk, rdk, 1e-30), "dV": relerr(dv, rdv, 1e-30)}
    bad = {k: e for k, e in errs.items() if not e <= tol}
    assert not bad, errs


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [384, 600])
def test_bf16(cuda_dev, d, causal, n):
    w = Workload("sparse", 1, 2, n, d, "bf16", causal, 1.0, 1100 + n + d)
    mask = _pattern(n, 7 + n + d, empty_row=2, empty_col=3)
    x, outs = _run(w, mask, cuda_dev)
    _check(w, x, mask, outs, TOL["bf16"])
    o, lse = outs[0].float().cpu(), outs[1].cpu()
    rows = slice(256, min(n, 384))            # block row 2 keeps nothing
    assert torch.all(o[:, :, rows] == 0) and torch.all(torch.isneginf(lse[:, :, rows]))
    assert torch.all(outs[2][:, :, rows].float().cpu() == 0)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_dq_pass_mode(cuda_dev, d, causal):
    from io_aware_exact_05_gb300 import attn

    w = Workload("sparse_pass", 2, 1, 520, d, "bf16", causal, 1.0, 1200 + d)
    mask = _pattern(520, 11 + d, empty_row=1)
    x, outs = _run(w, mask, cuda_dev, attn.ATTN_DQ_PASS)
    _check(w, x, mask, outs, TOL["bf16"])


@pytest.mark.parametrize("d,n,causal", [(32, 300, True), (100, 260, False)])
def test_f32(cuda_dev, d, n, causal):
    w = Workload("sparse_f32", 1, 2, n, d, "f32", causal, 1.0, 1300 + n + d)
    mask = _pattern(n, 13, empty_row=1, empty_col=0)
    x, outs = _run(w, mask, cuda_dev)
    _check(w, x, mask, outs, TOL["f32"])


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_all_kept_equals_dense(cuda_dev, d, causal):
    # every block kept: the same tiles in the same order as the dense kernels
    from io_aware_exact_05_gb300 import attn

    w = Workload("allkept", 1, 2, 520, d, "bf16", causal, 1.0, 1400 + d)
    x = make_inputs(w)
    q, k, v, do = (x[n].to(cuda_dev) for n in ("q", "k", "v", "do"))
    ones = torch.ones(5, 5, dtype=torch.uint8, device=cuda_dev)
    o1, l1 = attn.forward(q, k, v, causal=causal)
    o2, l2 = attn.forward(q, k, v, causal=causal, block_mask=ones)
    g1 = attn.backward(q, k, v, o1, do, l1, causal=causal)
    g2 = attn.backward(q, k, v, o2, do, l2, causal=causal, block_mask=ones)
    assert attn.attn_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])   # dK, dV: same arithmetic
    # dQ adds its per-key-tile shares with atomics, in an order that varies
    # from run to run: the bf16 rounding of a few elements can differ
    assert relerr(g1[0], g2[0]) <= 1e-2


def test_nothing_kept(cuda_dev):
    from io_aware_exact_05_gb300 import attn

    w = Workload("nothing", 1, 2, 300, 128, "bf16", False, 1.0, 1500)
    zeros = torch.zeros(3, 3, dtype=torch.uint8)
    x, outs = _run(w, zeros, cuda_dev)
    o, lse, dq, dk, dv = (t.float().cpu() for t in outs)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    assert torch.all(dq == 0) and torch.all(dk == 0) and torch.all(dv == 0)


def test_full_head_16k_pattern(cuda_dev):
    # b2h16_n16k_d128_sparse: every element of head 0 against the oracle
    from io_aware_exact_05_gb300 import attn

    w = workload("b2h16_n16k_d128_sparse")
    mask = make_block_mask(w.n, *w.sparse, w.seed)
    x = make_inputs(w)
    q, k, v, do = (x[n].to(cuda_dev) for n in ("q", "k", "v", "do"))
    bm = mask.to(cuda_dev)
    o, lse = attn.forward(q, k, v, causal=w.causal, block_mask=bm)
    dq, dk, dv = attn.backward(q, k, v, o, do, lse, causal=w.causal, block_mask=bm)
    assert attn.attn_status() == 0
    b = mask.numpy().astype(bool)
    ro, rl = oracle.attention_forward_head(x["q"][0, 0], x["k"][0, 0], x["v"][0, 0], w.scale,
                                           w.causal, None, b)
    rdq, rdk, rdv, _ = oracle.attention_backward_head(x["q"][0, 0], x["k"][0, 0], x["v"][0, 0],
                                                      x["do"][0, 0], w.scale, w.causal, b)
    errs = {"O": relerr(o[0, 0].cpu(), ro), "LSE": _lse_err(lse[0, 0].cpu(), rl),
            "dQ": relerr(dq[0, 0].cpu(), rdq), "dK": relerr(dk[0, 0].cpu(), rdk),
            "dV": relerr(dv[0, 0].cpu(), rdv)}
    assert all(e <= TOL["bf16"] for e in errs.values()), errs
