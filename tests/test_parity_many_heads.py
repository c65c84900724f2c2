"""Parity at the largest head counts the boundary accepts (B * H <= 65535):
every grid that maps heads to a grid dimension runs at or near its limit.
d = 64 and 128 at 65535 heads; d = 256 at 40000 heads, where the backward's
two CTAs per key tile would exceed the grid's y limit if both were mapped
to heads (they share a grid.x entry's neighbourhood instead), in the
automatic dQ mode (spill) and the pass.

The inputs repeat seven seeded heads along H (the large tensors are built on
the device from them), so the float64 oracle runs seven heads; sampled heads
(the first, the last, the middle and seeded others, at different residues
modulo 7) are compared element by element with the oracle's head h mod 7."""

import numpy as np
import pytest
import torch

import oracle
from io_aware_exact_05_gb300.inputs import Workload, make_inputs
from parity_util import TOL, relerr

pytestmark = pytest.mark.gpu

NBASE = 7
CASES = [  # (heads, n, d, causal, dQ mode name or None for the default)
    (65535, 128, 64, False, None),
    (65535, 128, 128, True, None),
    (40000, 128, 256, False, None),
    (40000, 128, 256, False, "ATTN_DQ_PASS"),
]


def _sample_heads(H, seed):
    rng = np.random.default_rng(seed)
    return sorted({0, 1, NBASE, H // 2, H - 2, H - 1, *(int(h) for h in rng.choice(H, 6, replace=False))})


@pytest.mark.parametrize("H,n,d,causal,mode", CASES,
                         ids=["h%d_n%d_d%d_%s%s" % (H, n, d, "causal" if c else "full",
                                                    "_pass" if m else "") for H, n, d, c, m in CASES])
def test_many_heads(cuda_dev, H, n, d, causal, mode):
    from io_aware_exact_05_gb300 import attn

    base = Workload("many_heads_base", 1, NBASE, n, d, "bf16", causal, 1.0, 3100 + d)
    x = make_inputs(base)
    reps = (H + NBASE - 1) // NBASE
    q, k, v, do = (x[nm].to(cuda_dev).repeat(1, reps, 1, 1)[:, :H].contiguous()
                   for nm in ("q", "k", "v", "do"))
    o, lse = attn.forward(q, k, v, causal=causal)
    kw = {} if mode is None else {"mode": getattr(attn, mode)}
    dq, dk, dv = attn.backward(q, k, v, o, do, lse, causal=causal, **kw)
    assert attn.attn_status() == 0
    heads = _sample_heads(H, base.seed)
    got = {nm: t[0, heads].float().cpu().numpy() for nm, t in
           (("O", o), ("dQ", dq), ("dK", dk), ("dV", dv))}
    got["LSE"] = lse[0, heads].float().cpu().numpy()
    ref = {}
    for b in range(NBASE):
        qb, kb, vb, db = (x[nm][0, b] for nm in ("q", "k", "v", "do"))
        ro, rl = oracle.attention_forward_head(qb, kb, vb, base.scale, causal)
        rdq, rdk, rdv, _ = oracle.attention_backward_head(qb, kb, vb, db, base.scale, causal)
        ref[b] = {"O": ro, "LSE": rl, "dQ": rdq, "dK": rdk, "dV": rdv}
    errs = {}
    for i, h in enumerate(heads):
        for nm in ("O", "LSE", "dQ", "dK", "dV"):
            errs["%s[h%d]" % (nm, h)] = relerr(got[nm][i], ref[h % NBASE][nm])
    assert all(e <= TOL["bf16"] for e in errs.values()), errs
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()
