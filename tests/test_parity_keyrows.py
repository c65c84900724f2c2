"""The IO study's key-tile instances (attn_bwd_dkdv_keys: a CTA owns 64 or 32
of its 128 key rows) against the float64 oracle: every element of dQ, dK
and dV on ragged shapes, both masks and every head dim, through the C ABI
and the same stage sequence as the benchmark (preprocess, key-tile kernel,
dQ stage)."""

import pytest
import torch

import oracle
from io_aware_exact_05_gb300.inputs import Workload, make_inputs
from parity_util import TOL, relerr

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows", [32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_key_rows(cuda_dev, d, causal, rows):
    from io_aware_exact_05_gb300 import attn

    w = Workload("keyrows", 1, 2, 333, d, "bf16", causal, 1.0, 2700 + d + rows)
    x = make_inputs(w)
    q, k, v, do = (x[n].to(cuda_dev) for n in ("q", "k", "v", "do"))
    o, lse = attn.forward(q, k, v, causal=causal)
    mode = attn.ATTN_DQ_PASS if d == 256 else attn.ATTN_DQ_ATOMIC
    ws = torch.empty(attn.attn_bwd_workspace_size(1, 2, w.n, d, attn.ATTN_BF16, causal, mode),
                     dtype=torch.uint8, device=cuda_dev)
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    attn.attn_bwd_preprocess(o, do, lse, causal, mode, ws)
    attn.attn_bwd_dkdv_keys(q, k, v, do, dk, dv, w.scale, causal, mode, rows, ws)
    attn.attn_bwd_dq(q, k, v, do, dq, w.scale, causal, mode, ws)
    assert attn.attn_status() == 0
    rdq, rdk, rdv, _ = oracle.attention_backward(x["q"], x["k"], x["v"], x["do"], w.scale, causal)
    errs = {"dQ": relerr(dq, rdq), "dK": relerr(dk, rdk), "dV": relerr(dv, rdv)}
    assert all(e <= TOL["bf16"] for e in errs.values()), (rows, errs)
