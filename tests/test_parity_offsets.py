"""Parity with every tensor starting 16 bytes into its allocation (the
weakest alignment the boundary accepts), so that no kernel may assume more:
TMA tensor maps, vector loads and stores, the fp32 accumulators and the
row statistics all run from these base addresses.  Inputs and outputs of
the forward and the backward, in bf16 at every head dim and in fp32, both
masks and both dQ modes, on a ragged length; every element is compared with
the float64 oracle."""

import pytest
import torch

import oracle
from io_aware_exact_05_gb300.inputs import Workload, make_inputs
from parity_util import TOL, relerr

pytestmark = pytest.mark.gpu


def _offset_like(shape, dtype, dev):
    """A contiguous tensor of `shape` whose first element is 16 bytes past the
    start of its allocation."""
    shift = 16 // torch.empty((), dtype=dtype).element_size()
    n = 1
    for s in shape:
        n *= s
    buf = torch.empty(n + shift, dtype=dtype, device=dev)
    t = buf[shift:].view(shape)
    assert t.data_ptr() % 16 == 0 and t.data_ptr() % 32 != 0
    return t


CASES = [(d, "bf16", c, m) for d in (64, 128, 256) for c in (False, True) for m in ("auto", "pass")]
CASES += [(64, "f32", c, "auto") for c in (False, True)]


@pytest.mark.parametrize("d,dtype,causal,mode", CASES,
                         ids=["d%d_%s_%s_%s" % (d, t, "causal" if c else "full", m) for d, t, c, m in CASES])
def test_offset_pointers(cuda_dev, d, dtype, causal, mode):
    from io_aware_exact_05_gb300 import attn

    w = Workload("offsets", 1, 2, 333, d, dtype, causal, 1.0, 3300 + d)
    x = make_inputs(w)
    tdt = x["q"].dtype
    shape = (w.B, w.H, w.n, w.d)
    q, k, v, do = (_offset_like(shape, tdt, cuda_dev) for _ in range(4))
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (do, "do")):
        t.copy_(x[nm].to(cuda_dev))
    o, dq, dk, dv = (_offset_like(shape, tdt, cuda_dev) for _ in range(4))
    lse = _offset_like((w.B, w.H, w.n), torch.float32, cuda_dev)
    attn.attn_fwd(q, k, v, o, lse, w.scale, causal)
    m = attn.ATTN_DQ_PASS if mode == "pass" else attn.ATTN_DQ_AUTO
    attn.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, w.scale, causal, m)
    assert attn.attn_status() == 0
    ro, rl = oracle.attention_forward(x["q"], x["k"], x["v"], w.scale, causal)
    rdq, rdk, rdv, _ = oracle.attention_backward(x["q"], x["k"], x["v"], x["do"], w.scale, causal)
    errs = {"O": relerr(o, ro), "LSE": relerr(lse, rl), "dQ": relerr(dq, rdq),
            "dK": relerr(dk, rdk), "dV": relerr(dv, rdv)}
    assert all(e <= TOL[dtype] for e in errs.values()), errs
