"""Device-side failure detection, without a GPU fault: a bounded wait that
nothing completes must end, record ATTN_ERR_DEVICE_TIMEOUT for the host, and
leave the context usable."""

import pytest

import oracle
from io_aware_exact_05_gb300.inputs import Workload, make_inputs
from parity_util import TOL, relerr

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda_dev):
    from io_aware_exact_05_gb300 import attn

    assert attn.attn_status() == attn.ATTN_OK
    attn.attn_selftest_wait_timeout(2_000_000)          # 2 ms, no arrival
    assert attn.attn_status() == attn.ATTN_ERR_DEVICE_TIMEOUT
    assert attn.attn_status() == attn.ATTN_OK           # read and cleared
    # the same context still computes correct results
    w = Workload("after_timeout", 1, 2, 300, 128, "bf16", True, 1.0, 1900)
    x = make_inputs(w)
    q, k, v = (x[n].to(cuda_dev) for n in ("q", "k", "v"))
    o, lse = attn.forward(q, k, v, causal=True)
    assert attn.attn_status() == attn.ATTN_OK
    ro, rl = oracle.attention_forward(x["q"], x["k"], x["v"], w.scale, True)
    assert relerr(o, ro) <= TOL["bf16"] and relerr(lse, rl) <= TOL["bf16"]
