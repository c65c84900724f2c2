"""Concurrent use: two host threads, each on its own CUDA stream, run forward
and backward passes at the same time on different inputs (ctypes releases
the interpreter lock during each library call, so the calls overlap on the
host and the kernels on the device).  The boundary keeps no per-call global
state (tensor maps are built per call and passed by value); every result
must still match the float64 oracle."""

import threading

import pytest
import torch

import oracle
from io_aware_exact_05_gb300.inputs import Workload, make_inputs
from parity_util import TOL, relerr

pytestmark = pytest.mark.gpu

ROUNDS = 4


def test_two_threads_two_streams(cuda_dev):
    from io_aware_exact_05_gb300 import attn

    works = [Workload("conc_a", 1, 4, 333, 64, "bf16", True, 1.0, 3400),
             Workload("conc_b", 2, 2, 520, 128, "bf16", False, 1.0, 3401)]
    xs = [make_inputs(w) for w in works]
    refs = []
    for w, x in zip(works, xs):
        ro, rl = oracle.attention_forward(x["q"], x["k"], x["v"], w.scale, w.causal)
        rdq, rdk, rdv, _ = oracle.attention_backward(x["q"], x["k"], x["v"], x["do"], w.scale, w.causal)
        refs.append((ro, rl, rdq, rdk, rdv))
    results = [[None] * ROUNDS for _ in works]
    failures = []

    def run(i):
        try:
            w, x = works[i], xs[i]
            stream = torch.cuda.Stream(device=cuda_dev)
            with torch.cuda.stream(stream):
                q, k, v, do = (x[n].to(cuda_dev, non_blocking=False) for n in ("q", "k", "v", "do"))
                for r in range(ROUNDS):
                    o, lse = attn.forward(q, k, v, causal=w.causal)
                    dq, dk, dv = attn.backward(q, k, v, o, do, lse, causal=w.causal)
                    results[i][r] = tuple(t.float().cpu() for t in (o, lse, dq, dk, dv))
            stream.synchronize()
        except Exception as e:   # reported on the main thread
            failures.append((i, repr(e)))

    threads = [threading.Thread(target=run, args=(i,)) for i in range(len(works))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not failures, failures
    assert attn.attn_status() == 0
    for i, w in enumerate(works):
        for r in range(ROUNDS):
            errs = {nm: relerr(g, ref) for nm, g, ref in
                    zip(("O", "LSE", "dQ", "dK", "dV"), results[i][r], refs[i])}
            assert all(e <= TOL["bf16"] for e in errs.values()), (w.name, r, errs)
