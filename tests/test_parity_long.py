"""Parity at sequence lengths beyond the workloads' (n = 131072 and 2^20 at
d = 64 and 128, n = 65536 at d = 256, causal), through the default API
calls: row offsets up to 2^20 in every kernel, up to 8192 key tiles in a
causal grid, and (at
d = 256) the automatic dQ mode falling back to the query-tile pass because
the n x n dS^T buffer would exceed 4 GiB.

The float64 oracle cannot form a whole head at these lengths (n^2 d per
head), so it checks rows it can compute exactly in O(n d) each:
- a causal query row i is the one-row problem "q_i against keys 0..i, no
  mask", so O, LSE and dQ of sampled query rows are exact;
- key j receives gradient only from query rows i >= j, so dK and dV of the
  last 16 keys are the sum over the last 16 query rows' one-row backward
  passes.
Every element of those rows is compared (max|err| / max|ref| per output)."""

import numpy as np
import pytest

import oracle
from io_aware_exact_05_gb300.inputs import Workload, make_inputs
from parity_util import TOL, relerr

LAST_KEYS = 16
CASES = [
    Workload("long_n128k_d64", 1, 2, 131072, 64, "bf16", True, 1.0, 2910),
    Workload("long_n128k_d128", 1, 2, 131072, 128, "bf16", True, 1.0, 2920),
    Workload("long_n64k_d256", 1, 1, 65536, 256, "bf16", True, 1.0, 2930),
    Workload("long_n1m_d64", 1, 1, 1 << 20, 64, "bf16", True, 1.0, 2950),
    Workload("long_n1m_d128", 1, 1, 1 << 20, 128, "bf16", True, 1.0, 2960),
]


def _rows(n, seed):
    fixed = [0, 1, 127, 128, n // 2 - 1, n // 2, n - 129, n - LAST_KEYS - 1, n - 1]
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([fixed, rng.choice(n, size=8, replace=False)]))


def _one_row_backward(q, k, v, do, scale, i, k_rows):
    """dQ_i and the contributions of query row i to dK, dV at k_rows (<= i)."""
    dq, dk, dv, _ = oracle.attention_backward_head_sampled(
        q[i:i + 1], k[:i + 1], v[:i + 1], do[i:i + 1], scale, False,
        q_rows=np.array([0]), k_rows=np.asarray(k_rows))
    return dq[0], dk, dv


def _reference_rows(x, w, hh, rows):
    """O, LSE, dQ at `rows` and dK, dV of the last LAST_KEYS keys of head hh."""
    BH, n, d = w.B * w.H, w.n, w.d
    qh, kh, vh, dh = (np.asarray(x[nm].reshape(BH, n, d)[hh].double()) for nm in ("q", "k", "v", "do"))
    ro, rl = oracle.attention_forward_head(qh, kh, vh, w.scale, True, rows=rows)
    rdq = np.stack([_one_row_backward(qh, kh, vh, dh, w.scale, int(i), [int(i)])[0] for i in rows])
    last = np.arange(n - LAST_KEYS, n)
    rdk = np.zeros((LAST_KEYS, d))
    rdv = np.zeros((LAST_KEYS, d))
    for i in last:
        keys = last[last <= i]
        _, ck, cv = _one_row_backward(qh, kh, vh, dh, w.scale, int(i), keys)
        rdk[:keys.size] += ck
        rdv[:keys.size] += cv
    return ro, rl, rdq, rdk, rdv


def test_row_decomposition_is_exact():
    """The rows above equal the whole-head oracle's on a short causal head."""
    w = Workload("long_check", 1, 1, 300, 64, "bf16", True, 1.0, 2940)
    x = make_inputs(w)
    rows = _rows(w.n, w.seed)
    ro, rl, rdq, rdk, rdv = _reference_rows(x, w, 0, rows)
    q, k, v, do = (np.asarray(x[nm][0, 0].double()) for nm in ("q", "k", "v", "do"))
    fo, fl = oracle.attention_forward_head(q, k, v, w.scale, True)
    fdq, fdk, fdv, _ = oracle.attention_backward_head(q, k, v, do, w.scale, True)
    last = np.arange(w.n - LAST_KEYS, w.n)
    for a, b in ((ro, fo[rows]), (rl, fl[rows]), (rdq, fdq[rows]), (rdk, fdk[last]), (rdv, fdv[last])):
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(b).max())


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_long_sequence(cuda_dev, w):
    from io_aware_exact_05_gb300 import attn

    x = make_inputs(w)
    q, k, v, do = (x[n].to(cuda_dev) for n in ("q", "k", "v", "do"))
    o, lse = attn.forward(q, k, v, causal=w.causal)
    dq, dk, dv = attn.backward(q, k, v, o, do, lse, causal=w.causal)
    assert attn.attn_status() == 0
    BH, n, d = w.B * w.H, w.n, w.d
    got = {nm: t.float().cpu().reshape(BH, n, -1).numpy() for nm, t in
           (("O", o), ("dQ", dq), ("dK", dk), ("dV", dv))}
    got_lse = lse.float().cpu().reshape(BH, n).numpy()
    rows = _rows(n, w.seed)
    last = np.arange(n - LAST_KEYS, n)
    errs = {}
    for hh in range(BH):
        ro, rl, rdq, rdk, rdv = _reference_rows(x, w, hh, rows)
        for name, g, ref in (("O", got["O"][hh][rows], ro), ("LSE", got_lse[hh][rows], rl),
                             ("dQ", got["dQ"][hh][rows], rdq), ("dK", got["dK"][hh][last], rdk),
                             ("dV", got["dV"][hh][last], rdv)):
            errs["%s[h%d]" % (name, hh)] = relerr(g, ref)
    assert all(e <= TOL["bf16"] for e in errs.values()), errs
