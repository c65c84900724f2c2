"""Pins for the float64 oracle, independent of the oracle's own code.

Each check compares the oracle against something other than itself:
hand-derived values, brute-force loops with the explicit softmax Jacobian,
central finite differences, torch's float64 CPU attention with autograd,
closed forms and invariants that follow from the mathematics.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import (attention_backward, attention_backward_head,
                    attention_backward_head_sampled, attention_forward,
                    attention_forward_head)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------------------
# hand-derived example


@pytest.mark.parametrize("mode", ["noncausal", "causal"])
def test_hand_example(mode):
    fx = json.load(open(os.path.join(GOLDEN, "hand_example_n2_d1.json")))
    q, k, v, do = (np.array(fx[x]) for x in ("Q", "K", "V", "dO"))
    causal = mode == "causal"
    o, lse = attention_forward_head(q, k, v, fx["scale"], causal)
    dq, dk, dv, D = attention_backward_head(q, k, v, do, fx["scale"], causal)
    exp = fx[mode]
    np.testing.assert_allclose(o, exp["O"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, exp["LSE"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dq, exp["dQ"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk, exp["dK"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv, exp["dV"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(D, exp["D"], rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# brute force, pure Python loops, explicit softmax Jacobian


def _brute(q, k, v, do, scale, causal):
    n, d = len(q), len(q[0])
    dv_cols = len(v[0])
    allowed = [[(not causal) or j <= i for j in range(n)] for i in range(n)]
    P = [[0.0] * n for _ in range(n)]
    O = [[0.0] * dv_cols for _ in range(n)]
    LSE = [0.0] * n
    for i in range(n):
        s = {}
        for j in range(n):
            if allowed[i][j]:
                s[j] = scale * sum(q[i][c] * k[j][c] for c in range(d))
        mx = max(s.values())
        tot = sum(math.exp(x - mx) for x in s.values())
        for j, x in s.items():
            P[i][j] = math.exp(x - mx) / tot
        LSE[i] = mx + math.log(tot)
        for c in range(dv_cols):
            O[i][c] = sum(P[i][j] * v[j][c] for j in range(n))
    # g_ij = dL/dP_ij = dO_i . v_j ; dL/ds_il = sum_j g_ij P_ij (delta_jl - P_il)
    dS = [[0.0] * n for _ in range(n)]
    for i in range(n):
        g = [sum(do[i][c] * v[j][c] for c in range(dv_cols)) for j in range(n)]
        for l in range(n):
            if not allowed[i][l]:
                continue
            acc = 0.0
            for j in range(n):
                if allowed[i][j]:
                    jac = P[i][j] * ((1.0 if j == l else 0.0) - P[i][l])
                    acc += g[j] * jac
            dS[i][l] = acc
    dQ = [[scale * sum(dS[i][l] * k[l][c] for l in range(n)) for c in range(d)]
          for i in range(n)]
    dK = [[scale * sum(dS[i][l] * q[i][c] for i in range(n)) for c in range(d)]
          for l in range(n)]
    dV = [[sum(P[i][j] * do[i][c] for i in range(n)) for c in range(dv_cols)]
          for j in range(n)]
    return O, LSE, dQ, dK, dV


@pytest.mark.parametrize("n,d,causal,seed", [
    (1, 3, False, 1), (2, 2, True, 2), (5, 4, False, 3), (7, 3, True, 4),
    (8, 5, False, 5), (8, 2, True, 6)])
def test_bruteforce(n, d, causal, seed):
    rng = _rng(seed)
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    scale = 0.7
    O, LSE, dQ, dK, dV = _brute(q.tolist(), k.tolist(), v.tolist(),
                                do.tolist(), scale, causal)
    o, lse = attention_forward_head(q, k, v, scale, causal)
    dq, dk, dv, _ = attention_backward_head(q, k, v, do, scale, causal)
    for a, b in ((o, O), (lse, LSE), (dq, dQ), (dk, dK), (dv, dV)):
        np.testing.assert_allclose(a, np.array(b), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# central finite differences of L = sum(dO o O)


@pytest.mark.parametrize("n,d,causal,seed", [(6, 3, False, 11), (16, 8, True, 12),
                                             (9, 5, True, 13)])
def test_finite_differences(n, d, causal, seed):
    rng = _rng(seed)
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    scale = 1.0 / math.sqrt(d)

    def loss(qq, kk, vv):
        o, _ = attention_forward_head(qq, kk, vv, scale, causal)
        return float((o * do).sum())

    dq, dk, dv, _ = attention_backward_head(q, k, v, do, scale, causal)
    h = 1e-5
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        fd = np.zeros_like(grad)
        for i in range(n):
            for c in range(d):
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[which][i, c] += h
                args_m[which][i, c] -= h
                fd[i, c] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(fd - grad).max() / max(np.abs(grad).max(), 1e-30)
        assert err < 1e-7, (which, err)


# ---------------------------------------------------------------------------
# torch float64 CPU attention + autograd (a library routine, used as a check)


@pytest.mark.parametrize("n,d,causal", [(33, 16, False), (64, 32, True),
                                        (100, 8, True)])
def test_torch_sdpa_fp64(n, d, causal):
    g = torch.Generator().manual_seed(n * 7 + d)
    q, k, v, do = (torch.randn(2, 3, n, d, generator=g, dtype=torch.float64)
                   for _ in range(4))
    scale = 1.0 / math.sqrt(d)
    qt, kt, vt = (x.clone().requires_grad_(True) for x in (q, k, v))
    ot = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, is_causal=causal, scale=scale)
    ot.backward(do)
    o, lse = attention_forward(q, k, v, scale, causal)
    dq, dk, dv, _ = attention_backward(q, k, v, do, scale, causal)
    np.testing.assert_allclose(o, ot.detach().numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=1e-10, atol=1e-12)
    # LSE against scipy's logsumexp over the masked scores
    from scipy.special import logsumexp

    s = scale * np.einsum("bhid,bhjd->bhij", q.numpy(), k.numpy())
    if causal:
        s = np.where(np.triu(np.ones((n, n), bool), 1), -np.inf, s)
    np.testing.assert_allclose(lse, logsumexp(s, axis=-1), rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------------------
# closed forms


def test_q_zero_noncausal_is_mean():
    rng = _rng(21)
    n, d = 37, 6
    q = np.zeros((n, d))
    k, v, do = (_rand(rng, n, d) for _ in range(3))
    o, lse = attention_forward_head(q, k, v, 0.3, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(0), (n, d)), atol=1e-14)
    np.testing.assert_allclose(lse, np.log(n), atol=1e-14)
    dq, dk, dv, _ = attention_backward_head(q, k, v, do, 0.3, False)
    np.testing.assert_allclose(dk, 0.0, atol=1e-15)          # Q = 0 => dK = 0
    np.testing.assert_allclose(dv, np.broadcast_to(do.sum(0) / n, (n, d)), atol=1e-14)


def test_q_zero_causal_is_prefix_mean():
    rng = _rng(22)
    n, d = 29, 4
    q = np.zeros((n, d))
    k, v = _rand(rng, n, d), _rand(rng, n, d)
    o, lse = attention_forward_head(q, k, v, 0.5, True)
    prefix = np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(o, prefix, atol=1e-14)
    np.testing.assert_allclose(lse, np.log(np.arange(1, n + 1)), atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_single_row(causal):
    rng = _rng(23)
    q, k, v, do = (_rand(rng, 1, 9) for _ in range(4))
    o, lse = attention_forward_head(q, k, v, 0.25, causal)
    np.testing.assert_allclose(o, v, atol=1e-15)
    np.testing.assert_allclose(lse, 0.25 * (q * k).sum(), atol=1e-15)
    dq, dk, dv, _ = attention_backward_head(q, k, v, do, 0.25, causal)
    np.testing.assert_allclose(dq, 0.0, atol=1e-15)
    np.testing.assert_allclose(dk, 0.0, atol=1e-15)
    np.testing.assert_allclose(dv, do, atol=1e-15)


def test_causal_first_row_and_last_key():
    rng = _rng(24)
    n, d = 20, 5
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    scale = 0.4
    o, lse = attention_forward_head(q, k, v, scale, True)
    np.testing.assert_allclose(o[0], v[0], atol=1e-15)
    np.testing.assert_allclose(lse[0], scale * q[0] @ k[0], atol=1e-14)
    # only the last query row sees the last key: dV_{n-1} = P_{n-1,n-1} dO_{n-1}
    p_last = math.exp(scale * q[-1] @ k[-1] - lse[-1])
    _, _, dv, _ = attention_backward_head(q, k, v, do, scale, True)
    np.testing.assert_allclose(dv[-1], p_last * do[-1], rtol=1e-12)


# ---------------------------------------------------------------------------
# invariants


@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(causal):
    # with V = I the output rows are the rows of P
    rng = _rng(31)
    n, d = 24, 7
    q, k = _rand(rng, n, d), _rand(rng, n, d)
    p, _ = attention_forward_head(q, k, np.eye(n), 0.8, causal)
    np.testing.assert_allclose(p.sum(1), 1.0, atol=1e-14)
    assert (p >= 0).all()
    if causal:
        assert np.abs(np.triu(p, 1)).max() == 0.0


@pytest.mark.parametrize("causal", [False, True])
def test_lse_bounds(causal):
    rng = _rng(32)
    n, d = 40, 6
    q, k, v = (3 * _rand(rng, n, d) for _ in range(3))
    scale = 0.6
    _, lse = attention_forward_head(q, k, v, scale, causal)
    s = scale * q @ k.T
    if causal:
        s = np.where(np.triu(np.ones((n, n), bool), 1), -np.inf, s)
    m = s.max(1)
    cnt = np.arange(1, n + 1) if causal else np.full(n, n)
    assert (lse >= m - 1e-12).all()
    assert (lse <= m + np.log(cnt) + 1e-12).all()


@pytest.mark.parametrize("causal", [False, True])
def test_shift_invariances(causal):
    rng = _rng(33)
    n, d = 18, 5
    q, k, v = (_rand(rng, n, d) for _ in range(3))
    o, _ = attention_forward_head(q, k, v, 0.5, causal)
    c = _rand(rng, d)
    o2, _ = attention_forward_head(q, k, v + c, 0.5, causal)   # O shifts by c
    np.testing.assert_allclose(o2, o + c, atol=1e-13)
    o3, _ = attention_forward_head(q, k + c, v, 0.5, causal)   # row-constant score shift
    np.testing.assert_allclose(o3, o, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_invariants(causal):
    rng = _rng(34)
    n, d = 31, 6
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    scale = 0.45
    dq, dk, dv, D = attention_backward_head(q, k, v, do, scale, causal)
    o, _ = attention_forward_head(q, k, v, scale, causal)
    np.testing.assert_allclose(D, (do * o).sum(1), atol=1e-13)      # D_i = dO_i . O_i
    np.testing.assert_allclose(dk.sum(0), 0.0, atol=1e-13)          # rowsum(dS) = 0
    np.testing.assert_allclose(dv.sum(0), do.sum(0), atol=1e-13)     # rows of P sum to 1
    np.testing.assert_allclose((q * dq).sum(), (k * dk).sum(), atol=1e-12)
    p, _ = attention_forward_head(q, k, np.eye(n), scale, causal)
    np.testing.assert_allclose(dv, p.T @ do, atol=1e-13)             # dV = P^T dO


def test_sampled_backward_matches_full():
    rng = _rng(35)
    n, d = 600, 8   # spans several of the oracle's row groups
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv, D = attention_backward_head(q, k, v, do, 0.3, causal)
        qr = np.array([0, 5, 255, 256, 599])
        kr = np.array([1, 300, 598])
        sq, sk, sv, sD = attention_backward_head_sampled(q, k, v, do, 0.3, causal,
                                                         qr, kr)
        np.testing.assert_allclose(sq, dq[qr], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(sk, dk[kr], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(sv, dv[kr], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(sD, D, rtol=1e-13, atol=1e-14)
        o, lse = attention_forward_head(q, k, v, 0.3, causal)
        o2, lse2 = attention_forward_head(q, k, v, 0.3, causal, rows=qr)
        np.testing.assert_allclose(o2, o[qr], rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(lse2, lse[qr], rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------------------
# the blocked online-softmax update read from the pages


def _blocked_forward(q, k, v, scale, block, keep_l_old):
    """Q-outer, KV-inner block loop with running max m and sum l per row."""
    n, d = q.shape
    o = np.zeros_like(v)
    for i in range(0, n, block):
        qi = q[i:i + block]
        m = np.full(qi.shape[0], -np.inf)
        l = np.zeros(qi.shape[0])
        oi = np.zeros((qi.shape[0], v.shape[1]))
        for j in range(0, n, block):
            s = scale * qi @ k[j:j + block].T
            m_new = np.maximum(m, s.max(1))
            e = np.exp(s - m_new[:, None])
            alpha = np.exp(m - m_new)
            l_new = alpha * l + e.sum(1)
            if keep_l_old:   # O kept normalised: rescale by alpha * l_old / l_new
                oi = (alpha[:, None] * l[:, None] * oi + e @ v[j:j + block]) / l_new[:, None]
            else:            # update as printed: the l_old factor is missing
                oi = (alpha[:, None] * oi + e @ v[j:j + block]) / l_new[:, None]
            m, l = m_new, l_new
        o[i:i + block] = oi
    return o


def test_online_softmax_reading():
    rng = _rng(41)
    n, d = 70, 8
    q, k, v = (_rand(rng, n, d) for _ in range(3))
    ref, _ = attention_forward_head(q, k, v, 0.35, False)
    fixed = _blocked_forward(q, k, v, 0.35, 16, keep_l_old=True)
    np.testing.assert_allclose(fixed, ref, rtol=1e-12, atol=1e-13)
    printed = _blocked_forward(q, k, v, 0.35, 16, keep_l_old=False)
    assert np.abs(printed - ref).max() > 1e-2     # the printed form is not exact


def test_quadratic_cost_fixture():
    from io_aware_exact_05_gb300.flops import attention_flops, score_entries

    fx = json.load(open(os.path.join(GOLDEN, "quadratic_cost.json")))
    for e in fx["score_entries"]:
        assert score_entries(e["n"]) == e["entries"]
    for r in fx["cost_ratio"]:
        n = 1024
        a = attention_flops(1, 1, n, 64, causal=False)
        b = attention_flops(1, 1, n * r["length_ratio"], 64, causal=False)
        assert b["fwd"] == r["cost_ratio"] * a["fwd"]
        assert b["bwd"] == r["cost_ratio"] * a["bwd"]


# ---------------------------------------------------------------------------
# grouped-query attention: H query heads share H_kv key/value heads


@pytest.mark.parametrize("H,Hkv,causal", [(4, 2, False), (3, 1, True), (6, 3, True)])
def test_gqa_finite_differences(H, Hkv, causal):
    # L = sum over every query head of sum(dO o O); the gradient with respect
    # to a shared key/value element is checked by central differences, which
    # knows nothing of how the oracle combines the heads of a group.
    rng = _rng(50 + H + Hkv)
    B, n, d = 2, 5, 3
    q, do = _rand(rng, B, H, n, d), _rand(rng, B, H, n, d)
    k, v = _rand(rng, B, Hkv, n, d), _rand(rng, B, Hkv, n, d)
    scale = 0.7

    def loss(kk, vv, qq=q):
        o, _ = attention_forward(qq, kk, vv, scale, causal)
        return float((o * do).sum())

    dq, dk, dv, _ = attention_backward(q, k, v, do, scale, causal)
    assert dk.shape == k.shape and dv.shape == v.shape and dq.shape == q.shape
    h = 1e-5
    for which, grad in ((0, dk), (1, dv)):
        fd = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            kp, vp = k.copy(), v.copy()
            km, vm = k.copy(), v.copy()
            (kp if which == 0 else vp)[idx] += h
            (km if which == 0 else vm)[idx] -= h
            fd[idx] = (loss(kp, vp) - loss(km, vm)) / (2 * h)
        err = np.abs(fd - grad).max() / np.abs(grad).max()
        assert err < 1e-7, (which, err)
    fdq = np.zeros_like(dq)
    for idx in np.ndindex(*dq.shape):
        qp, qm = q.copy(), q.copy()
        qp[idx] += h
        qm[idx] -= h
        fdq[idx] = (loss(k, v, qp) - loss(k, v, qm)) / (2 * h)
    assert np.abs(fdq - dq).max() / np.abs(dq).max() < 1e-7


def test_gqa_one_kv_head_per_query_head_and_repeat():
    # H_kv = H is plain multi-head attention; a group of g heads equals
    # multi-head attention on K, V repeated g times, with dK, dV summed back.
    rng = _rng(60)
    B, H, n, d, g = 1, 4, 7, 5, 2
    q, do = _rand(rng, B, H, n, d), _rand(rng, B, H, n, d)
    k, v = _rand(rng, B, H // g, n, d), _rand(rng, B, H // g, n, d)
    kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    o_g, l_g = attention_forward(q, k, v, 0.5, True)
    o_r, l_r = attention_forward(q, kr, vr, 0.5, True)
    np.testing.assert_array_equal(o_g, o_r)
    np.testing.assert_array_equal(l_g, l_r)
    dq_g, dk_g, dv_g, _ = attention_backward(q, k, v, do, 0.5, True)
    dq_r, dk_r, dv_r, _ = attention_backward(q, kr, vr, do, 0.5, True)
    np.testing.assert_array_equal(dq_g, dq_r)
    np.testing.assert_allclose(dk_g, dk_r.reshape(B, H // g, g, n, d).sum(2), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dv_g, dv_r.reshape(B, H // g, g, n, d).sum(2), rtol=1e-13, atol=1e-14)
    with pytest.raises(ValueError):
        attention_forward(q, k[:, :1].repeat(3, axis=1), v[:, :1].repeat(3, axis=1))


# ---------------------------------------------------------------------------
# block-sparse attention: scores outside the kept blocks are removed


def _sparse_rows_loop(q, k, v, scale, causal, mask, block):
    # per row: a plain softmax over the kept keys only, written with loops
    n = q.shape[0]
    o = np.zeros_like(v)
    lse = np.full(n, -np.inf)
    for i in range(n):
        keys = [j for j in range(n)
                if mask[i // block, j // block] and (not causal or j <= i)]
        if not keys:
            continue
        s = [scale * sum(q[i, c] * k[j, c] for c in range(q.shape[1])) for j in keys]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        tot = sum(e)
        lse[i] = m + math.log(tot)
        for jj, j in enumerate(keys):
            o[i] += e[jj] / tot * v[j]
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_block_sparse_matches_kept_key_loops(causal):
    rng = _rng(70 + causal)
    n, d, block = 22, 3, 4
    q, k, v = (_rand(rng, n, d) for _ in range(3))
    nb = (n + block - 1) // block
    mask = rng.random((nb, nb)) < 0.45
    mask[2, :] = False                       # block row 2: rows 8..11 keep nothing
    o, lse = attention_forward_head(q, k, v, 0.6, causal, None, mask, block)
    ro, rl = _sparse_rows_loop(q, k, v, 0.6, causal, mask, block)
    np.testing.assert_allclose(o, ro, rtol=1e-12, atol=1e-13)
    assert np.array_equal(np.isinf(lse), np.isinf(rl))
    fin = np.isfinite(rl)
    np.testing.assert_allclose(lse[fin], rl[fin], rtol=1e-12)
    assert np.all(o[8:12] == 0.0) and np.all(np.isneginf(lse[8:12]))


@pytest.mark.parametrize("causal", [False, True])
def test_block_sparse_finite_differences(causal):
    rng = _rng(80 + causal)
    n, d, block = 9, 3, 3
    q, k, v, do = (_rand(rng, n, d) for _ in range(4))
    mask = np.array([[1, 0, 1], [0, 1, 0], [1, 1, 0]], dtype=bool)
    mask_empty = mask.copy()
    mask_empty[1] = False                    # rows 3..5 attend to nothing

    for m in (mask, mask_empty):
        def loss(qq, kk, vv):
            o, _ = attention_forward_head(qq, kk, vv, 0.5, causal, None, m, block)
            return float((o * do).sum())

        dq, dk, dv, _ = attention_backward_head(q, k, v, do, 0.5, causal, m, block)
        h = 1e-5
        for which, grad in ((0, dq), (1, dk), (2, dv)):
            fd = np.zeros_like(grad)
            for idx in np.ndindex(*grad.shape):
                ap = [q.copy(), k.copy(), v.copy()]
                am = [q.copy(), k.copy(), v.copy()]
                ap[which][idx] += h
                am[which][idx] -= h
                fd[idx] = (loss(*ap) - loss(*am)) / (2 * h)
            err = np.abs(fd - grad).max() / max(np.abs(grad).max(), 1e-30)
            assert err < 1e-7, (which, err)
    _, _, _, D = attention_backward_head(q, k, v, do, 0.5, causal, mask_empty, block)
    dq, _, _, _ = attention_backward_head(q, k, v, do, 0.5, causal, mask_empty, block)
    assert np.all(dq[3:6] == 0.0) and np.all(D[3:6] == 0.0)


def test_block_sparse_all_ones_is_dense():
    rng = _rng(90)
    q, k, v, do = (_rand(rng, 2, 2, 40, 6) for _ in range(4))
    ones = np.ones((3, 3), dtype=bool)
    for causal in (False, True):
        a = attention_forward(q, k, v, 0.4, causal)
        b = attention_forward(q, k, v, 0.4, causal, ones, 16)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])
        ga = attention_backward(q, k, v, do, 0.4, causal)
        gb = attention_backward(q, k, v, do, 0.4, causal, ones, 16)
        for x, y in zip(ga, gb):
            np.testing.assert_array_equal(x, y)
