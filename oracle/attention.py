"""Float64 CPU oracle for exact softmax attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
module.  The library never calls it and shares no code with it.

What is computed (per head, Q, K, V, dO of shape (n, d)):

  forward  -- the definition of scaled dot-product attention,
              O = softmax(Q K^T * scale) V, with scale = 1/sqrt(d) by default
              ("Chapter 3.1 -- The cost of attention", section 2, the
              scaled dot-product formula; "Flash Attention: Revolutionizing
              Transformer Efficiency", section "Standard attention: a quick
              summary", the attention equation and the PyTorch listing that
              follows it).  The row softmax subtracts the row maximum first
              (same blog post, "The mathematics behind Flash Attention",
              formula 1), and the oracle is two-pass per row, never online.
              Alongside O it returns the natural-log row logsumexp
              LSE_i = m_i + ln(sum_j exp(s_ij - m_i)).

  backward -- none of the pages prints the backward formulas; they only say
              that the backward pass differentiates the same function and
              recomputes the attention matrix ("Chapter 3.1", section 5;
              "On the fine-grained I/O complexity of attention backward
              passes", Methodology step 1).  The plainest reading is the
              exact chain-rule derivative of the forward map for a scalar
              loss whose gradient with respect to O is dO:
                  dV = P^T dO
                  dP = dO V^T
                  D_i = sum_j P_ij dP_ij
                  dS = P o (dP - D 1^T)
                  dQ = scale * dS K
                  dK = scale * dS^T Q

  causal   -- optional mask s_ij = -inf for j > i, applied before the row
              maximum (so P_ij = 0 there).  Every row keeps j = i.

  block mask -- optional block-sparse pattern: a boolean matrix over blocks
              of `block` (default 128) query rows x `block` keys; scores in
              a False block are -inf, the rest are exact.  This is sparse
              attention over a block pattern ("Chapter 3.1", section 3:
              local windows, global tokens and random links of Longformer
              and BigBird; "On the fine-grained I/O complexity of attention
              backward passes", item 2, sparse attention with Z_QK kept
              entries), computed exactly on the kept entries.  The pages
              are silent on a row with no kept score; the plain reading
              taken here is that it attends to nothing: O_i = 0,
              LSE_i = -inf, and it contributes nothing to any gradient.

Each step is the definition written out with numpy float64 arithmetic; the
only library primitive is the matrix product.  Large heads are processed a
group of query rows at a time purely to bound memory: every row is computed
exactly as the per-row definition says, and the sums over rows for dK and dV
are accumulated in the order of the groups.

Pinned by tests/test_oracle.py against: hand-derived values for a 2x1
example (tests/golden/hand_example_n2_d1.json), brute-force per-element
loops with the explicit softmax Jacobian at n <= 8, central finite
differences of L = sum(dO o O), torch's float64 CPU scaled-dot-product
attention with autograd, closed forms (Q = 0, n = 1, causal row 0) and
invariants (rows of P sum to 1, LSE bounds, shift invariances,
rowsum(dS) = 0, sum_j dV_j = sum_i dO_i, <Q,dQ> = <K,dK>).  The grouped-query
form (fewer key/value heads) is pinned by central finite differences with
respect to the shared K and V, and by its one-key/value-head-per-query-head
special case.
"""

import numpy as np

__all__ = [
    "attention_forward",
    "attention_backward",
    "attention_forward_head",
    "attention_backward_head",
    "attention_backward_head_sampled",
    "default_scale",
]

_ROW_GROUP = 256


def default_scale(d):
    """scale = 1/sqrt(d): the QK^T divisor of the attention definition."""
    return 1.0 / np.sqrt(float(d))


def _as_f64(x):
    """Exact upcast of whatever the caller holds (float32, bfloat16 via
    torch, float64) to a float64 numpy array."""
    try:
        import torch  # only for converting torch tensors the tests pass in

        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _scores(q_rows, k, scale, row_index, causal, block_mask=None, block=128):
    """s_ij = scale * q_i . k_j for the requested query rows i; -inf where
    the causal mask removes j > i, and where the block mask removes the
    (i // block, j // block) block."""
    s = scale * (q_rows @ k.T)
    if causal:
        cols = np.arange(k.shape[0])[None, :]
        s = np.where(cols > row_index[:, None], -np.inf, s)
    if block_mask is not None:
        keep = np.asarray(block_mask, dtype=bool)[row_index // block][:, np.arange(k.shape[0]) // block]
        s = np.where(keep, s, -np.inf)
    return s


def _row_softmax(s):
    """Two-pass softmax of each row: subtract the row maximum, exponentiate,
    divide by the row sum.  Returns P, the row maximum m and the row sum l.
    A row with no finite score (every key masked) has P = 0, m = -inf and
    l = 0."""
    m = s.max(axis=1)
    empty = ~np.isfinite(m)
    e = np.exp(s - np.where(empty, 0.0, m)[:, None])   # exp(-inf) = 0 off the mask
    l = e.sum(axis=1)
    p = e / np.where(empty, 1.0, l)[:, None]
    return p, m, l


def _lse(m, l):
    """LSE = m + ln l, and -inf for a row with no kept score (l = 0)."""
    out = np.full(m.shape, -np.inf)
    ok = l > 0
    out[ok] = m[ok] + np.log(l[ok])
    return out


def attention_forward_head(q, k, v, scale=None, causal=False, rows=None, block_mask=None,
                           block=128):
    """Forward pass of one head.

    q, k, v: (n, d).  rows: optional 1-D array of query indices to compute
    (default: all).  block_mask: optional boolean (ceil(n/block), ceil(n/block))
    array; scores outside its True blocks are masked (block-sparse exact
    attention).  Returns (O[rows], LSE[rows]) in float64; a row with no kept
    score gets O = 0 and LSE = -inf.
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    n, d = q.shape
    if scale is None:
        scale = default_scale(d)
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    o = np.empty((rows.size, v.shape[1]), dtype=np.float64)
    lse = np.empty(rows.size, dtype=np.float64)
    for g in range(0, rows.size, _ROW_GROUP):
        r = rows[g:g + _ROW_GROUP]
        s = _scores(q[r], k, scale, r, causal, block_mask, block)
        p, m, l = _row_softmax(s)
        o[g:g + r.size] = p @ v
        lse[g:g + r.size] = _lse(m, l)
    return o, lse


def attention_backward_head(q, k, v, do, scale=None, causal=False, block_mask=None,
                            block=128):
    """Backward pass of one head: exact gradients (dQ, dK, dV) of
    L = sum(dO o O) with respect to Q, K and V, plus D (length n)."""
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    n, d = q.shape
    return attention_backward_head_sampled(q, k, v, do, scale, causal,
                                           q_rows=np.arange(n),
                                           k_rows=np.arange(n),
                                           block_mask=block_mask, block=block)


def attention_backward_head_sampled(q, k, v, do, scale=None, causal=False,
                                    q_rows=None, k_rows=None, block_mask=None, block=128):
    """Backward pass of one head, returning only the requested rows.

    dQ is returned for the query indices ``q_rows``; dK and dV for the key
    indices ``k_rows``; D for all n rows.  dK_j and dV_j are sums over every
    query row i, so every row of P and dP is formed; nothing else is skipped.
    Returns (dQ[q_rows], dK[k_rows], dV[k_rows], D).
    """
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    n, d = q.shape
    dv_cols = v.shape[1]
    if scale is None:
        scale = default_scale(d)
    q_rows = np.arange(n) if q_rows is None else np.asarray(q_rows, np.int64)
    k_rows = np.arange(n) if k_rows is None else np.asarray(k_rows, np.int64)
    want_q = np.full(n, -1, dtype=np.int64)
    want_q[q_rows] = np.arange(q_rows.size)

    dq = np.zeros((q_rows.size, d))
    dk = np.zeros((k_rows.size, d))
    dv = np.zeros((k_rows.size, dv_cols))
    D = np.empty(n)
    for g in range(0, n, _ROW_GROUP):
        r = np.arange(g, min(g + _ROW_GROUP, n))
        s = _scores(q[r], k, scale, r, causal, block_mask, block)
        p, _, _ = _row_softmax(s)                 # P rows i in r
        dp = do[r] @ v.T                          # dP_ij = dO_i . v_j
        D[r] = (p * dp).sum(axis=1)               # D_i = sum_j P_ij dP_ij
        ds = p * (dp - D[r][:, None])             # dS = P o (dP - D)
        dv += p[:, k_rows].T @ do[r]              # dV_j += sum_i P_ij dO_i
        dk += scale * (ds[:, k_rows].T @ q[r])    # dK_j += scale sum_i dS_ij q_i
        sel = want_q[r]
        hit = sel >= 0
        if hit.any():                             # dQ_i = scale sum_j dS_ij k_j
            dq[sel[hit]] = scale * (ds[hit] @ k)
    return dq, dk, dv, D


def _group(H, H_kv):
    """Query heads per key/value head.  Grouped-query attention ("Flash
    Attention: Revolutionizing Transformer Efficiency", section
    FlashAttention-2, item 3): query head h reads key/value head h // g."""
    if H_kv < 1 or H % H_kv:
        raise ValueError("H_kv = %d must divide H = %d" % (H_kv, H))
    return H // H_kv


def attention_forward(q, k, v, scale=None, causal=False, block_mask=None, block=128):
    """Forward over a batch: q of shape (B, H, n, d); k, v of shape
    (B, H_kv, n, d) with H_kv dividing H (H_kv = H: one key/value head per
    query head).  Returns (O, LSE) as float64 arrays of shape (B, H, n, d)
    and (B, H, n)."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, n, d = q.shape
    g = _group(H, k.shape[1])
    o = np.empty((B, H, n, v.shape[-1]))
    lse = np.empty((B, H, n))
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = attention_forward_head(
                q[b, h], k[b, h // g], v[b, h // g], scale, causal, None, block_mask, block)
    return o, lse


def attention_backward(q, k, v, do, scale=None, causal=False, block_mask=None, block=128):
    """Backward over a batch (shapes as attention_forward).  Returns float64
    (dQ, dK, dV, D) with D of shape (B, H, n).  A key/value head read by
    several query heads gets the sum of the gradients through each of them
    (the loss depends on it through every head of its group)."""
    q, k, v, do = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(do)
    B, H, n, d = q.shape
    g = _group(H, k.shape[1])
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    D = np.empty((B, H, n))
    for b in range(B):
        for h in range(H):
            dq[b, h], dk_h, dv_h, D[b, h] = attention_backward_head(
                q[b, h], k[b, h // g], v[b, h // g], do[b, h], scale, causal, block_mask, block)
            dk[b, h // g] += dk_h
            dv[b, h // g] += dv_h
    return dq, dk, dv, D
