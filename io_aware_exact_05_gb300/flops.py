"""Algorithmic work and traffic counts used for reporting throughput.

FLOPs follow the usual convention for exact attention: the forward pass is
two n x n x d contractions (QK^T and PV), 4*n^2*d per head; the backward pass
is five (QK^T recomputed, dP = dO V^T, dV = P^T dO, dQ = dS K, dK = dS^T Q),
10*n^2*d per head.  A causal mask halves both.  The n^2 growth is the
quadratic cost described in "Chapter 3.1 -- The cost of attention",
section 2.
"""

__all__ = ["attention_flops", "score_entries", "algorithmic_bytes", "kept_entries",
           "sparse_attention_flops"]


def score_entries(n):
    """Entries of the n x n score matrix QK^T."""
    return n * n


def attention_flops(B, H, n, d, causal):
    """FLOPs per call: {'fwd': ..., 'bwd': ..., 'total': ...}."""
    base = B * H * n * n * d
    fwd, bwd = 4 * base, 10 * base
    if causal:
        fwd //= 2
        bwd //= 2
    return {"fwd": fwd, "bwd": bwd, "total": fwd + bwd}


def algorithmic_bytes(B, H, n, d, elt):
    """Compulsory HBM bytes per call for the forward (read Q,K,V; write O and
    the fp32 LSE), the D preprocess (read O, dO; write fp32 D) and the fused
    backward (read Q,K,V,dO, LSE, D; write dQ, dK, dV)."""
    t = B * H * n * d * elt
    r = B * H * n * 4
    return {"fwd": 4 * t + r, "pre": 2 * t + r, "bwd": 7 * t + 2 * r}


def kept_entries(block_mask, n, causal, block=128):
    """Score entries a block pattern keeps (per head): the entries of every
    kept block clipped to n x n, without j > i when causal."""
    import numpy as np

    m = np.asarray(block_mask, dtype=bool)
    nb = m.shape[0]
    sizes = np.minimum(block, n - np.arange(nb) * block)       # rows (or keys) per block
    total = 0
    for bi in range(nb):
        for bj in np.nonzero(m[bi])[0]:
            if not causal or bj < bi:
                total += int(sizes[bi]) * int(sizes[bj])
            elif bj == bi:                                     # lower triangle of a diagonal block
                s = int(sizes[bi])
                total += s * (s + 1) // 2
    return total


def sparse_attention_flops(B, H, d, kept):
    """FLOPs per call of block-sparse attention: 4 d (fwd) and 10 d (bwd) per
    kept score entry and head (the dense counts with n^2 -> kept entries)."""
    fwd, bwd = 4 * B * H * d * kept, 10 * B * H * d * kept
    return {"fwd": fwd, "bwd": bwd, "total": fwd + bwd}
