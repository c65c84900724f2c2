"""Float64 CPU oracle for the FP8 operand encoding of the FP8 attention
forward: e4m3 rounding, per-head scaling, and the Hadamard rotation of
incoherent processing.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
module.  The library never calls it and shares no code with it.

The pages list two FlashAttention-3 techniques without defining either
("Flash Attention: Revolutionizing Transformer Efficiency", section
FlashAttention-3, items 2 and 3; "Chapter 3.1 -- The cost of attention",
section 6, the FlashAttention-3 paragraph): computing parts of attention in
FP8, and "incoherent processing", which lowers the quantisation error of
low-precision formats.  Readings taken here:

  * FP8 is e4m3 with the encoding of torch.float8_e4m3fn: 1 sign bit, 4
    exponent bits with bias 7, 3 mantissa bits, no infinities; the largest
    finite value is 448, normals start at 2^-6, subnormals are multiples of
    2^-9.  Rounding is to the nearest value, ties to the even code (even
    mantissa); magnitudes above 448 saturate to 448.
  * Scaling is per head: descale_h = amax_h / 448 over the head's n x d
    values, and the code stands for code * descale_h.  The value rounded is
    x * (448 / amax_h) formed in float32 (the reciprocal rounded to float32,
    then the product rounded to float32): where a floating-point value
    decides an integer code, it is decided in the device's precision, and
    with bf16 inputs and a bf16 amax exact rounding ties are common.  A head
    of zeros gets descale 1 and codes 0.
  * Incoherent processing multiplies every row of Q and of K by the same
    orthogonal matrix R = diag(s) H_d / sqrt(d) (H_d the Sylvester Hadamard
    matrix, s a vector of random signs) before quantising.  Since
    R R^T = I, (Q R)(K R)^T = Q K^T: the scores are unchanged, but a few
    large entries of a row are spread over all d entries, so the head's
    amax and with it the rounding step shrink.  V is not rotated.

Every function is pinned by tests/test_oracle_fp8.py.
"""

import numpy as np
from scipy.linalg import hadamard

E4M3_MAX = 448.0

__all__ = ["E4M3_MAX", "e4m3_values", "round_e4m3", "rotation", "quantize_per_head",
           "dequantize"]


def e4m3_values():
    """The 127 non-negative finite e4m3 values, indexed by their code
    (0x00 .. 0x7E; 0x7F is NaN): exponent field e = code >> 3, mantissa
    m = code & 7; e = 0 gives m * 2^-9, otherwise (1 + m / 8) * 2^(e - 7)."""
    out = np.empty(127)
    for code in range(127):
        e, m = code >> 3, code & 7
        out[code] = m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_GRID = e4m3_values()


def round_e4m3(x):
    """Round float64 values to e4m3 values: nearest, ties to the even code,
    saturating at +-448.  Returns float64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_GRID, a, side="left"), 0, len(_GRID) - 1)  # first >= a
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - _GRID[lo], _GRID[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(_GRID[hi] == a, hi, code)          # exact values
    return np.copysign(_GRID[code], x)


def rotation(d, signs):
    """R = diag(signs) H_d / sqrt(d), the rotation applied to rows (x -> x R)."""
    s = np.asarray(signs, dtype=np.float64)
    assert s.shape == (d,) and np.all(np.abs(s) == 1.0)
    return (s[:, None] * hadamard(d).astype(np.float64)) / np.sqrt(d)


def quantize_per_head(x, signs=None):
    """Per-head e4m3 quantisation of x (..., n, d), optionally after the
    rotation of incoherent processing.

    Returns (codes, descale, scaled): codes are the e4m3 values (float64),
    descale has x's leading shape, and scaled = float32((rotated) x) *
    float32(448 / amax) is the value that was rounded."""
    x = np.asarray(x, dtype=np.float64)
    if signs is not None:
        x = x @ rotation(x.shape[-1], signs)
    amax = np.abs(x).max(axis=(-2, -1))
    descale = np.where(amax > 0, amax / E4M3_MAX, 1.0)
    amax32 = np.where(amax > 0, amax, 1.0).astype(np.float32)
    inv = np.where(amax > 0, np.float32(E4M3_MAX) / amax32, np.float32(1.0)).astype(np.float32)
    scaled = (x.astype(np.float32) * inv[..., None, None]).astype(np.float64)
    return round_e4m3(scaled), descale, scaled


def dequantize(codes, descale):
    """The real values the codes stand for: code * descale (per head)."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(descale)[..., None, None]
