"""Seeded synthetic inputs for the five attention workloads.

This module holds no attention arithmetic: it only draws Gaussian Q, K, V and
dO from a seeded CPU generator, rounds them to the workload's dtype and
(optionally) moves them to a device.  Both the CUDA path and the float64
oracle are fed from here, so the two see bit-identical inputs.

Workloads (batch B, heads H, sequence n, head dim d):

  tiny_f32        B1  H1  n128   d64   fp32  non-causal  N(0,1)
  b4h16_n2k_d64   B4  H16 n2048  d64   bf16  non-causal  N(0,1)
  b2h16_n8k_d128  B2  H16 n8192  d128  bf16  causal      N(0,1)
  b1h8_n32k_d128  B1  H8  n32768 d128  bf16  causal      Q,K ~ N(0,4); V,dO ~ N(0,1)
  b2h8_n4k_d256   B2  H8  n4096  d256  bf16  non-causal  N(0,1)

Grouped-query workloads (H query heads sharing H_kv key/value heads; K and
V are drawn with H_kv heads):

  b2h16kv4_n8k_d128  B2 H16 H_kv 4  n8192 d128 bf16 causal  N(0,1)
  b1h32kv1_n4k_d128  B1 H32 H_kv 1  n4096 d128 bf16 causal  N(0,1)

Block-sparse workloads (a 128 x 128-block pattern shared by every head, from
make_block_mask: a local window of w blocks on each side of the diagonal,
g global blocks that attend to and are attended by every block, and r
random blocks per block row, as in Longformer and BigBird):

  b2h16_n16k_d128_sparse  B2 H16 n16384 d128 bf16 non-causal  w 2, g 1, r 2

FP8 workloads (forward only): bf16 draws that the FP8 path quantises to
e4m3 itself (per-head scales, V transposed); the outlier variant adds to each
entry of Q and K, with probability 1e-3, an extra N(0, 10^2) draw (a few
large activations, the case incoherent processing is for):

  b2h16_n8k_d128_fp8           B2 H16 n8192 d128 causal  N(0,1)
  b1h4_n4k_d128_fp8_outliers   B1 H4  n4096 d128 causal  N(0,1) + outliers on Q, K

make_signs draws the random signs of the incoherent-processing rotation.

Values are drawn in float32 and rounded to bf16 round-to-nearest-even; the
Q/K factor 2.0 of the sharp-softmax workload is a power of two, so it is
exact in either dtype.
"""

from dataclasses import dataclass, replace

import torch

__all__ = ["Workload", "WORKLOADS", "GQA_WORKLOADS", "SPARSE_WORKLOADS", "FP8_WORKLOADS",
           "workload", "make_inputs", "make_signs", "make_block_mask"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    n: int
    d: int
    dtype: str          # "bf16" or "f32"
    causal: bool
    qk_gain: float = 1.0
    seed: int = 0
    H_kv: int = 0       # key/value heads; 0 means one per query head (H)
    sparse: tuple = ()  # (window, global, random) blocks of a block mask; () = dense
    fp8: bool = False   # forward-only e4m3 workload (quantised by the FP8 path)
    outliers: tuple = ()  # (probability, std) of an extra Gaussian on Q, K entries

    @property
    def kv_heads(self):
        return self.H_kv or self.H

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def scale(self):
        return 1.0 / float(self.d) ** 0.5

    def with_shape(self, **kw):
        """A copy with some fields replaced (used for ragged/small variants)."""
        return replace(self, **kw)


WORKLOADS = [
    Workload("tiny_f32", 1, 1, 128, 64, "f32", False, 1.0, 1001),
    Workload("b4h16_n2k_d64", 4, 16, 2048, 64, "bf16", False, 1.0, 1002),
    Workload("b2h16_n8k_d128", 2, 16, 8192, 128, "bf16", True, 1.0, 1003),
    Workload("b1h8_n32k_d128", 1, 8, 32768, 128, "bf16", True, 2.0, 1004),
    Workload("b2h8_n4k_d256", 2, 8, 4096, 256, "bf16", False, 1.0, 1005),
]


GQA_WORKLOADS = [
    Workload("b2h16kv4_n8k_d128", 2, 16, 8192, 128, "bf16", True, 1.0, 1006, H_kv=4),
    Workload("b1h32kv1_n4k_d128", 1, 32, 4096, 128, "bf16", True, 1.0, 1007, H_kv=1),
]


SPARSE_WORKLOADS = [
    Workload("b2h16_n16k_d128_sparse", 2, 16, 16384, 128, "bf16", False, 1.0, 1008,
             sparse=(2, 1, 2)),
]


FP8_WORKLOADS = [
    Workload("b2h16_n8k_d128_fp8", 2, 16, 8192, 128, "bf16", True, 1.0, 1003, fp8=True),
    Workload("b1h4_n4k_d128_fp8_outliers", 1, 4, 4096, 128, "bf16", True, 1.0, 1009, fp8=True,
             outliers=(1e-3, 10.0)),
]


def workload(name):
    for w in WORKLOADS + GQA_WORKLOADS + SPARSE_WORKLOADS + FP8_WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def make_inputs(w, device="cpu", pin=False):
    """Draw q, do of shape (B, H, n, d) and k, v of shape (B, H_kv, n, d)
    for workload ``w``.

    Draw order is fixed (q, k, v, do) from ``torch.Generator().manual_seed(w.seed)``,
    then, for an outlier workload, the outlier mask and values of q and of k.
    Returns a dict of tensors in ``w.torch_dtype`` on ``device`` (pinned host
    memory if ``pin`` and device is cpu).
    """
    g = torch.Generator(device="cpu").manual_seed(int(w.seed))
    raw = {}
    for name in ("q", "k", "v", "do"):
        heads = w.kv_heads if name in ("k", "v") else w.H
        raw[name] = torch.randn((w.B, heads, w.n, w.d), generator=g, dtype=torch.float32)
    if w.outliers:
        prob, std = w.outliers
        for name in ("q", "k"):
            hit = torch.rand(raw[name].shape, generator=g) < prob
            extra = torch.randn(raw[name].shape, generator=g) * std
            raw[name] = raw[name] + hit * extra
    out = {}
    for name in ("q", "k", "v", "do"):
        x = raw[name]
        if name in ("q", "k") and w.qk_gain != 1.0:
            x.mul_(w.qk_gain)
        x = x.to(w.torch_dtype)
        if device != "cpu":
            x = x.to(device)
        elif pin:
            x = x.pin_memory()
        out[name] = x
    return out


def make_block_mask(n, window, n_global, n_random, seed, block=128):
    """A uint8 (ceil(n/block), ceil(n/block)) block pattern: block (i, j) is 1
    when |i - j| <= window, when i < n_global or j < n_global, or when j is one
    of n_random distinct blocks drawn for row i from a seeded generator."""
    nb = (n + block - 1) // block
    i = torch.arange(nb)[:, None]
    j = torch.arange(nb)[None, :]
    m = ((i - j).abs() <= window) | (i < n_global) | (j < n_global)
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    for row in range(nb):
        if n_random > 0:
            pick = torch.randperm(nb, generator=g)[:min(n_random, nb)]
            m[row, pick] = True
    return m.to(torch.uint8)


def make_signs(d, seed):
    """d random signs (+1.0 / -1.0, float32) for the incoherent-processing
    rotation, from ``torch.Generator().manual_seed(seed)``."""
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    return torch.randint(0, 2, (d,), generator=g).float() * 2.0 - 1.0
