"""FP8 path through the C ABI against the float64 oracle.

* attn_quantize_fp8: e4m3 codes and per-head descales against oracle.fp8,
  plain, rotated (incoherent processing) and transposed, on ragged and
  full-size heads.  Without the rotation both sides round the same float32
  product x * fl32(448 / amax), so every code must be equal.  With it the
  kernel's fp32 butterflies and the oracle's float64 product differ by
  rounding: a code must equal the oracle's unless the value lies within
  that rounding error of a midpoint, and then be one of the two neighbours.
* attn_fwd_fp8 on the oracle's codes: against the exact attention of the
  values those codes stand for.  The only rounding that is not at fp32 level
  is the e4m3 rounding of P, which puts the RMS of O - O_ref near 0.027 of
  the RMS of O (see attn_fwd_fp8 in include/attn.h): RMS ratio <= 0.035,
  max|O - O_ref| <= 0.08 max|O_ref|, LSE to 1e-5.
* the two chained on device against the oracle chained, and incoherent
  processing against plain quantisation on a workload with outliers, both
  measured against attention of the unquantised bf16 inputs.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from io_aware_exact_05_gb300.inputs import Workload, make_inputs, make_signs, workload
from parity_util import relerr, to64

pytestmark = pytest.mark.gpu

RMS_O, MAX_O, TOL_LSE = 0.035, 0.08, 1e-5
U = 2.0 ** -24     # fp32 unit roundoff


def _rms_ratio(got, ref):
    g, r = to64(got), to64(ref)
    return float(np.sqrt(((g - r) ** 2).mean() / (r ** 2).mean()))


def _code_window(x, signs):
    """Oracle codes, descales and the lowest / highest code the kernel may
    produce given its fp32 arithmetic (x float64 (..., n, 128))."""
    codes, descale, scaled = fp8.quantize_per_head(x, signs)
    if signs is None:
        win = np.zeros_like(scaled)          # the same float32 operations
    else:
        # seven butterfly stages: |error| <= 8 U sum_i |x_i| per row
        # (unnormalised), the amax inherits it, and each side rounds the
        # reciprocal and the product (3 U each)
        l1 = np.abs(x).sum(axis=-1, keepdims=True)
        amax_u = descale * fp8.E4M3_MAX * np.sqrt(x.shape[-1])
        inv = (fp8.E4M3_MAX / amax_u)[..., None, None]
        rel_amax = (8 * U * l1.max(axis=(-2, -1)) / amax_u)[..., None, None]
        win = 8 * U * l1 * inv + np.abs(scaled) * (6 * U + rel_amax)
    return codes, descale, fp8.round_e4m3(scaled - win), fp8.round_e4m3(scaled + win)


def _check_codes(got8, lo, hi, codes):
    g = got8.double().cpu().numpy()
    assert np.all((g >= lo) & (g <= hi)), "code outside the rounding window"
    assert np.array_equal(g[lo == hi], codes[lo == hi])
    return float((g != codes).mean())


def _quantise(x, transpose, signs, dev):
    from io_aware_exact_05_gb300 import attn

    s = None if signs is None else signs.to(dev)
    x8, ds = attn.quantize_fp8(x.to(dev), transpose=transpose, signs=s)
    assert attn.attn_status() == 0
    return x8, ds


@pytest.mark.parametrize("n", [200, 1024])
@pytest.mark.parametrize("rotate", [False, True])
def test_quantize_rows(cuda_dev, n, rotate):
    w = Workload("q8", 1, 3, n, 128, "bf16", False, 1.0, 1700 + n)
    x = make_inputs(w)["q"]
    x[0, 2] = 0                                  # a zero head: descale 1, codes 0
    signs = make_signs(128, 5) if rotate else None
    x8, ds = _quantise(x, False, signs, cuda_dev)
    codes, descale, lo, hi = _code_window(x.double().numpy(),
                                          None if signs is None else signs.double().numpy())
    frac = _check_codes(x8, lo, hi, codes)
    assert frac < 1e-3, frac
    assert np.allclose(ds.double().cpu().numpy(), descale, rtol=4e-6, atol=0)
    assert float(ds[0, 2]) == 1.0 and torch.all(x8[0, 2].float() == 0)


@pytest.mark.parametrize("n", [208, 1024])
def test_quantize_transposed(cuda_dev, n):
    w = Workload("v8", 2, 2, n, 128, "bf16", False, 1.0, 1800 + n)
    x = make_inputs(w)["v"]
    x8, ds = _quantise(x, True, None, cuda_dev)
    assert x8.shape == (2, 2, 128, n)
    codes, descale, lo, hi = _code_window(x.double().numpy(), None)
    t = lambda a: np.swapaxes(a, -1, -2)   # noqa: E731
    _check_codes(x8, t(lo), t(hi), t(codes))
    assert np.allclose(ds.double().cpu().numpy(), descale, rtol=4e-6, atol=0)


@pytest.mark.parametrize("rotate", [False, True])
def test_quantize_full_size(cuda_dev, rotate):
    w = workload("b2h16_n8k_d128_fp8")
    x = make_inputs(w)
    signs = make_signs(128, 9) if rotate else None
    s64 = None if signs is None else signs.double().numpy()
    for name, tr in (("q", False), ("k", False), ("v", not rotate)):
        x8, ds = _quantise(x[name], tr, None if name == "v" else signs, cuda_dev)
        codes, descale, lo, hi = _code_window(x[name].double().numpy(),
                                              None if name == "v" else s64)
        if tr:
            codes, lo, hi = (np.swapaxes(a, -1, -2) for a in (codes, lo, hi))
        frac = _check_codes(x8, lo, hi, codes)
        assert frac < 1e-3, (name, frac)
        assert np.allclose(ds.double().cpu().numpy(), descale, rtol=4e-6, atol=0)


def _oracle_operands(x, signs=None):
    """e4m3 codes from the oracle, as the kernel takes them, and the float64
    values they stand for (with the fp32 descales actually passed)."""
    out = {}
    for name in ("q", "k", "v"):
        s = signs if name != "v" else None
        codes, descale, _ = fp8.quantize_per_head(x[name].double().numpy(), s)
        d32 = descale.astype(np.float32)
        c = torch.from_numpy(codes)
        if name == "v":
            c = c.transpose(-1, -2).contiguous()
        out[name + "8"] = c.to(torch.float8_e4m3fn)
        out["ds_" + name] = torch.from_numpy(d32)
        out[name] = fp8.dequantize(codes, d32.astype(np.float64))
    return out


def _forward(ops, causal, dev):
    from io_aware_exact_05_gb300 import attn

    o, lse = attn.forward_fp8(ops["q8"].to(dev), ops["k8"].to(dev), ops["v8"].to(dev),
                              (ops["ds_q"].to(dev), ops["ds_k"].to(dev), ops["ds_v"].to(dev)),
                              causal=causal)
    assert attn.attn_status() == 0
    return o, lse


def _check_forward(o, lse, ro, rl):
    er, em, el = _rms_ratio(o, ro), relerr(o, ro), relerr(lse, rl)
    assert er <= RMS_O and em <= MAX_O and el <= TOL_LSE, (er, em, el)
    return er, em, el


@pytest.mark.parametrize("n", [128, 400, 1024])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_small(cuda_dev, n, causal):
    w = Workload("fp8", 1, 2, n, 128, "bf16", causal, 1.0, 1600 + n)
    ops = _oracle_operands(make_inputs(w))
    o, lse = _forward(ops, causal, cuda_dev)
    ro, rl = oracle.attention_forward(ops["q"], ops["k"], ops["v"], w.scale, causal)
    _check_forward(o, lse, ro, rl)


def test_forward_full_size(cuda_dev):
    w = workload("b2h16_n8k_d128_fp8")
    ops = _oracle_operands(make_inputs(w))
    o, lse = _forward(ops, w.causal, cuda_dev)
    for hh in (0, w.B * w.H - 1):
        b, h = divmod(hh, w.H)
        ro, rl = oracle.attention_forward_head(ops["q"][b, h], ops["k"][b, h], ops["v"][b, h],
                                               w.scale, True)
        _check_forward(o[b, h].cpu(), lse[b, h].cpu(), ro, rl)


def test_descale_v_scales_the_result(cuda_dev):
    # the same codes with descale_v doubled: O doubles exactly, LSE unchanged
    w = Workload("fp8d", 1, 2, 256, 128, "bf16", False, 1.0, 1710)
    ops = _oracle_operands(make_inputs(w))
    o1, l1 = _forward(ops, False, cuda_dev)
    ops["ds_v"] = ops["ds_v"] * 2
    o2, l2 = _forward(ops, False, cuda_dev)
    assert torch.equal(o2.float(), 2 * o1.float()) and torch.equal(l1, l2)


def test_chained_on_device(cuda_dev):
    # device quantiser -> FP8 forward, against the oracle's quantiser -> exact
    # attention; measured against attention of the unquantised inputs, the
    # two differ only by the e4m3 rounding of P (and rare code ties)
    from io_aware_exact_05_gb300 import attn

    w = Workload("chain", 1, 2, 1024, 128, "bf16", True, 1.0, 1720)
    x = make_inputs(w)
    q8, dq = _quantise(x["q"], False, None, cuda_dev)
    k8, dk = _quantise(x["k"], False, None, cuda_dev)
    v8, dv = _quantise(x["v"], True, None, cuda_dev)
    o, lse = attn.forward_fp8(q8, k8, v8, (dq, dk, dv), causal=True)
    assert attn.attn_status() == 0
    ops = _oracle_operands(x)
    ro, rl = oracle.attention_forward(ops["q"], ops["k"], ops["v"], w.scale, True)
    _check_forward(o, lse, ro, rl)


def test_incoherent_processing_lowers_error_with_outliers(cuda_dev):
    # Q and K with rare large entries: quantising after the Hadamard rotation
    # gives a smaller error against attention of the unquantised inputs
    from io_aware_exact_05_gb300 import attn

    w = workload("b1h4_n4k_d128_fp8_outliers")
    x = make_inputs(w)
    signs = make_signs(128, 77)
    ref, _ = oracle.attention_forward(*(x[t].double().numpy() for t in "qkv"), w.scale,
                                      w.causal)
    errs = {}
    for rotate in (False, True):
        s = signs if rotate else None
        q8, dq = _quantise(x["q"], False, s, cuda_dev)
        k8, dk = _quantise(x["k"], False, s, cuda_dev)
        v8, dv = _quantise(x["v"], True, None, cuda_dev)
        o, _ = attn.forward_fp8(q8, k8, v8, (dq, dk, dv), causal=w.causal)
        assert attn.attn_status() == 0
        errs[rotate] = _rms_ratio(o, ref)
    assert errs[True] < 0.75 * errs[False], errs


def test_unsupported_shapes(cuda_dev):
    from io_aware_exact_05_gb300 import attn

    z = lambda *s: torch.zeros(*s, dtype=torch.float8_e4m3fn, device=cuda_dev)   # noqa: E731
    with pytest.raises(attn.AttnError) as e:
        attn.forward_fp8(z(1, 1, 64, 64), z(1, 1, 64, 64), z(1, 1, 64, 64))
    assert e.value.code == 2                 # d = 64
    with pytest.raises(attn.AttnError) as e:
        attn.forward_fp8(z(1, 1, 100, 128), z(1, 1, 100, 128), z(1, 1, 128, 100))
    assert e.value.code == 2                 # n not a multiple of 16
    xb = torch.zeros(1, 1, 100, 128, dtype=torch.bfloat16, device=cuda_dev)
    with pytest.raises(attn.AttnError) as e:
        attn.quantize_fp8(xb, transpose=True)
    assert e.value.code == 2                 # transposed output needs n % 16 == 0
    with pytest.raises(attn.AttnError) as e:
        attn.quantize_fp8(xb[..., :64].contiguous())
    assert e.value.code == 2                 # d = 64
