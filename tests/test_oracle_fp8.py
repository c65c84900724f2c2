"""Pins of the FP8 oracle (oracle/fp8.py) against things other than itself:
the e4m3 encoding as torch decodes and rounds it, hand-worked ties and
limits, the orthogonality of the rotation and the invariance of the scores,
and the rounding-error bound of the per-head quantisation."""

import numpy as np
import pytest
import torch

from oracle import fp8


def test_grid_matches_torch_decoding():
    # torch.float8_e4m3fn decodes every byte: codes 0..126 are our grid
    dec = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(fp8.e4m3_values(), dec[:127])
    assert np.isnan(dec[127]) and np.array_equal(dec[128:255], -dec[:127])


def test_grid_landmarks():
    g = fp8.e4m3_values()
    assert g[0] == 0 and g[1] == 2.0 ** -9 and g[8] == 2.0 ** -6 and g[-1] == 448.0
    assert np.all(np.diff(g) > 0)
    assert g[56] == 1.0 and g[57] == 1.125            # spacing 2^-3 in [1, 2)


@pytest.mark.parametrize("x,want", [
    (1.0625, 1.0),            # tie between 1 (mantissa 0) and 1.125 (mantissa 1): even
    (1.1875, 1.25),           # tie between 1.125 (1) and 1.25 (2): even
    (2.0 ** -10, 0.0),        # tie between 0 and the smallest subnormal: 0
    (3 * 2.0 ** -10, 2.0 ** -8),   # tie between 2^-9 (code 1) and 2^-8 (code 2)
    (-1.1875, -1.25),
    (448.0, 448.0), (470.0, 448.0), (1e9, 448.0), (-1e9, -448.0),   # saturation
    (0.3, 0.3125),            # [0.25, 0.5): step 2^-5, nearest of 0.28125 / 0.3125
])
def test_round_hand_cases(x, want):
    assert fp8.round_e4m3(x) == want


def test_round_matches_torch_below_saturation():
    g = torch.Generator().manual_seed(5)
    x = torch.cat([torch.randn(200000, generator=g) * s for s in (1e-3, 0.1, 1.0, 30.0)])
    x = x[x.abs() < 448.0]
    # torch rounds float32 to e4m3 to nearest, ties to even (no saturation needed here)
    ref = x.to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(fp8.round_e4m3(x.double().numpy()), ref)
    # every midpoint between neighbours, both signs
    gv = fp8.e4m3_values()
    mids = torch.tensor((gv[:-1] + gv[1:]) / 2, dtype=torch.float32)
    mids = torch.cat([mids, -mids])
    assert np.array_equal(fp8.round_e4m3(mids.double().numpy()),
                          mids.to(torch.float8_e4m3fn).double().numpy())


def test_rotation_d2_by_hand():
    r = fp8.rotation(2, [1.0, -1.0])
    s = 1 / np.sqrt(2)
    assert np.allclose(r, [[s, s], [-s, s]], atol=0, rtol=1e-15)


@pytest.mark.parametrize("d", [2, 16, 128])
def test_rotation_orthogonal_and_scores_invariant(d):
    rng = np.random.default_rng(d)
    s = rng.choice([-1.0, 1.0], size=d)
    r = fp8.rotation(d, s)
    assert np.allclose(r @ r.T, np.eye(d), atol=1e-13)
    q, k = rng.standard_normal((7, d)), rng.standard_normal((5, d))
    assert np.allclose((q @ r) @ (k @ r).T, q @ k.T, atol=1e-12)


def test_rotation_spreads_a_one_hot_row():
    d = 128
    s = np.where(np.arange(d) % 3 == 0, -1.0, 1.0)
    r = fp8.rotation(d, s)
    for j in (0, 5, 127):
        row = np.zeros(d)
        row[j] = 10.0
        assert np.allclose(np.abs(row @ r), 10.0 / np.sqrt(d), atol=1e-13)


def test_quantize_error_bound_and_amax():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 3, 64, 32)).astype(np.float32).astype(np.float64)
    x[1, 2] = 0.0                                   # an all-zero head
    codes, descale, scaled = fp8.quantize_per_head(x)
    assert descale[1, 2] == 1.0 and np.all(codes[1, 2] == 0)
    amax = np.abs(x).max(axis=(-2, -1))
    nz = amax > 0
    assert np.allclose(descale[nz], amax[nz] / 448.0, rtol=1e-15)
    assert np.isclose(np.abs(codes).max(axis=(-2, -1))[nz], 448.0).all()
    # |code - scaled| <= half a step: 2^-4 |scaled| for normals, 2^-10 below 2^-6
    err = np.abs(codes - scaled)
    bound = np.maximum(2.0 ** -4 * np.abs(scaled), 2.0 ** -10)
    assert np.all(err <= bound * (1 + 1e-12))
    # scaled is x / descale up to the two float32 roundings of the scaling
    exact = x / descale[..., None, None]
    assert np.all(np.abs(scaled - exact) <= 2 * 2.0 ** -24 * np.abs(exact) * (1 + 1e-9))
    deq = fp8.dequantize(codes, descale)
    assert np.all(np.abs(deq - x) <= (bound + 2 * 2.0 ** -24 * np.abs(exact))
                  * descale[..., None, None] * (1 + 1e-9))


def test_quantize_decides_ties_in_float32():
    # bf16 inputs with amax = 3.5 make 448 / amax = 128 exact: x * 128 lands on
    # e4m3 midpoints and ties go to the even code
    x = np.zeros((1, 4, 4))
    x[0, 0, 0] = 3.5
    x[0, 1, 0] = 1.0625 / 128        # 1.0625: midpoint of 1 and 1.125 -> 1
    x[0, 2, 0] = 1.1875 / 128        # midpoint of 1.125 and 1.25 -> 1.25
    codes, descale, scaled = fp8.quantize_per_head(x)
    assert descale[0] == 3.5 / 448 and scaled[0, 0, 0] == 448.0
    assert codes[0, 1, 0] == 1.0 and codes[0, 2, 0] == 1.25
    # amax = 3.0: 448 / 3 is not exact; the float32 reciprocal decides
    x[0, 0, 0] = 3.0
    inv = np.float32(448.0) / np.float32(3.0)
    codes, _, scaled = fp8.quantize_per_head(x)
    assert scaled[0, 1, 0] == float(np.float32(1.0625 / 128) * inv)


def test_incoherent_processing_shrinks_amax_of_outlier_rows():
    # a head whose rows each carry one large entry: after the rotation the
    # large entry is spread, so amax (and the rounding step) drops by ~sqrt(d)
    rng = np.random.default_rng(11)
    d = 128
    x = rng.standard_normal((1, 256, d)) * 0.1
    x[0, np.arange(256), rng.integers(0, d, 256)] = 50.0
    s = rng.choice([-1.0, 1.0], size=d)
    _, ds_plain, _ = fp8.quantize_per_head(x)
    _, ds_rot, _ = fp8.quantize_per_head(x, s)
    assert ds_rot[0] < ds_plain[0] / 4
