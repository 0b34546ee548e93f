"""Pins of the FP8 (e4m3) oracle against things other than itself (no GPU).

* The rounding is checked against the format's own definition: every finite
  code decoded from its bit fields is a fixed point, midpoints between
  neighbours go to the even code, magnitudes past 448 saturate; and against
  a library routine, torch's CPU conversion to float8_e4m3fn.
* The quantised attention equals the plain fp64 oracle when the rotated
  operands already sit on the scaled e4m3 grid, and its scales are per head:
  rescaling one head's V rescales that head's output and leaves the others
  bit for bit.
"""
import math

import numpy as np
import pytest

from oracle import fp8, ref

RNG = np.random.default_rng(77)


def _finite_codes():
    codes = np.arange(256)
    vals = fp8.e4m3_decode(codes)
    return codes[np.isfinite(vals)], vals[np.isfinite(vals)]


def test_decode_matches_the_format_table():
    codes, vals = _finite_codes()
    assert len(codes) == 254                      # 0x7F and 0xFF are NaN
    pos = np.unique(vals[vals > 0])
    assert len(pos) == 126
    assert pos.max() == 448.0 and pos.min() == 2.0 ** -9
    assert fp8.e4m3_decode(0x08) == 2.0 ** -6     # smallest normal
    assert fp8.e4m3_decode(0x07) == 7 * 2.0 ** -9  # largest subnormal
    assert fp8.e4m3_decode(0x38) == 1.0           # exponent field 7 = bias
    assert fp8.e4m3_decode(0xB8) == -1.0


def test_every_finite_value_is_a_fixed_point():
    _, vals = _finite_codes()
    np.testing.assert_array_equal(fp8.e4m3_round(vals), vals)


def test_midpoints_round_to_the_even_code():
    _, vals = _finite_codes()
    pos = np.unique(vals[vals >= 0])              # 0, 2^-9, ..., 448
    mids = (pos[:-1] + pos[1:]) / 2
    got = fp8.e4m3_round(mids)
    for lo, hi, g in zip(pos[:-1], pos[1:], got):
        # the code's last bit is the mantissa's; the even neighbour wins
        lo_code = int(np.where(fp8.e4m3_decode(np.arange(128)) == lo)[0][0])
        want = lo if lo_code % 2 == 0 else hi
        assert g == want, (lo, hi, g)
    # just off the midpoints the nearer neighbour wins
    np.testing.assert_array_equal(fp8.e4m3_round(np.nextafter(mids, 0)), pos[:-1])
    np.testing.assert_array_equal(fp8.e4m3_round(np.nextafter(mids, np.inf)), pos[1:])


def test_saturation_and_sign():
    np.testing.assert_array_equal(fp8.e4m3_round([449.0, 463.9, 464.0, 500.0, 1e9]), 448.0)
    np.testing.assert_array_equal(fp8.e4m3_round([-449.0, -1e9]), -448.0)
    assert fp8.e4m3_round(0.0) == 0.0
    assert fp8.e4m3_round(2.0 ** -11) == 0.0      # below half the smallest subnormal
    x = RNG.standard_normal(1000) * 30
    np.testing.assert_array_equal(fp8.e4m3_round(-x), -fp8.e4m3_round(x))


def test_relative_error_bound_in_the_normal_range():
    x = np.exp(RNG.uniform(math.log(2.0 ** -6), math.log(440.0), 100000))
    r = fp8.e4m3_round(x)
    assert np.max(np.abs(r - x) / x) <= 2.0 ** -4


def test_matches_torch_float8_conversion():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch has no float8_e4m3fn")
    x = np.concatenate([RNG.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 40.0)])
    x = x[np.abs(x) <= 440.0]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(fp8.e4m3_round(x), lib)


def test_quantise_scale_is_amax_over_448():
    x = RNG.standard_normal((50, 8))
    x8, s = fp8.quantise(x)
    assert s == np.abs(x).max() / 448.0
    assert np.abs(x8).max() == 448.0
    z8, zs = fp8.quantise(np.zeros((4, 4)))
    assert zs == 1.0 and np.all(z8 == 0)


def _on_grid_inputs(grid, H, d, rng):
    """Pre-RoPE q, k, v whose rotated values are c * G with G on the e4m3 grid
    and max|G| = 448 (so quantisation is exact)."""
    L = grid[0] * grid[1] * grid[2]
    ang = ref.rope_angles(*grid, d)
    _, vals = _finite_codes()
    out = []
    for rotate in (True, True, False):
        x = np.zeros((1, L, H, d))
        for h in range(H):
            g = rng.choice(vals[np.abs(vals) <= 64], size=(L, d))
            g[rng.integers(L), rng.integers(d)] = 448.0
            c = 2.0 ** rng.integers(-12, -4) * rng.uniform(1, 2)
            x[0, :, h] = ref.rope_rotate(c * g, ang, inverse=True) if rotate else c * g
        out.append(x)
    return out


def test_exact_when_operands_are_on_the_grid():
    grid, H, d = (2, 3, 4), 2, 128
    q, k, v = _on_grid_inputs(grid, H, d, np.random.default_rng(5))
    o8, lse8 = fp8.fp8_self_attention_fwd(q, k, v, grid)
    o, lse = ref.self_attention_fwd(q, k, v, grid)
    np.testing.assert_allclose(o8, o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse8, lse, rtol=1e-12, atol=1e-12)


def test_scales_are_per_head():
    grid, H, d = (2, 2, 3), 3, 128
    L = 12
    q, k, v = (RNG.standard_normal((1, L, H, d)) for _ in range(3))
    o, lse = fp8.fp8_self_attention_fwd(q, k, v, grid)
    v2 = v.copy()
    v2[0, :, 1] *= 4.0                            # a power of two: the scaled head is exactly 4x
    o2, lse2 = fp8.fp8_self_attention_fwd(q, k, v2, grid)
    np.testing.assert_array_equal(o2[0, :, 0], o[0, :, 0])
    np.testing.assert_array_equal(o2[0, :, 2], o[0, :, 2])
    np.testing.assert_array_equal(o2[0, :, 1], 4.0 * o[0, :, 1])
    v3 = v.copy()
    v3[0, :, 1] *= 3.0
    o3, _ = fp8.fp8_self_attention_fwd(q, k, v3, grid)
    np.testing.assert_allclose(o3[0, :, 1], 3.0 * o[0, :, 1], rtol=1e-12)
    np.testing.assert_array_equal(lse2, lse)


def test_quantisation_noise_has_the_e4m3_size():
    """Against the plain oracle the quantised attention differs by the noise
    of 3-bit mantissas: neither zero nor larger than a few times 2^-4."""
    grid, H, d = (2, 4, 4), 2, 128
    q, k, v = (RNG.standard_normal((1, 32, H, d)) for _ in range(3))
    o8, _ = fp8.fp8_self_attention_fwd(q, k, v, grid)
    o, _ = ref.self_attention_fwd(q, k, v, grid)
    rel = np.linalg.norm(o8 - o) / np.linalg.norm(o)
    assert 0.005 < rel < 0.15, rel
