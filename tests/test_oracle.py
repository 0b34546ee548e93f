"""Pins of the fp64 oracle against things other than itself (no GPU).

Each check is chosen so that a plausible slip in the oracle (a dropped term,
a wrong sign, a transposed operand, a band offset off by one) fails it:
brute-force loops written independently, closed forms, library routines
(scipy softmax / logsumexp, numpy complex multiplication), invariants of
rotations and of softmax, and central finite differences.
"""
import cmath
import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from oracle import ref

RNG = np.random.default_rng(1234)


def _rand(*shape):
    return RNG.standard_normal(shape)


# ---------------------------------------------------------------------------
# Brute force: an independent triple loop in pure Python on an 8-token grid


def _brute_rope(vec, t, h, w, d, theta):
    """Rotate one vector by walking its dims and deciding each pair's band."""
    w_hw = 2 * (d // 6)
    w_t = d - 2 * w_hw
    out = list(vec)
    for p in range(d // 2):
        dim = 2 * p
        if dim < w_t:
            pos, j, width = t, p, w_t
        elif dim < w_t + w_hw:
            pos, j, width = h, p - w_t // 2, w_hw
        else:
            pos, j, width = w, p - (w_t + w_hw) // 2, w_hw
        ang = pos * math.pow(theta, -2.0 * j / width)
        z = complex(vec[dim], vec[dim + 1]) * cmath.exp(1j * ang)
        out[dim], out[dim + 1] = z.real, z.imag
    return out


def _brute_attention(q, k, v, grid, theta, scale):
    F, Hp, Wp = grid
    B, L, H, d = q.shape
    coords = [(t, h, w) for t in range(F) for h in range(Hp) for w in range(Wp)]
    o = np.zeros_like(q)
    lse = np.zeros((B, H, L))
    for b in range(B):
        for hd in range(H):
            qr = [_brute_rope(q[b, i, hd], *coords[i], d, theta) for i in range(L)]
            kr = [_brute_rope(k[b, j, hd], *coords[j], d, theta) for j in range(L)]
            for i in range(L):
                logits = [scale * sum(qr[i][x] * kr[j][x] for x in range(d)) for j in range(L)]
                top = max(logits)
                ws = [math.exp(s - top) for s in logits]
                tot = sum(ws)
                for x in range(d):
                    o[b, i, hd, x] = sum(ws[j] * v[b, j, hd, x] for j in range(L)) / tot
                lse[b, hd, i] = top + math.log(tot)
    return o, lse


@pytest.mark.parametrize("d", [12, 128])
def test_bruteforce_8_tokens(d):
    grid = (2, 2, 2)
    q, k, v = _rand(1, 8, 2, d), _rand(1, 8, 2, d), _rand(1, 8, 2, d)
    scale = 1.0 / math.sqrt(d)
    o, lse = ref.self_attention_fwd(q, k, v, grid, 10000.0, scale)
    ob, lseb = _brute_attention(q, k, v, grid, 10000.0, scale)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lseb, rtol=0, atol=1e-12)


def test_bruteforce_asymmetric_grid():
    # F, Hp, Wp all different so a swapped axis cannot pass.
    grid = (3, 2, 4)
    L, d = 24, 12
    q, k, v = _rand(1, L, 1, d), _rand(1, L, 1, d), _rand(1, L, 1, d)
    o, lse = ref.self_attention_fwd(q, k, v, grid, 100.0, 0.3)
    ob, lseb = _brute_attention(q, k, v, grid, 100.0, 0.3)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lseb, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Closed forms


def test_zero_queries_give_mean_of_values():
    grid = (3, 4, 5)
    L, H, d = 60, 2, 128
    q = np.zeros((1, L, H, d))
    k, v = _rand(1, L, H, d), _rand(1, L, H, d)
    o, lse = ref.self_attention_fwd(q, k, v, grid)
    mean_v = v.mean(axis=1, keepdims=True)
    np.testing.assert_allclose(o, np.broadcast_to(mean_v, o.shape), atol=1e-13)
    np.testing.assert_allclose(lse, math.log(L), atol=1e-13)


def test_zero_queries_cross_attention_mean_of_valid_values():
    B, Lq, Lk, H, d = 2, 5, 64, 2, 128
    q = np.zeros((B, Lq, H, d))
    k, v = _rand(B, Lk, H, d), _rand(B, Lk, H, d)
    lens = np.array([17, 64])
    o, lse = ref.cross_attention_fwd(q, k, v, lens)
    for b in range(B):
        mean_v = v[b, :lens[b]].mean(axis=0)
        np.testing.assert_allclose(o[b], np.broadcast_to(mean_v, o[b].shape), atol=1e-13)
        np.testing.assert_allclose(lse[b], math.log(lens[b]), atol=1e-13)


def test_one_hot_dominant_logit_returns_that_value_row():
    grid = (2, 4, 4)
    L, d = 32, 128
    q, k, v = _rand(1, L, 1, d), _rand(1, L, 1, d), _rand(1, L, 1, d)
    i0 = 13
    u = _rand(d)
    u /= np.linalg.norm(u)
    q[0, i0, 0] = 60.0 * u
    k[0, i0, 0] = 60.0 * u          # same token => same rotation => logit scale*|q|^2
    o, lse = ref.self_attention_fwd(q, k, v, grid)
    np.testing.assert_allclose(o[0, i0, 0], v[0, i0, 0], atol=1e-12)
    assert abs(lse[0, 0, i0] - 3600.0 / math.sqrt(d)) < 1e-9


# ---------------------------------------------------------------------------
# 3D RoPE


def test_rope_is_complex_multiplication():
    grid = (3, 5, 7)
    L, d = 105, 128
    x = _rand(L, d)
    ang = ref.rope_angles(*grid, d)
    got = ref.rope_rotate(x, ang)
    z = (x[:, 0::2] + 1j * x[:, 1::2]) * np.exp(1j * ang)
    np.testing.assert_allclose(got[:, 0::2], z.real, atol=1e-13)
    np.testing.assert_allclose(got[:, 1::2], z.imag, atol=1e-13)


def test_rope_bands_touch_only_their_dims():
    d = 128
    grid = (4, 4, 4)
    ang = ref.rope_angles(*grid, d)
    t, h, w = ref.token_coords(*grid)
    x = _rand(64, d)
    y = ref.rope_rotate(x, ang)
    only_t = np.where((t == 3) & (h == 0) & (w == 0))[0][0]
    only_h = np.where((t == 0) & (h == 3) & (w == 0))[0][0]
    only_w = np.where((t == 0) & (h == 0) & (w == 3))[0][0]
    np.testing.assert_array_equal(y[only_t, 44:], x[only_t, 44:])
    assert np.all(y[only_t, :44] != x[only_t, :44])
    np.testing.assert_array_equal(y[only_h, :44], x[only_h, :44])
    np.testing.assert_array_equal(y[only_h, 86:], x[only_h, 86:])
    assert np.all(y[only_h, 44:86] != x[only_h, 44:86])
    np.testing.assert_array_equal(y[only_w, :86], x[only_w, :86])
    assert np.all(y[only_w, 86:] != x[only_w, 86:])
    np.testing.assert_array_equal(y[0], x[0])  # token (0,0,0) is not rotated


def test_rope_frequency_closed_values():
    d, theta = 128, 10000.0
    # Token (1,1,1) of a 2x2x2 grid is token 7: its angles are the frequencies.
    ang = ref.rope_angles(2, 2, 2, d, theta)[7]
    assert ang.shape == (64,)
    assert ang[0] == 1.0 and ang[22] == 1.0 and ang[43] == 1.0      # j = 0 of t, h, w
    assert abs(ang[11] - 0.01) < 1e-15                             # t band: 1e4^(-22/44)
    assert abs(ang[22 + 7] - 10000.0 ** (-1.0 / 3.0)) < 1e-15       # h band: 1e4^(-14/42)
    assert abs(ang[43 + 7] - 10000.0 ** (-1.0 / 3.0)) < 1e-15       # w band
    assert abs(ang[21] - 10000.0 ** (-42.0 / 44.0)) < 1e-18         # last t pair
    # geometric within each band
    for lo, hi, width in ((0, 22, 44), (22, 43, 42), (43, 64, 42)):
        r = ang[lo + 1:hi] / ang[lo:hi - 1]
        np.testing.assert_allclose(r, theta ** (-2.0 / width), rtol=1e-13)


def test_rope_depends_only_on_relative_offset():
    d = 128
    grid = (6, 7, 8)
    ang = ref.rope_angles(*grid, d)
    t, h, w = ref.token_coords(*grid)
    idx = {(a, b, c): i for i, (a, b, c) in enumerate(zip(t, h, w))}
    for _ in range(20):
        q, k = _rand(d), _rand(d)
        p = RNG.integers(0, 3, 3)
        pp = RNG.integers(0, 3, 3)
        delta = RNG.integers(0, 3, 3)
        i1, j1 = idx[tuple(p)], idx[tuple(pp)]
        i2, j2 = idx[tuple(p + delta)], idx[tuple(pp + delta)]
        a = ref.rope_rotate(q[None], ang[[i1]])[0] @ ref.rope_rotate(k[None], ang[[j1]])[0]
        b = ref.rope_rotate(q[None], ang[[i2]])[0] @ ref.rope_rotate(k[None], ang[[j2]])[0]
        assert abs(a - b) < 1e-12


def test_rope_orthogonal_and_inverse():
    grid = (3, 4, 5)
    ang = ref.rope_angles(*grid, 128)
    x = _rand(60, 128)
    y = ref.rope_rotate(x, ang)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)
    np.testing.assert_allclose(ref.rope_rotate(y, ang, inverse=True), x, atol=1e-13)


def test_token_count_and_band_split():
    assert ref.rope_bands(128) == ((0, 44), (44, 42), (86, 42))
    t, h, w = ref.token_coords(21, 30, 52)
    assert t.size == 32760 and t[-1] == 20 and h[-1] == 29 and w[-1] == 51
    assert (t[53], h[53], w[53]) == (0, 1, 1)


# ---------------------------------------------------------------------------
# Softmax core against library routines


def test_core_matches_scipy():
    q, k, v = _rand(37, 128), _rand(300, 128), _rand(300, 128)
    scale = 0.0884
    o, lse = ref.softmax_attention(q, k, v, scale)
    s = scale * q @ k.T
    np.testing.assert_allclose(o, softmax(s, axis=1) @ v, atol=1e-13)
    np.testing.assert_allclose(lse, logsumexp(s, axis=1), atol=1e-12)


def test_self_attention_is_core_on_rotated_inputs():
    grid = (2, 3, 4)
    q, k, v = _rand(2, 24, 3, 128), _rand(2, 24, 3, 128), _rand(2, 24, 3, 128)
    o, lse = ref.self_attention_fwd(q, k, v, grid)
    ang = ref.rope_angles(*grid, 128)
    for b in range(2):
        for h in range(3):
            qr = (q[b, :, h, 0::2] + 1j * q[b, :, h, 1::2]) * np.exp(1j * ang)
            kr = (k[b, :, h, 0::2] + 1j * k[b, :, h, 1::2]) * np.exp(1j * ang)
            s = (qr @ np.conj(kr).T).real / math.sqrt(128)
            np.testing.assert_allclose(o[b, :, h], softmax(s, axis=1) @ v[b, :, h], atol=1e-12)
            np.testing.assert_allclose(lse[b, h], logsumexp(s, axis=1), atol=1e-12)


def test_cross_attention_mask_and_empty_rows():
    B, Lq, Lk, H, d = 3, 9, 40, 2, 128
    q, k, v = _rand(B, Lq, H, d), _rand(B, Lk, H, d), _rand(B, Lk, H, d)
    lens = np.array([0, 1, 23])
    o, lse = ref.cross_attention_fwd(q, k, v, lens)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    np.testing.assert_allclose(o[1], np.broadcast_to(v[1, :1], o[1].shape), atol=1e-14)
    k2, v2 = k.copy(), v.copy()
    k2[2, 23:] = 1e3
    v2[2, 23:] = -7.0
    o2, lse2 = ref.cross_attention_fwd(q, k2, v2, lens)
    np.testing.assert_array_equal(o2, o)
    np.testing.assert_array_equal(lse2, lse)
    s = q[2, :, 1] @ k[2, :23, 1].T / math.sqrt(d)
    np.testing.assert_allclose(o[2, :, 1], softmax(s, axis=1) @ v[2, :23, 1], atol=1e-13)


def test_two_part_merge_equals_whole():
    q, k, v = _rand(20, 128), _rand(333, 128), _rand(333, 128)
    scale = 1 / math.sqrt(128)
    o, lse = ref.softmax_attention(q, k, v, scale)
    oa, la = ref.softmax_attention(q, k[:100], v[:100], scale)
    ob, lb = ref.softmax_attention(q, k[100:], v[100:], scale)
    om, lm = ref.merge_partials(oa, la, ob, lb)
    np.testing.assert_allclose(om, o, atol=1e-13)
    np.testing.assert_allclose(lm, lse, atol=1e-12)
    # an empty part is the identity
    oe, le = ref.softmax_attention(q, k[:0], v[:0], scale, n_valid=0)
    om2, lm2 = ref.merge_partials(oe, le, o, lse)
    np.testing.assert_allclose(om2, o, atol=1e-15)
    np.testing.assert_allclose(lm2, lse, atol=1e-15)


def test_row_subset_helpers_match_full():
    grid = (2, 4, 5)
    L, d = 40, 128
    q, k, v, do = (_rand(1, L, 1, d) for _ in range(4))
    o, lse = ref.self_attention_fwd(q, k, v, grid)
    dq, dk, dv = ref.self_attention_bwd(q, k, v, do, grid)
    rows = np.array([0, 7, 39, 21])
    o_r, lse_r = ref.self_attention_fwd_rows(q[0, rows, 0], rows, k[0, :, 0], v[0, :, 0], grid)
    np.testing.assert_allclose(o_r, o[0, rows, 0], atol=1e-14)
    np.testing.assert_allclose(lse_r, lse[0, 0, rows], atol=1e-14)
    dq_r = ref.self_attention_bwd_dq_rows(q[0, rows, 0], do[0, rows, 0], rows,
                                          k[0, :, 0], v[0, :, 0], grid)
    np.testing.assert_allclose(dq_r, dq[0, rows, 0], atol=1e-13)


def test_key_row_gradients_match_full_backward():
    """dK / dV of selected key rows (all query rows visited, LSE and D from
    the oracle's own forward) equal those rows of the full backward, whether
    the forward blocks run in order or through a thread pool, and with a
    block that does not divide L."""
    from concurrent.futures import ThreadPoolExecutor

    grid = (3, 5, 7)
    L, d = 105, 128
    q, k, v, do = (_rand(1, L, 1, d) for _ in range(4))
    _, dk, dv = ref.self_attention_bwd(q, k, v, do, grid)
    keys = np.array([0, 104, 51, 7, 52])
    args = (q[0, :, 0], k[0, :, 0], v[0, :, 0], do[0, :, 0], keys, grid)
    dk_r, dv_r = ref.self_attention_bwd_dkdv_rows(*args, block=16)
    np.testing.assert_allclose(dk_r, dk[0, keys, 0], atol=1e-12)
    np.testing.assert_allclose(dv_r, dv[0, keys, 0], atol=1e-12)
    with ThreadPoolExecutor(4) as ex:
        dk_t, dv_t = ref.self_attention_bwd_dkdv_rows(*args, block=10, row_map=ex.map)
    np.testing.assert_allclose(dk_t, dk_r, atol=1e-13)
    np.testing.assert_allclose(dv_t, dv_r, atol=1e-13)


def test_key_row_gradients_central_differences():
    """The key-row helper against central differences of sum(O * dO) taken
    directly (not through the full backward)."""
    grid = (2, 2, 3)
    L, d = 12, 128
    theta, scale = 10000.0, 1.0 / math.sqrt(d)
    q, k, v, do = (_rand(1, L, 1, d) for _ in range(4))
    keys = np.array([3, 11])
    dk_r, dv_r = ref.self_attention_bwd_dkdv_rows(q[0, :, 0], k[0, :, 0], v[0, :, 0], do[0, :, 0], keys, grid)
    eps = 1e-5
    for name, g in (("k", dk_r), ("v", dv_r)):
        for a, j in enumerate(keys):
            for x in (0, 45, 90, 127):
                plus, minus = {"k": k.copy(), "v": v.copy()}, {"k": k.copy(), "v": v.copy()}
                plus[name][0, j, 0, x] += eps
                minus[name][0, j, 0, x] -= eps
                fd = (_objective(q, plus["k"], plus["v"], do, grid, theta, scale)
                      - _objective(q, minus["k"], minus["v"], do, grid, theta, scale)) / (2 * eps)
                assert abs(fd - g[a, x]) < 1e-7 * max(1.0, abs(g[a, x])), (name, j, x, fd, g[a, x])


# ---------------------------------------------------------------------------
# Backward


def _objective(q, k, v, do, grid, theta, scale):
    o, _ = ref.self_attention_fwd(q, k, v, grid, theta, scale)
    return float(np.sum(o * do))


@pytest.mark.parametrize("d,grid", [(12, (2, 2, 2)), (128, (2, 2, 3))])
def test_backward_central_differences(d, grid):
    L = grid[0] * grid[1] * grid[2]
    theta, scale = 10000.0, 1.0 / math.sqrt(d)
    q, k, v, do = (_rand(1, L, 2, d) for _ in range(4))
    dq, dk, dv = ref.self_attention_bwd(q, k, v, do, grid, theta, scale)
    eps = 1e-5
    picks = [tuple(RNG.integers(0, s) for s in q.shape) for _ in range(25)]
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in picks:
            xp = x.copy()
            xm = x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd = (_objective(args_p["q"], args_p["k"], args_p["v"], do, grid, theta, scale)
                  - _objective(args_m["q"], args_m["k"], args_m["v"], do, grid, theta, scale)) / (2 * eps)
            assert abs(fd - g[idx]) < 1e-7 * max(1.0, abs(g[idx])), (name, idx, fd, g[idx])


def test_backward_sum_invariants():
    grid = (3, 4, 4)
    L, H, d = 48, 2, 128
    q, k, v, do = (_rand(1, L, H, d) for _ in range(4))
    dq, dk, dv = ref.self_attention_bwd(q, k, v, do, grid)
    # every softmax row sums to one: sum_j dV_j = sum_i dO_i
    np.testing.assert_allclose(dv.sum(axis=1), do.sum(axis=1), atol=1e-11)
    # rows of dS sum to zero: the rotated key gradients sum to zero
    ang = ref.rope_angles(*grid, d)
    for h in range(H):
        dkr = ref.rope_rotate(dk[0, :, h], ang)
        np.testing.assert_allclose(dkr.sum(axis=0), 0.0, atol=1e-11)
    # zero upstream gradient => zero gradients
    z = ref.self_attention_bwd(q, k, v, np.zeros_like(do), grid)
    assert all(np.all(g == 0) for g in z)


def test_backward_given_o_lse_equals_the_backward_with_exact_outputs():
    """With the exact O and LSE, the backward from given outputs is the
    backward that recomputes them (P = exp(s - LSE) is the softmax)."""
    m, n, d, scale = 24, 40, 16, 0.3
    qr, kr, vh, do = (RNG.standard_normal(sh) for sh in ((m, d), (n, d), (n, d), (m, d)))
    o, lse = ref.softmax_attention(qr, kr, vh, scale)
    got = ref.head_backward_given_o_lse(qr, do, kr, vh, o, lse, scale)
    want = ref._head_backward(qr, do, kr, vh, scale, 7)
    for g, w in zip(got, want):
        np.testing.assert_allclose(g, w, rtol=1e-10, atol=1e-12)


def test_backward_given_o_lse_uses_the_given_outputs():
    """A perturbed O row i moves only D_i: dQ_rot_i shifts by
    -scale (dO_i . delta) sum_j P_ij k_j, dK_rot_j by -scale (dO_i . delta) P_ij q_i,
    dV not at all. A shifted LSE row i scales that row's P, so its dQ_rot by e^-c."""
    m, n, d, scale = 6, 9, 8, 0.7
    qr, kr, vh, do = (RNG.standard_normal(sh) for sh in ((m, d), (n, d), (n, d), (m, d)))
    o, lse = ref.softmax_attention(qr, kr, vh, scale)
    base = ref.head_backward_given_o_lse(qr, do, kr, vh, o, lse, scale)
    p = np.exp(scale * (qr @ kr.T) - lse[:, None])
    i, delta = 2, RNG.standard_normal(d)
    o2 = o.copy()
    o2[i] += delta
    got = ref.head_backward_given_o_lse(qr, do, kr, vh, o2, lse, scale)
    c = float(do[i] @ delta)
    want_dq = base[0].copy()
    want_dq[i] -= scale * c * (p[i] @ kr)
    want_dk = base[1] - scale * c * np.outer(p[i], qr[i])
    np.testing.assert_allclose(got[0], want_dq, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got[1], want_dk, rtol=1e-10, atol=1e-12)
    np.testing.assert_array_equal(got[2], base[2])
    lse2 = lse.copy()
    lse2[i] += 0.75
    got = ref.head_backward_given_o_lse(qr, do, kr, vh, o, lse2, scale)
    np.testing.assert_allclose(got[0][i], np.exp(-0.75) * base[0][i], rtol=1e-10)
    np.testing.assert_allclose(np.delete(got[0], i, axis=0), np.delete(base[0], i, axis=0), rtol=1e-12)


def test_flop_convention():
    assert ref.attention_flops(1, 40, 75600, 75600, 128) == pytest.approx(1.1705e14, rel=1e-4)
    assert ref.attention_flops(1, 12, 32760, 32760, 128) == pytest.approx(6.594e12, rel=1e-3)
    assert ref.attention_flops(1, 12, 262144, 262144, 128, backward=True) == pytest.approx(1.0555e15, rel=1e-3)


# ---------------------------------------------------------------------------
# Decoupled image/text cross-attention and Ring-attention chunks


def test_decoupled_cross_attention_identical_paths_double():
    rng = np.random.default_rng(21)
    q = rng.standard_normal((2, 9, 2, 16))
    k = rng.standard_normal((2, 5, 2, 16))
    v = rng.standard_normal((2, 5, 2, 16))
    lens = [5, 3]
    o, lse = ref.decoupled_cross_attention_fwd(q, k, v, lens, k, v, lens)
    o1, lse1 = ref.cross_attention_fwd(q, k, v, lens)
    np.testing.assert_allclose(o, 2.0 * o1, rtol=0, atol=1e-14)
    np.testing.assert_array_equal(lse, lse1)


def test_decoupled_cross_attention_empty_image_path_is_text_path():
    rng = np.random.default_rng(22)
    q = rng.standard_normal((1, 7, 1, 8))
    kt, vt = rng.standard_normal((1, 4, 1, 8)), rng.standard_normal((1, 4, 1, 8))
    ki, vi = rng.standard_normal((1, 6, 1, 8)), 1e6 * rng.standard_normal((1, 6, 1, 8))
    o, _ = ref.decoupled_cross_attention_fwd(q, kt, vt, [4], ki, vi, [0])
    # brute force of the text path alone
    for i in range(7):
        s = np.array([q[0, i, 0] @ kt[0, j, 0] for j in range(4)]) / math.sqrt(8)
        p = np.exp(s - s.max())
        p /= p.sum()
        np.testing.assert_allclose(o[0, i, 0], p @ vt[0, :, 0], rtol=1e-12, atol=1e-12)


def test_ring_chunks_of_all_keys_merge_to_full_attention():
    grid = (2, 3, 4)
    L = 24
    rng = np.random.default_rng(23)
    q, k, v = (rng.standard_normal((1, L, 1, 12)) for _ in range(3))
    o_full, lse_full = ref.self_attention_fwd(q, k, v, grid)
    q_start, m = 5, 11
    bounds = [0, 7, 8, 19, 24]
    o_run, lse_run = None, None
    for a, b in zip(bounds[:-1], bounds[1:]):
        o_c, lse_c = ref.self_attention_fwd_chunk(q[0, q_start:q_start + m, 0], q_start, k[0, a:b, 0], v[0, a:b, 0],
                                                  a, grid)
        if o_run is None:
            o_run, lse_run = o_c, lse_c
        else:
            o_run, lse_run = ref.merge_partials(o_run, lse_run, o_c, lse_c)
    np.testing.assert_allclose(o_run, o_full[0, q_start:q_start + m, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse_run, lse_full[0, 0, q_start:q_start + m], rtol=1e-13, atol=1e-13)


def test_ring_chunk_uses_grid_positions():
    # Shifting both chunks' token offsets by a whole number of frames keeps the
    # relative (t, h, w) offsets, hence the result (3D RoPE relativity).
    grid = (4, 2, 3)
    rng = np.random.default_rng(24)
    qr, kc, vc = rng.standard_normal((3, 16)), rng.standard_normal((5, 16)), rng.standard_normal((5, 16))
    o1, l1 = ref.self_attention_fwd_chunk(qr, 0, kc, vc, 6, grid)
    o2, l2 = ref.self_attention_fwd_chunk(qr, 6, kc, vc, 12, grid)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=1e-12, atol=1e-12)
    # ...but a shift of one token (changing w) does not.
    o3, _ = ref.self_attention_fwd_chunk(qr, 1, kc, vc, 6, grid)
    assert np.abs(o3 - o1).max() > 1e-3
