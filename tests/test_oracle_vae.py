"""Pins of the causal Conv3d oracle (CPU only).

Each check is independent of the oracle's own formulation (shifted windows
and einsum): brute-force loops, the chunked == whole-sequence property the
pages state for the feature cache, causality, closed forms for one-hot and
centre-tap kernels.
"""
import numpy as np
import pytest

from oracle import vae


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _brute(x, wt, bias, cache):
    """Seven nested loops over (b, t, h, w, o) and the 27 taps, reading the
    past frames from the cache (or zero) and zero outside the picture."""
    B, T, H, W, Ci = x.shape
    Co = wt.shape[0]
    y = np.zeros((B, T, H, W, Co))
    for b in range(B):
        for t in range(T):
            for h in range(H):
                for w in range(W):
                    for o in range(Co):
                        s = bias[o]
                        for kt in range(3):
                            for kh in range(3):
                                for kw in range(3):
                                    ti, hi, wi = t + kt - 2, h + kh - 1, w + kw - 1
                                    if not (0 <= hi < H and 0 <= wi < W):
                                        continue
                                    if ti >= 0:
                                        src = x[b, ti, hi, wi]
                                    elif cache is not None:
                                        src = cache[b, ti + 2, hi, wi]
                                    else:
                                        continue
                                    for c in range(Ci):
                                        s += wt[o, kt, kh, kw, c] * src[c]
                        y[b, t, h, w, o] = s
    return y


@pytest.mark.parametrize("with_cache", [False, True])
def test_brute_force_tiny(with_cache):
    rng = np.random.default_rng(1)
    x = _rand(rng, 2, 3, 3, 4, 2)
    wt = _rand(rng, 3, 3, 3, 3, 2)
    bias = _rand(rng, 3)
    cache = _rand(rng, 2, 2, 3, 4, 2) if with_cache else None
    y, _ = vae.causal_conv3d(x, wt, bias, cache)
    np.testing.assert_allclose(y, _brute(x, wt, bias, cache), rtol=0, atol=1e-12)


@pytest.mark.parametrize("chunks", [None, [1, 4, 4], [2, 1, 3, 3], [9]])
def test_chunked_with_cache_equals_whole_sequence(chunks):
    rng = np.random.default_rng(2)
    x = _rand(rng, 1, 9, 5, 6, 3)
    wt = _rand(rng, 4, 3, 3, 3, 3)
    bias = _rand(rng, 4)
    whole, _ = vae.causal_conv3d(x, wt, bias)
    np.testing.assert_allclose(vae.causal_conv3d_chunked(x, wt, bias, chunks), whole, rtol=0, atol=1e-12)


def test_chunks_without_cache_differ_at_the_boundary():
    # zero padding every chunk instead of the cache: the first frame of the
    # second chunk changes, frames of the first chunk do not
    rng = np.random.default_rng(3)
    x = _rand(rng, 1, 5, 4, 4, 2)
    wt = _rand(rng, 2, 3, 3, 3, 2)
    whole, _ = vae.causal_conv3d(x, wt)
    y0, _ = vae.causal_conv3d(x[:, :1], wt)
    y1, _ = vae.causal_conv3d(x[:, 1:], wt)
    np.testing.assert_allclose(y0, whole[:, :1], atol=1e-12)
    assert np.abs(y1[:, 0] - whole[:, 1]).max() > 1e-3


def test_causality():
    rng = np.random.default_rng(4)
    x = _rand(rng, 1, 6, 4, 5, 2)
    wt = _rand(rng, 3, 3, 3, 3, 2)
    y, _ = vae.causal_conv3d(x, wt)
    x2 = x.copy()
    x2[:, 3] += 1.0
    y2, _ = vae.causal_conv3d(x2, wt)
    assert np.array_equal(y[:, :3], y2[:, :3])          # the past does not see frame 3
    for t in (3, 4, 5):                                 # frames 3..5 read it
        assert np.abs(y[:, t] - y2[:, t]).max() > 1e-6


def test_centre_tap_is_a_per_pixel_matrix_product():
    rng = np.random.default_rng(5)
    x = _rand(rng, 2, 3, 4, 5, 3)
    m = _rand(rng, 4, 3)
    bias = _rand(rng, 4)
    wt = np.zeros((4, 3, 3, 3, 3))
    wt[:, 2, 1, 1, :] = m            # current frame, same pixel
    y, _ = vae.causal_conv3d(x, wt, bias)
    np.testing.assert_allclose(y, x @ m.T + bias, atol=1e-12)


def test_one_hot_taps_shift_by_the_expected_offsets():
    rng = np.random.default_rng(6)
    x = _rand(rng, 1, 4, 4, 5, 2)
    cache = _rand(rng, 1, 2, 4, 5, 2)
    eye = np.eye(2)
    # kt = 0: two frames back; with no cache the first two frames read zeros
    wt = np.zeros((2, 3, 3, 3, 2))
    wt[:, 0, 1, 1, :] = eye
    y, _ = vae.causal_conv3d(x, wt)
    np.testing.assert_array_equal(y[:, 2:], x[:, :2])
    np.testing.assert_array_equal(y[:, :2], 0 * y[:, :2])
    y, _ = vae.causal_conv3d(x, wt, cache=cache)
    np.testing.assert_array_equal(y[:, :2], cache)
    # kh = 0: the pixel one row up (zero in row 0); kw = 2: one column right
    wt = np.zeros((2, 3, 3, 3, 2))
    wt[:, 2, 0, 1, :] = eye
    y, _ = vae.causal_conv3d(x, wt)
    np.testing.assert_array_equal(y[:, :, 1:], x[:, :, :-1])
    assert not y[:, :, 0].any()
    wt = np.zeros((2, 3, 3, 3, 2))
    wt[:, 2, 1, 2, :] = eye
    y, _ = vae.causal_conv3d(x, wt)
    np.testing.assert_array_equal(y[:, :, :, :-1], x[:, :, :, 1:])
    assert not y[:, :, :, -1].any()


def test_cache_update():
    rng = np.random.default_rng(7)
    wt = _rand(rng, 2, 3, 3, 3, 2)
    x1 = _rand(rng, 1, 1, 3, 3, 2)
    x4 = _rand(rng, 1, 4, 3, 3, 2)
    _, c = vae.causal_conv3d(x1, wt)                    # first chunk, one frame: [zero, x1[0]]
    assert not c[:, 0].any()
    np.testing.assert_array_equal(c[:, 1], x1[:, 0])
    _, c2 = vae.causal_conv3d(x4, wt, cache=c)          # a four-frame chunk keeps its own last two
    np.testing.assert_array_equal(c2, x4[:, 2:])
    _, c3 = vae.causal_conv3d(x1, wt, cache=c2)         # a one-frame chunk: [old last, new]
    np.testing.assert_array_equal(c3[:, 0], x4[:, 3])
    np.testing.assert_array_equal(c3[:, 1], x1[:, 0])


def test_sampled_positions_match_the_layer():
    rng = np.random.default_rng(8)
    x = _rand(rng, 2, 3, 5, 6, 3)
    wt = _rand(rng, 4, 3, 3, 3, 3)
    bias = _rand(rng, 4)
    cache = _rand(rng, 2, 2, 5, 6, 3)
    y, _ = vae.causal_conv3d(x, wt, bias, cache)
    pos = [(0, 0, 0, 0), (1, 2, 4, 5), (0, 1, 2, 3), (1, 0, 4, 0)]
    got = vae.causal_conv3d_at(x, wt, bias, cache, pos)
    np.testing.assert_allclose(got, np.stack([y[p] for p in pos]), atol=1e-12)


def test_flop_count():
    assert vae.conv3d_flops(1, 4, 90, 160, 384, 384) == 2 * 4 * 90 * 160 * 384 * 27 * 384


# ---------------------------------------------------------------------------
# Time-downsampling layer (stride 2 in time, one cached frame)


def _brute_down(x, wt, bias, cache):
    """Loops over (b, j, h, w, o) and the three taps: output frame j reads
    frames 2j - 1, 2j and 2j + 1 of the chunk, frame -1 being the cache."""
    B, T, H, W, Ci = x.shape
    Co = wt.shape[0]
    y = np.zeros((B, T // 2, H, W, Co))
    for b in range(B):
        for j in range(T // 2):
            for h in range(H):
                for w in range(W):
                    for o in range(Co):
                        s = bias[o]
                        for kt in range(3):
                            ti = 2 * j + kt - 1
                            src = x[b, ti, h, w] if ti >= 0 else cache[b, 0, h, w]
                            for c in range(Ci):
                                s += wt[o, kt, c] * src[c]
                        y[b, j, h, w, o] = s
    return y


def test_time_downsample_matches_brute_force():
    rng = np.random.default_rng(61)
    x, cache = _rand(rng, 2, 4, 3, 2, 5), _rand(rng, 2, 1, 3, 2, 5)
    wt, bias = _rand(rng, 4, 3, 5), _rand(rng, 4)
    y, new_cache = vae.causal_time_downsample(x, wt, bias, cache)
    np.testing.assert_allclose(y, _brute_down(x, wt, bias, cache), atol=1e-12)
    assert y.shape[1] == 2                              # exactly half the frames
    np.testing.assert_array_equal(new_cache, x[:, -1:])


def test_time_downsample_first_chunk_passes_through():
    rng = np.random.default_rng(62)
    x = _rand(rng, 1, 1, 4, 3, 6)
    y, new_cache = vae.causal_time_downsample(x, _rand(rng, 6, 3, 6), _rand(rng, 6), None)
    np.testing.assert_array_equal(y, x)
    np.testing.assert_array_equal(new_cache, x)


def test_time_downsample_one_hot_taps_select_frames():
    rng = np.random.default_rng(63)
    x, cache = _rand(rng, 1, 6, 2, 2, 3), _rand(rng, 1, 1, 2, 2, 3)
    for kt, shift in ((0, -1), (1, 0), (2, 1)):
        wt = np.zeros((3, 3, 3))
        wt[:, kt, :] = np.eye(3)
        y, _ = vae.causal_time_downsample(x, wt, None, cache)
        for j in range(3):
            src = x[:, 2 * j + shift] if 2 * j + shift >= 0 else cache[:, 0]
            np.testing.assert_array_equal(y[:, j], src)


def test_time_downsample_chunks_equal_the_whole_sequence():
    """Chunks of 1, 4, 4 frames through the one-frame cache give the
    whole-sequence definition: frame 0 unchanged, then output j >= 1 reads
    frames 2j - 2, 2j - 1 and 2j of the video."""
    rng = np.random.default_rng(64)
    T = 9
    x = _rand(rng, 1, T, 3, 4, 5)
    wt, bias = _rand(rng, 5, 3, 5), _rand(rng, 5)
    got = vae.causal_time_downsample_chunked(x, wt, bias)
    assert got.shape[1] == 1 + (T - 1) // 2
    want = np.zeros_like(got)
    want[:, 0] = x[:, 0]
    for j in range(1, got.shape[1]):
        want[:, j] = bias + sum(np.einsum("bhwc,oc->bhwo", x[:, 2 * j - 2 + kt], wt[:, kt]) for kt in range(3))
    np.testing.assert_allclose(got, want, atol=1e-12)
    other = vae.causal_time_downsample_chunked(x, wt, bias, chunks=[1, 2, 6])
    np.testing.assert_allclose(other, want, atol=1e-12)
