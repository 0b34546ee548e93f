"""Causal Conv3d of the Wan-VAE (with its feature cache) on the GPU, through
the C ABI, against the fp64 oracle.

Inputs are seeded N(0, 1) bf16; weights are N(0, 1) bf16 scaled by a power of
two near 1/sqrt(27 * C_in) (exact in bf16), so outputs are O(1) and the
workload tolerances (max-abs 2e-2, relative L2 5e-3) apply: the only
rounding beyond fp32 accumulation is the bf16 output (relative 2^-9).
"""
import math

import numpy as np
import pytest

import long_sequence_attention_02_b300 as wan
from long_sequence_attention_02_b300 import synth
from oracle import vae
from tests._util import bf16_round, bits, compare, dev_to_f64, f64, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _layer(seed, B, T, H, W, c_in, c_out, with_cache, with_bias):
    x = bits(seed, synth.STREAM_Q, (B, T, H, W, c_in))
    cache = bits(seed, synth.STREAM_K, (B, 2, H, W, c_in)) if with_cache else None
    shift = round(math.log2(math.sqrt(27 * c_in)))
    wt = bf16_round(f64(bits(seed, synth.STREAM_V, (c_out, 3, 3, 3, c_in))) * 2.0 ** -shift)
    bias = (f64(bits(seed, synth.STREAM_DO, (c_out,))) * 0.25).astype(np.float32) if with_bias else None
    return x, cache, wt, bias


def _run(x, cache, wt, bias, cache_out=True, stream=None):
    B, T, H, W, c_in = x.shape
    c_out = wt.shape[0]
    y = torch.empty(B, T, H, W, c_out, dtype=torch.bfloat16, device="cuda")
    co = torch.empty(B, 2, H, W, c_in, dtype=torch.bfloat16, device="cuda") if cache_out else None
    xd = x if isinstance(x, torch.Tensor) else to_dev(x)
    cd = None if cache is None else (cache if isinstance(cache, torch.Tensor) else to_dev(cache))
    bd = None if bias is None else torch.from_numpy(bias).cuda()
    wan.check(wan.wan_vae_causal_conv3d(xd, cd, to_dev(wt), bd, y, co, B, T, H, W, c_in, c_out, stream), "conv3d")
    wan.check(wan.wan_get_device_status())
    return y, co


@pytest.mark.parametrize("B,T,H,W,c_in,c_out,with_cache,with_bias", [
    (2, 3, 10, 19, 64, 128, True, True),     # ragged 8 x 16 patches, N = 128
    (1, 1, 8, 16, 128, 192, False, True),    # first chunk of one frame, N = 192
    (1, 2, 5, 33, 64, 256, True, False),     # N = 256, no bias
    (1, 4, 9, 17, 128, 320, False, True),    # N = 64 (320 = 5 x 64)
    (1, 2, 9, 17, 96, 96, True, True),       # 32-channel K steps (C_in 96), N = 96
    (1, 3, 8, 16, 32, 64, False, True),      # C_in 32: one K step per tap
    (2, 1, 5, 33, 160, 224, True, False),    # C_in 160 = 5 x 32, N = 224
    (1, 2, 7, 18, 96, 320, True, True),      # 32-channel K steps, N = 64 x 5
    (1, 2, 9, 17, 64, 32, True, True),       # C_out 32: one 32-channel store per tile, ragged
    # widths at (or near) a multiple of 128: tiles are 1 x 128 strips whose
    # three kw taps share one 130-pixel input box; with N <= 128 a tile
    # stacks two strips (rows h0, h0 + 1), the second below the picture when
    # H is odd
    (1, 2, 3, 128, 64, 128, True, True),     # two strips per tile, one tile per row pair, odd H
    (1, 2, 4, 250, 64, 192, True, True),     # one strip per tile (N = 192), ragged last strip (122 of 128)
    (1, 2, 3, 128, 64, 256, True, True),     # one strip per tile, N = 256
    (1, 1, 5, 250, 128, 160, False, True),   # one strip per tile, N = 160, ragged, first chunk
    (2, 1, 3, 256, 96, 96, False, True),     # two strips, 32-channel K steps, first chunk, B = 2
    (1, 3, 2, 128, 128, 320, True, False),   # two strips, N = 64 x 5
    (1, 2, 3, 124, 64, 64, True, True),      # two strips wider than the picture
    (1, 2, 1, 256, 32, 32, True, True),      # two strips, H = 1: every second strip below the picture
])
def test_conv3d_every_output(B, T, H, W, c_in, c_out, with_cache, with_bias):
    x, cache, wt, bias = _layer(21, B, T, H, W, c_in, c_out, with_cache, with_bias)
    y, co = _run(x, cache, wt, bias)
    y_ref, cache_ref = vae.causal_conv3d(f64(x), f64(wt), None if bias is None else bias.astype(np.float64),
                                         None if cache is None else f64(cache))
    compare(dev_to_f64(y), y_ref, "y")
    assert np.array_equal(dev_to_f64(co), cache_ref), "next cache"


def test_conv3d_chunks_through_the_cache_equal_the_whole_video():
    """Nine frames in chunks of 1, 4 and 4, each chunk fed the cache the
    previous call returned: equal to the oracle's whole-sequence layer, and
    bit for bit equal to the GPU's own whole-sequence call."""
    B, T, H, W, c_in, c_out = 1, 9, 8, 20, 64, 128
    x, _, wt, bias = _layer(22, B, T, H, W, c_in, c_out, False, True)
    xd = to_dev(x)
    whole, _ = _run(xd, None, wt, bias)
    outs, cache, t0 = [], None, 0
    for n in (1, 4, 4):
        y, cache = _run(xd[:, t0:t0 + n].contiguous(), cache, wt, bias)
        outs.append(y)
        t0 += n
    chunked = torch.cat(outs, dim=1)
    assert torch.equal(chunked, whole)
    y_ref, _ = vae.causal_conv3d(f64(x), f64(wt), bias.astype(np.float64))
    compare(dev_to_f64(chunked), y_ref, "chunked y")


def test_conv3d_strip_chunks_through_the_cache_equal_the_whole_video():
    """The same in two-strip tiles (width 128, N = 64): chunks of 2, 1 and 3 frames."""
    B, T, H, W, c_in, c_out = 1, 6, 3, 128, 64, 64
    x, _, wt, bias = _layer(24, B, T, H, W, c_in, c_out, False, True)
    xd = to_dev(x)
    whole, _ = _run(xd, None, wt, bias)
    outs, cache, t0 = [], None, 0
    for n in (2, 1, 3):
        y, cache = _run(xd[:, t0:t0 + n].contiguous(), cache, wt, bias)
        outs.append(y)
        t0 += n
    chunked = torch.cat(outs, dim=1)
    assert torch.equal(chunked, whole)
    y_ref, _ = vae.causal_conv3d(f64(x), f64(wt), bias.astype(np.float64))
    compare(dev_to_f64(chunked), y_ref, "chunked y (strips)")


def test_conv3d_without_cache_output_on_a_side_stream():
    x, cache, wt, bias = _layer(23, 1, 2, 8, 16, 64, 64, True, True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y, co = _run(x, cache, wt, bias, cache_out=False, stream=s)
    s.synchronize()
    assert co is None
    y_ref, _ = vae.causal_conv3d(f64(x), f64(wt), bias.astype(np.float64), f64(cache))
    compare(dev_to_f64(y), y_ref, "y (side stream)")


def test_conv3d_full_size_sampled():
    """The 720p decoder-scale layer (4 frames of 90 x 160, 384 -> 384 channels,
    with a cache) on 512 seeded sampled output positions."""
    from long_sequence_attention_02_b300.workloads import CONV_WORKLOADS

    w = CONV_WORKLOADS["wan_vae_conv3d_720p_384"]
    x, cache, wt, bias = _layer(24, w.B, w.T, w.H, w.W, w.c_in, w.c_out, True, True)
    y, co = _run(x, cache, wt, bias)
    rng = np.random.default_rng(25)
    n = 512
    pos = list(zip(rng.integers(0, w.B, n), rng.integers(0, w.T, n), rng.integers(0, w.H, n),
                   rng.integers(0, w.W, n)))
    pos[:4] = [(0, 0, 0, 0), (0, w.T - 1, w.H - 1, w.W - 1), (0, 0, w.H - 1, 0), (0, 1, 0, w.W - 1)]
    got = dev_to_f64(torch.stack([y[p] for p in pos]))
    ref = vae.causal_conv3d_at(f64(x), f64(wt), bias.astype(np.float64), f64(cache), pos)
    compare(got, ref, "y (sampled)")
    assert np.array_equal(dev_to_f64(co), f64(x[:, -2:])), "next cache"


def test_conv3d_timed_layer_sampled():
    """The layer the benchmark times (4 frames of 360 x 640, 192 -> 192
    channels, with a cache: 360 x 5 output strips of 128 pixels per frame) on
    512 seeded sampled positions plus the corners, the last row and column,
    and both sides of every strip boundary."""
    from long_sequence_attention_02_b300.workloads import CONV_WORKLOADS

    w = CONV_WORKLOADS["wan_vae_conv3d_360x640_192"]
    x, cache, wt, bias = _layer(26, w.B, w.T, w.H, w.W, w.c_in, w.c_out, True, True)
    y, co = _run(x, cache, wt, bias)
    rng = np.random.default_rng(27)
    n = 512
    pos = list(zip(rng.integers(0, w.B, n), rng.integers(0, w.T, n), rng.integers(0, w.H, n),
                   rng.integers(0, w.W, n)))
    T, H, W = w.T, w.H, w.W
    edges = [(0, 0, 0, 0), (0, T - 1, H - 1, W - 1), (0, 0, H - 1, 0), (0, T - 1, 0, W - 1),
             (0, 1, H - 8, W - 16), (0, 2, H - 1, W - 17), (0, 3, H - 9, W - 1), (0, 0, 7, 15), (0, 0, 8, 16)]
    edges += [(0, t, H - 1, int(c)) for t in range(T) for c in rng.integers(0, W, 8)]
    edges += [(0, t, int(r), W - 1) for t in range(T) for r in rng.integers(0, H, 8)]
    edges += [(0, int(rng.integers(T)), int(rng.integers(H)), w0 + d) for w0 in range(128, W, 128) for d in (-1, 0)]
    pos = edges + pos
    got = dev_to_f64(torch.stack([y[p] for p in pos]))
    ref = vae.causal_conv3d_at(f64(x), f64(wt), bias.astype(np.float64), f64(cache), pos)
    compare(got, ref, "y (timed layer, sampled)")
    assert np.array_equal(dev_to_f64(co), f64(x[:, -2:])), "next cache"


def test_conv3d_96_channels_chunks_equal_the_whole_video():
    """The 32-channel K-step path through the cache: chunks of 1, 4 and 4 frames
    are bit for bit the whole-sequence call, and match the oracle."""
    B, T, H, W, c_in, c_out = 1, 9, 8, 20, 96, 96
    x, _, wt, bias = _layer(28, B, T, H, W, c_in, c_out, False, True)
    xd = to_dev(x)
    whole, _ = _run(xd, None, wt, bias)
    outs, cache, t0 = [], None, 0
    for n in (1, 4, 4):
        y, cache = _run(xd[:, t0:t0 + n].contiguous(), cache, wt, bias)
        outs.append(y)
        t0 += n
    assert torch.equal(torch.cat(outs, dim=1), whole)
    y_ref, _ = vae.causal_conv3d(f64(x), f64(wt), bias.astype(np.float64))
    compare(dev_to_f64(whole), y_ref, "96-channel y")


def test_conv3d_96_channel_720p_layer_sampled():
    """A full-resolution 720p outer-stage layer (4 frames of 720 x 1280, 96 -> 96
    channels, with a cache) on 512 seeded positions plus corners and edges."""
    from long_sequence_attention_02_b300.workloads import CONV_WORKLOADS

    w = CONV_WORKLOADS["wan_vae_conv3d_720x1280_96"]
    x, cache, wt, bias = _layer(29, w.B, w.T, w.H, w.W, w.c_in, w.c_out, True, True)
    y, co = _run(x, cache, wt, bias)
    rng = np.random.default_rng(30)
    n = 512
    T, H, W = w.T, w.H, w.W
    pos = [(0, 0, 0, 0), (0, T - 1, H - 1, W - 1), (0, 0, H - 1, 0), (0, T - 1, 0, W - 1), (0, 1, H - 8, W - 16)]
    pos += [(0, int(rng.integers(T)), int(rng.integers(H)), w0 + d) for w0 in range(128, W, 128) for d in (-1, 0)]
    pos += list(zip(rng.integers(0, w.B, n), rng.integers(0, T, n), rng.integers(0, H, n), rng.integers(0, W, n)))
    got = dev_to_f64(torch.stack([y[p] for p in pos]))
    ref = vae.causal_conv3d_at(f64(x), f64(wt), bias.astype(np.float64), f64(cache), pos)
    compare(got, ref, "y (96-channel 720p layer, sampled)")
    assert np.array_equal(dev_to_f64(co), f64(x[:, -2:])), "next cache"
