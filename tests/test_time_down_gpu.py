"""The Wan-VAE's time-downsampling layer (3 x 1 x 1 taps, stride 2 in time,
one cached frame) on the GPU, through the C ABI, against the fp64 oracle.

Inputs are seeded N(0, 1) bf16; weights are N(0, 1) bf16 scaled by a power of
two near 1/sqrt(3 * C_in) (exact in bf16), so outputs are O(1) and the
workload tolerances (max-abs 2e-2, relative L2 5e-3) apply: the only rounding
beyond fp32 accumulation is the bf16 output (relative 2^-9).
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
    cache = bits(seed, synth.STREAM_K, (B, 1, H, W, c_in)) if with_cache else None
    shift = round(math.log2(math.sqrt(3 * c_in)))
    wt = bf16_round(f64(bits(seed, synth.STREAM_V, (c_out, 3, c_in))) * 2.0 ** -shift)
    bias = (f64(bits(seed, synth.STREAM_DO, (c_out,))) * 0.25).astype(np.float32) if with_bias else None
    return x, cache, wt, bias


def _run(x, cache, wt, bias, cache_out=True, stream=None):
    B, T, H, W, c_in = x.shape
    c_out = c_in if cache is None else wt.shape[0]
    t_out = T if cache is None else T // 2
    y = torch.empty(B, t_out, H, W, c_out, dtype=torch.bfloat16, device="cuda")
    co = torch.empty(B, 1, H, W, c_in, dtype=torch.bfloat16, device="cuda") if cache_out else None
    xd = x if isinstance(x, torch.Tensor) else to_dev(x)
    cd = None if cache is None else (cache if isinstance(cache, torch.Tensor) else to_dev(cache))
    wd = None if wt is None else (wt if isinstance(wt, torch.Tensor) else to_dev(wt))
    bd = None if bias is None else torch.from_numpy(bias).cuda()
    wan.check(wan.wan_vae_time_downsample(xd, cd, wd, bd, y, co, B, T, H, W, c_in, c_out, stream), "time_down")
    wan.check(wan.wan_get_device_status())
    return y, co


@pytest.mark.parametrize("B,T,H,W,c_in,c_out,with_bias", [
    (2, 4, 10, 19, 64, 128, True),      # ragged 8 x 16 patches, N = 128
    (1, 2, 9, 17, 96, 96, True),        # 32-channel K steps (C_in 96)
    (1, 6, 8, 16, 128, 256, False),     # 3 output frames, N = 256, no bias
    (1, 4, 7, 33, 192, 320, True),      # N = 64 x 5, ragged
    (1, 2, 5, 18, 32, 64, True),        # C_in 32: one K step per tap
])
def test_time_down_every_output(B, T, H, W, c_in, c_out, with_bias):
    x, cache, wt, bias = _layer(41, B, T, H, W, c_in, c_out, True, with_bias)
    y, co = _run(x, cache, wt, bias)
    y_ref, cache_ref = vae.causal_time_downsample(f64(x), f64(wt), None if bias is None else bias.astype(np.float64),
                                                  f64(cache))
    compare(dev_to_f64(y), y_ref, "y")
    assert np.array_equal(dev_to_f64(co), cache_ref), "next cache"


def test_time_down_first_chunk_passes_through():
    """A first chunk (one frame, no cache) is copied to y and to the next
    cache bit for bit; the weights are not read."""
    x, _, _, _ = _layer(42, 2, 1, 9, 17, 64, 64, False, False)
    y, co = _run(x, None, None, None)
    assert np.array_equal(dev_to_f64(y), f64(x))
    assert np.array_equal(dev_to_f64(co), f64(x))


@pytest.mark.parametrize("chunks", [(1, 4, 4), (1, 2, 6), (1, 8)])
def test_time_down_chunks_through_the_cache(chunks):
    """Nine frames in chunks through the one-frame cache: the oracle's chunked
    layer (pinned to the whole-video convolution), and bit for bit the same
    GPU outputs whatever the chunking."""
    B, T, H, W, c_in, c_out = 1, 9, 8, 20, 64, 64
    x, _, wt, bias = _layer(43, B, T, H, W, c_in, c_out, False, True)
    xd, wd = to_dev(x), to_dev(wt)
    outs, cache, t0 = [], None, 0
    for n in chunks:
        y, cache = _run(xd[:, t0:t0 + n].contiguous(), cache, wd, bias)
        outs.append(y)
        t0 += n
    got = torch.cat(outs, dim=1)
    ref = vae.causal_time_downsample_chunked(f64(x), f64(wt), bias.astype(np.float64), list(chunks))
    compare(dev_to_f64(got), ref, f"chunks {chunks}")
    # the first chunk's frame passes through exactly
    assert np.array_equal(dev_to_f64(got[:, :1]), f64(x[:, :1]))
    if chunks != (1, 4, 4):
        base, cache, t0 = [], None, 0
        for n in (1, 4, 4):
            y, cache = _run(xd[:, t0:t0 + n].contiguous(), cache, wd, bias)
            base.append(y)
            t0 += n
        assert torch.equal(got, torch.cat(base, dim=1))


def test_time_down_cache_out_may_be_the_cache_it_reads():
    """cache_out == cache: the layer reads the old frame before it is replaced."""
    x, cache, wt, bias = _layer(44, 1, 4, 8, 16, 64, 64, True, True)
    cd = to_dev(cache)
    y = torch.empty(1, 2, 8, 16, 64, dtype=torch.bfloat16, device="cuda")
    wan.check(wan.wan_vae_time_downsample(to_dev(x), cd, to_dev(wt), torch.from_numpy(bias).cuda(), y, cd,
                                          1, 4, 8, 16, 64, 64, None))
    torch.cuda.synchronize()
    y_ref, cache_ref = vae.causal_time_downsample(f64(x), f64(wt), bias.astype(np.float64), f64(cache))
    compare(dev_to_f64(y), y_ref, "y (in-place cache)")
    assert np.array_equal(dev_to_f64(cd), cache_ref)


def test_time_down_on_a_side_stream_without_cache_out():
    x, cache, wt, bias = _layer(45, 1, 2, 8, 16, 64, 64, True, True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y, co = _run(x, cache, wt, bias, cache_out=False, stream=s)
    s.synchronize()
    assert co is None
    y_ref, _ = vae.causal_time_downsample(f64(x), f64(wt), bias.astype(np.float64), f64(cache))
    compare(dev_to_f64(y), y_ref, "y (side stream)")


@pytest.mark.parametrize("name", ["wan_vae_time_down_180x320_192", "wan_vae_time_down_90x160_384"])
def test_time_down_full_size_crops(name):
    """The encoder's two downsampling layers at 720p. The kernel is 1 x 1 in
    space, so the oracle on a spatial crop of the inputs gives exactly that
    crop of the outputs: four corner crops, one crossing patch boundaries in
    the middle, and the last patch row and column in full."""
    from long_sequence_attention_02_b300.workloads import CONV_WORKLOADS

    w = CONV_WORKLOADS[name]
    x, cache, wt, bias = _layer(46, w.B, w.T, w.H, w.W, w.c_in, w.c_out, True, True)
    y, co = _run(x, cache, wt, bias)
    H, W = w.H, w.W
    crops = [(0, 9, 0, 17), (H - 9, H, 0, 17), (0, 9, W - 17, W), (H - 9, H, W - 17, W),
             (H // 2 - 5, H // 2 + 5, W // 2 - 9, W // 2 + 9), (H - 1, H, 0, W), (0, H, W - 1, W)]
    b64 = bias.astype(np.float64)
    for h0, h1, w0, w1 in crops:
        y_ref, _ = vae.causal_time_downsample(f64(x[:, :, h0:h1, w0:w1]), f64(wt), b64,
                                              f64(cache[:, :, h0:h1, w0:w1]))
        compare(dev_to_f64(y[:, :, h0:h1, w0:w1]), y_ref, f"{name} crop {(h0, h1, w0, w1)}")
    assert np.array_equal(dev_to_f64(co), f64(x[:, -1:])), "next cache"
