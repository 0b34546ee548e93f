"""CPU oracle for the Wan-VAE causal 3D convolution with its feature cache (float64, numpy).

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this module. The CUDA
library never calls it and shares no code with it.

What it computes, and where the pages say so (gojay.top "Wan2.1" reading,
*Feature Cache 机制详解*, Fig. vae_cache and the table beside it):

* The VAE's 3D convolutions are causal: a time kernel of 3 frames, so the
  output at frame t reads frames t-2, t-1 and t; the time axis is padded only
  into the past.
* Video is processed in chunks of frames. The first chunk is padded with 2
  zero frames in time. Every later chunk is instead prefixed with the last 2
  input frames of the previous chunk (the feature cache, CACHE_T = 2). After
  the convolution the cache becomes the last 2 frames of (prefix ++ chunk).
* Chunked processing with the cache gives the same result as one
  convolution over the whole sequence (the pages' stated purpose of the cache).

Readings where the pages are silent (each is also listed in the design notes):

V1  The convolution is a cross-correlation, as a deep-learning Conv3d is:
    y[t, h, w, o] = bias[o] + sum_{kt, kh, kw, c} wt[o, kt, kh, kw, c] *
                    xp[t + kt, h + kh - 1, w + kw - 1, c],
    where xp is the input with its 2 past frames (zeros or the cache)
    prepended in time and 1 zero pixel on each side in height and width.
V2  Kernel 3 x 3 x 3, stride 1: the pages' plain causal layer, Fig. vae_cache
    (a). The stride-2 time-downsampling layer of Fig. vae_cache (b) is not
    covered.
V3  Layout channels-last: activations [B, T, H, W, C], weights
    [C_out, 3, 3, 3, C_in], bias [C_out]; the cache is [B, 2, H, W, C_in].
V4  Everything is float64 here; nothing is rounded to bf16.

The time-downsampling layer (same section, Fig. vae_cache (b) and the table
beside it): a causal convolution with stride 2 in time whose cache keeps
only the last frame. The first chunk gets no padding and is not convolved
in time (the first frame is compressed spatially only, as the VAE section
says); every later chunk is prefixed with the cached frame, so that its
output has exactly half its frames. Readings where the pages are silent:

V5  The kernel is 3 frames by 1 x 1 pixels (a purely temporal convolution:
    the spatial 2x downsampling is a separate layer), no padding, stride 2:
        y[t, h, w, o] = bias[o] + sum_{kt, c} wt[o, kt, c] * xq[2t + kt, h, w, c],
    where xq is the chunk with the cached frame in front of it.
V6  The first chunk (no cache) has one frame and passes through unchanged
    (so C_out = C_in); later chunks have an even number of frames.

Parity pins (tests/test_oracle_vae.py): pure-Python brute-force loops on a
tiny case, chunked-with-cache equals one whole-sequence convolution,
causality, a centre-tap kernel equals a per-pixel matrix product, one-hot
kernels shift the input by the expected frame and pixel offsets, and the
cache update for one-frame chunks; for the downsampling layer, a brute-force
loop, chunks of 1, 4, 4, ... through the cache equal the whole-sequence
definition, one-hot taps select frames 2t - 1, 2t and 2t + 1 of the chunk,
and the output has half the frames.
"""
from __future__ import annotations

import numpy as np

CACHE_T = 2  # past frames a time kernel of 3 needs


def _past_frames(x, cache):
    B, _, H, W, C = x.shape
    if cache is None:
        return np.zeros((B, CACHE_T, H, W, C), dtype=np.float64)
    cache = np.asarray(cache, dtype=np.float64)
    assert cache.shape == (B, CACHE_T, H, W, C), cache.shape
    return cache


def causal_conv3d(x, wt, bias=None, cache=None):
    """One causal Conv3d layer on one chunk (V1-V3).

    x: [B, T, H, W, C_in]; wt: [C_out, 3, 3, 3, C_in]; bias: [C_out] or None;
    cache: [B, 2, H, W, C_in] (the previous chunk's last two input frames) or
    None (the first chunk: two zero frames). Returns (y [B, T, H, W, C_out],
    new_cache [B, 2, H, W, C_in]).
    """
    x = np.asarray(x, dtype=np.float64)
    wt = np.asarray(wt, dtype=np.float64)
    B, T, H, W, _ = x.shape
    C_out = wt.shape[0]
    seq = np.concatenate([_past_frames(x, cache), x], axis=1)        # [B, 2 + T, H, W, C_in]
    xp = np.pad(seq, ((0, 0), (0, 0), (1, 1), (1, 1), (0, 0)))        # zero pixel border
    y = np.zeros((B, T, H, W, C_out), dtype=np.float64)
    for kt in range(3):
        for kh in range(3):
            for kw in range(3):
                window = xp[:, kt:kt + T, kh:kh + H, kw:kw + W, :]
                y += np.einsum("bthwc,oc->bthwo", window, wt[:, kt, kh, kw, :])
    if bias is not None:
        y += np.asarray(bias, dtype=np.float64)
    return y, seq[:, -CACHE_T:].copy()


def causal_conv3d_chunked(x, wt, bias=None, chunks=None):
    """The layer over a whole video in chunks, carrying the feature cache.

    chunks: frame counts summing to T; default 1, 4, 4, ... (the pages' split:
    the first chunk holds one frame, every later one four). Returns the
    outputs of all chunks concatenated in time.
    """
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[1]
    if chunks is None:
        chunks = [1] + [4] * ((T - 1) // 4)
        if sum(chunks) < T:
            chunks.append(T - sum(chunks))
    assert sum(chunks) == T and all(c > 0 for c in chunks)
    cache, outs, t0 = None, [], 0
    for n in chunks:
        y, cache = causal_conv3d(x[:, t0:t0 + n], wt, bias, cache)
        outs.append(y)
        t0 += n
    return np.concatenate(outs, axis=1)


def causal_conv3d_at(x, wt, bias, cache, positions):
    """Outputs at a list of (b, t, h, w) positions only, each computed
    directly from its 3 x 3 x 3 input window (for sampled checks of large
    layers). Returns [n, C_out]."""
    x = np.asarray(x)
    wt = np.asarray(wt, dtype=np.float64)
    B, T, H, W, C_in = x.shape
    out = np.zeros((len(positions), wt.shape[0]), dtype=np.float64)
    for i, (b, t, h, w) in enumerate(positions):
        acc = np.zeros(wt.shape[0], dtype=np.float64)
        for kt in range(3):
            ti = t + kt - CACHE_T
            if ti >= 0:
                frame = x[b, ti]
            elif cache is not None:
                frame = cache[b, ti + CACHE_T]
            else:
                continue
            for kh in range(3):
                hi = h + kh - 1
                if not 0 <= hi < H:
                    continue
                for kw in range(3):
                    wi = w + kw - 1
                    if not 0 <= wi < W:
                        continue
                    acc += wt[:, kt, kh, kw, :] @ np.asarray(frame[hi, wi], dtype=np.float64)
        out[i] = acc + (0.0 if bias is None else np.asarray(bias, dtype=np.float64))
    return out


def conv3d_flops(B, T, H, W, C_in, C_out):
    """Multiply-adds counted as 2 FLOP: 2 * outputs * C_out * 27 * C_in."""
    return 2.0 * B * T * H * W * C_out * 27 * C_in


# ---------------------------------------------------------------------------
# Time-downsampling layer (Fig. vae_cache (b))

TIME_DOWN_CACHE_T = 1  # frames the downsampling layer keeps for the next chunk


def causal_time_downsample(x, wt, bias=None, cache=None):
    """One time-downsampling layer on one chunk (V5, V6).

    x: [B, T, H, W, C_in]; wt: [C_out, 3, C_in]; bias: [C_out] or None;
    cache: [B, 1, H, W, C_in] (the previous chunk's last input frame) or None
    for the first chunk. Returns (y, new_cache): y [B, T/2, H, W, C_out] (the
    first chunk: x itself), new_cache = the chunk's last frame.
    """
    x = np.asarray(x, dtype=np.float64)
    new_cache = x[:, -TIME_DOWN_CACHE_T:].copy()
    if cache is None:
        assert x.shape[1] == 1, "the first chunk holds one frame"
        return x.copy(), new_cache
    wt = np.asarray(wt, dtype=np.float64)
    B, T, H, W, _ = x.shape
    assert T % 2 == 0, "later chunks hold an even number of frames"
    cache = np.asarray(cache, dtype=np.float64)
    assert cache.shape == (B, TIME_DOWN_CACHE_T, H, W, x.shape[4]), cache.shape
    xq = np.concatenate([cache, x], axis=1)                           # [B, 1 + T, H, W, C_in]
    y = np.zeros((B, T // 2, H, W, wt.shape[0]), dtype=np.float64)
    for kt in range(3):
        y += np.einsum("bthwc,oc->bthwo", xq[:, kt:kt + T - 1:2], wt[:, kt, :])
    if bias is not None:
        y += np.asarray(bias, dtype=np.float64)
    return y, new_cache


def causal_time_downsample_chunked(x, wt, bias=None, chunks=None):
    """The downsampling layer over a whole video of 1 + 4k frames in chunks of
    1, 4, 4, ... (or the given even-length chunks after the first one frame),
    carrying the one-frame cache. Returns the outputs concatenated in time:
    1 + 2k frames."""
    x = np.asarray(x, dtype=np.float64)
    T = x.shape[1]
    if chunks is None:
        chunks = [1] + [4] * ((T - 1) // 4)
    assert sum(chunks) == T and chunks[0] == 1
    cache, outs, t0 = None, [], 0
    for n in chunks:
        y, cache = causal_time_downsample(x[:, t0:t0 + n], wt, bias, cache)
        outs.append(y)
        t0 += n
    return np.concatenate(outs, axis=1)


def time_downsample_flops(B, T_out, H, W, C_in, C_out):
    """Multiply-adds counted as 2 FLOP: 2 * outputs * C_out * 3 * C_in."""
    return 2.0 * B * T_out * H * W * C_out * 3 * C_in
