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

Parity pins (tests/test_oracle_vae.py): pure-Python brute-force loops on a
tiny case, chunked-with-cache equals one whole-sequence convolution,
causality, a centre-tap kernel equals a per-pixel matrix product, one-hot
kernels shift the input by the expected frame and pixel offsets, and the
cache update for one-frame chunks.
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
