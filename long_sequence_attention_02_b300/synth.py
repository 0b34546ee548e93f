"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

Nothing here computes any part of attention. It draws i.i.d. N(0,1) values
rounded to bfloat16 (stored as raw uint16 bits) and integer key lengths from a
counter-based SplitMix64 stream, as the plain-C generator in
``csrc/synth.c`` defines; :func:`normal_bf16_numpy` is a second, pure-numpy
statement of the same generator used to cross-check it on small sizes.

Workload recipe (all configurations): every tensor element is N(0,1) drawn
from stream ``(seed, STREAM_<tensor>)``; cross-attention key lengths are
uniform integers on [16, 512] from ``(seed, STREAM_KV_LENS)``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

STREAM_Q = 1
STREAM_K = 2
STREAM_V = 3
STREAM_DO = 4
STREAM_KV_LENS = 5

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libwan_synth.so")
_lib = None

_GAMMA = 0x9E3779B97F4A7C15
_M64 = (1 << 64) - 1


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        from . import build as _build

        _build.build_synth()
    lib = ctypes.CDLL(_LIB_PATH)
    u64, p = ctypes.c_uint64, ctypes.c_void_p
    lib.wan_synth_normal_bf16.argtypes = [u64, u64, u64, u64, p]
    lib.wan_synth_normal_bf16_at.argtypes = [u64, u64, p, u64, p]
    lib.wan_synth_uniform_int.argtypes = [u64, u64, u64, ctypes.c_int64, ctypes.c_int64, p]
    lib.wan_synth_raw.argtypes = [u64, u64, p]
    for f in (lib.wan_synth_normal_bf16, lib.wan_synth_normal_bf16_at,
              lib.wan_synth_uniform_int, lib.wan_synth_raw):
        f.restype = None
    _lib = lib
    return lib


def normal_bf16(seed: int, stream: int, shape, offset: int = 0) -> np.ndarray:
    """bf16 bits (uint16) of N(0,1) elements ``offset .. offset+prod(shape)``."""
    n = int(np.prod(shape, dtype=np.int64))
    out = np.empty(n, dtype=np.uint16)
    if n:
        _load().wan_synth_normal_bf16(seed, stream, offset, n, out.ctypes.data)
    return out.reshape(shape)


def normal_bf16_at(seed: int, stream: int, flat_index: np.ndarray) -> np.ndarray:
    """bf16 bits of the elements at the given flat C-order indices."""
    idx = np.ascontiguousarray(flat_index, dtype=np.uint64)
    out = np.empty(idx.shape, dtype=np.uint16)
    if idx.size:
        _load().wan_synth_normal_bf16_at(seed, stream, idx.ctypes.data, idx.size,
                                         out.ctypes.data)
    return out


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    if n:
        _load().wan_synth_uniform_int(seed, stream, n, lo, hi, out.ctypes.data)
    return out


def kv_lens(seed: int, batch: int, lo: int = 16, hi: int = 512) -> np.ndarray:
    """Per-batch valid text-key lengths, uniform on [lo, hi] (int32)."""
    return uniform_int(seed, STREAM_KV_LENS, batch, lo, hi).astype(np.int32)


def raw_stream(key: int, n: int) -> np.ndarray:
    """First n SplitMix64 outputs from state ``key`` (generator self-check)."""
    out = np.empty(n, dtype=np.uint64)
    _load().wan_synth_raw(key, n, out.ctypes.data)
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32)


# ---------------------------------------------------------------------------
# Pure-numpy statement of the same generator (small sizes only).


def _mix(z):
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    a = int(_mix(np.uint64((seed + _GAMMA) & _M64)))
    return np.uint64((int(_mix(np.uint64((a + stream * _GAMMA) & _M64)))))


def normal_bf16_numpy(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    key = _key(seed, stream)
    e = np.arange(offset, offset + n, dtype=np.uint64)
    m = e >> np.uint64(1)
    with np.errstate(over="ignore"):
        x1 = _mix(key + (np.uint64(2) * m + np.uint64(1)) * np.uint64(_GAMMA))
        x2 = _mix(key + (np.uint64(2) * m + np.uint64(2)) * np.uint64(_GAMMA))
    u1 = ((x1 >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * 2.0 ** -53
    u2 = (x2 >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    a = 2.0 * np.pi * u2
    z = np.where((e & np.uint64(1)) == 1, r * np.sin(a), r * np.cos(a))
    b = z.view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    b = (b + np.uint64(0x1FFFFFFFFFFF) + lsb) & ~np.uint64(0x1FFFFFFFFFFF)
    f = b.view(np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
