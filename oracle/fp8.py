"""CPU oracle of the FP8 (e4m3) reading of the attention forward (float64).

TEST INFRASTRUCTURE ONLY, like ``oracle.ref``: only the test suite may import
this module; it shares no code with the CUDA path.

The pages name FP8 attention among the Wan inference speed-ups ("Wan Team,
Alibaba (2025)" anthology note, *Key takeaways*; ctol.digital article,
*Speed, Scale, and Efficiency*: diffusion cache, FP8 quantisation and
activation offload together give 1.62x) but give no scheme. The reading
taken is the plainest per-head one:

  for each (b, h): s_x = amax|X| / 448 over the whole head of X, where X is
  the rotated Q, the rotated K, or V; X8 = e4m3(X / s_x), rounded to nearest
  even and saturated at +-448; the attention is then computed from the
  dequantised operands s_x * X8.

This module applies exactly that quantisation and then the plain fp64
softmax attention of ``oracle.ref``. It does not round the probabilities P
to e4m3 (the CUDA kernel does, for its P V product): comparing the kernel
with this oracle isolates the error of P's rounding and of fp32 arithmetic.

The e4m3 format (the 8-bit "E4M3" float without infinities): 1 sign bit,
4 exponent bits with bias 7, 3 mantissa bits. A code with exponent field
e >= 1 is (1 + m/8) * 2^(e-7); e = 0 gives the subnormals (m/8) * 2^-6.
Exponent 15 with mantissa 7 is NaN, so the largest finite value is
1.75 * 2^8 = 448 and the smallest positive one is 2^-9.
"""
from __future__ import annotations

import math

import numpy as np

from oracle import ref

E4M3_MAX = 448.0


def e4m3_decode(code):
    """Value of each 8-bit e4m3 code (NaN for the two NaN codes)."""
    c = np.asarray(code, dtype=np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((e == 15) & ((c & 0x7) == 7), np.nan, val)
    return sign * val


def e4m3_round(x):
    """Round float64 values to the nearest e4m3 value, ties to the even
    mantissa, saturating magnitudes beyond 448 at +-448 (finite inputs).

    Below 2^-6 the spacing is that of the subnormals, 2^-9; in the binade
    [2^E, 2^(E+1)) it is 2^(E-3). Dividing by the spacing gives an integer
    grid whose parity is the mantissa's last bit, so numpy's round-half-even
    ``rint`` is the tie rule.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, ex = np.frexp(a)                      # a = f * 2^ex, f in [0.5, 1)
    binade = np.maximum(ex - 1, -6)          # floor(log2 a), subnormals share 2^-6's spacing
    spacing = np.exp2(binade.astype(np.float64) - 3.0)
    r = np.rint(a / spacing) * spacing
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, x)


def quantise(x):
    """(e4m3 values of x / s, s) with s = amax|x| / 448 over all of x; an
    all-zero x keeps s = 1."""
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    s = amax / E4M3_MAX if amax > 0 else 1.0
    return e4m3_round(x / s), s


def head_operands(q_head, k_head, v_head, grid, theta=ref.DEFAULT_THETA):
    """Dequantised operands s_q Q8, s_k K8, s_v V8 of one (b, h) whose
    pre-RoPE rows are q_head, k_head, v_head [L, d] (all L tokens of the
    head: the scales are the whole head's)."""
    F, Hp, Wp = grid
    d = q_head.shape[1]
    ang = ref.rope_angles(F, Hp, Wp, d, theta)
    out = []
    for x in (ref.rope_rotate(q_head, ang), ref.rope_rotate(k_head, ang), v_head):
        x8, s = quantise(x)
        out.append(s * x8)
    return tuple(out)


def fp8_self_attention_fwd(q, k, v, grid, theta=ref.DEFAULT_THETA, scale=None, block=1024):
    """3D-RoPE self-attention on e4m3-quantised operands with per-head scales.

    q, k, v: float64 [B, L, H, d]. Returns O [B, L, H, d] and LSE [B, H, L].
    """
    B, L, H, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = np.zeros((B, L, H, d))
    lse = np.zeros((B, H, L))
    for b in range(B):
        for h in range(H):
            qd, kd, vd = head_operands(q[b, :, h], k[b, :, h], v[b, :, h], grid, theta)
            for i0 in range(0, L, block):
                i1 = min(L, i0 + block)
                o[b, i0:i1, h], lse[b, h, i0:i1] = ref.softmax_attention(qd[i0:i1], kd, vd, scale)
    return o, lse
