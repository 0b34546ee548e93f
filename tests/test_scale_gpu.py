"""The softmax scale is an argument of every attention entry point: the
forward, cross-attention and backward at scales other than 1/sqrt(128), every
row.

At 0.25 and 1.0 the logits of N(0, 1) inputs have standard deviations of about
2.8 and 11, so the softmax rows are peaked and many of them move their
reference maximum after the first key tile; at 0.02 they are nearly uniform.

The GPU rounds the rotated Q and K to bf16 before the product (relative
2^-9), so a logit s carries an absolute error of about |s| 2^-9: negligible
at the workload's scale, where logits are O(1), but about 0.1 at scale 1.0,
where they reach +-45, and exp() turns it into a 10 % error on the largest
weight. So every scale is compared, at the workload tolerance, with the
oracle's attention on bf16-rounded rotated operands (the oracle's RoPE in fp64,
then rounded, as the GPU's operands are). The backward is compared with the
oracle's backward from the O and LSE the GPU forward handed on: with peaked
rows, dS = P (dP - D) subtracts nearly equal numbers, and D comes from that
bf16 O. The plain oracle is held to the same tolerance where logits stay O(1)
(scale 0.02).

The backward also rounds dS (and P, for dV) to bf16 before its gradient
products: each term scale * dS_ij * k_j carries a relative 2^-9, and with
|dP| ~ |dO| |v| ~ sqrt(d) and |k| ~ sqrt(d) those terms grow like scale * d.
Against the workload's scale of 1/sqrt(d), for which the tolerances
(max-abs 2e-2, relative L2 5e-3) were set, the gradients' error therefore
grows by scale * sqrt(d), and the backward's tolerances are multiplied by
max(1, scale * sqrt(128)): 2.8 at 0.25, 11.3 at 1.0. A wrong sign, scale or
key gives errors of order 1 and still fails.
"""
import math

import numpy as np
import pytest

import long_sequence_attention_02_b300 as wan
from long_sequence_attention_02_b300 import synth
from oracle import ref
from tests._util import MAX_ABS, REL_L2, bf16_round, bits, compare, dev_to_f64, f64, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SCALES = [0.02, 0.25, 1.0]


def _inputs(B, L, H, seed, streams):
    return [bits(seed, s, (B, L, H, 128)) for s in streams]


def _bf16(x):
    return f64(bf16_round(x))


def _rotated_bf16(x_head, ang):
    """The oracle's RoPE of one head's rows, rounded to bf16 as the GPU's operands are."""
    return _bf16(ref.rope_rotate(x_head, ang))


def _fwd_bf16_operands(qb, kb, vb, grid, scale):
    B, L, H, d = qb.shape
    ang = ref.rope_angles(*grid, d)
    o = np.zeros((B, L, H, d))
    lse = np.zeros((B, H, L))
    for b in range(B):
        for h in range(H):
            qr = _rotated_bf16(f64(qb[b, :, h]), ang)
            kr = _rotated_bf16(f64(kb[b, :, h]), ang)
            o[b, :, h], lse[b, h] = ref.softmax_attention(qr, kr, f64(vb[b, :, h]), scale)
    return o, lse


def _bwd_bf16_operands(qb, kb, vb, dob, o_gpu, lse_gpu, grid, scale):
    """The oracle's backward from the outputs the GPU forward handed on (bf16
    O, fp32 LSE), on bf16-rounded rotated operands: the values the backward
    kernel is given."""
    B, L, H, d = qb.shape
    ang = ref.rope_angles(*grid, d)
    dq, dk, dv = (np.zeros((B, L, H, d)) for _ in range(3))
    for b in range(B):
        for h in range(H):
            qr = _rotated_bf16(f64(qb[b, :, h]), ang)
            kr = _rotated_bf16(f64(kb[b, :, h]), ang)
            dqr, dkr, dvh = ref.head_backward_given_o_lse(qr, f64(dob[b, :, h]), kr, f64(vb[b, :, h]),
                                                          o_gpu[b, :, h], lse_gpu[b, h], scale)
            dq[b, :, h] = ref.rope_rotate(dqr, ang, inverse=True)
            dk[b, :, h] = ref.rope_rotate(dkr, ang, inverse=True)
            dv[b, :, h] = dvh
    return dq, dk, dv


@pytest.mark.parametrize("scale", SCALES)
def test_self_attention_at_other_scales(scale):
    grid, B, H = (4, 16, 16), 1, 2          # 1024 tokens: 8 key tiles per query tile
    L = grid[0] * grid[1] * grid[2]
    qb, kb, vb = _inputs(B, L, H, 51, (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V))
    o, lse = wan.attention_forward(to_dev(qb), to_dev(kb), to_dev(vb), grid, scale=scale)
    wan.check(wan.wan_get_device_status())
    o, lse = dev_to_f64(o), dev_to_f64(lse)
    o_ref, lse_ref = _fwd_bf16_operands(qb, kb, vb, grid, scale)
    compare(o, o_ref, f"O (scale {scale})")
    compare(lse, lse_ref, f"LSE (scale {scale})")
    if scale < 0.05:
        o_ref, lse_ref = ref.self_attention_fwd(f64(qb), f64(kb), f64(vb), grid, scale=scale)
        compare(o, o_ref, f"O against the plain oracle (scale {scale})")
        compare(lse, lse_ref, f"LSE against the plain oracle (scale {scale})")


@pytest.mark.parametrize("scale", SCALES)
def test_cross_attention_at_other_scales(scale):
    grid, B, H, Lk = (3, 7, 9), 2, 2, 300
    Lq = grid[0] * grid[1] * grid[2]
    qb = bits(52, synth.STREAM_Q, (B, Lq, H, 128))
    kb = bits(52, synth.STREAM_K, (B, Lk, H, 128))
    vb = bits(52, synth.STREAM_V, (B, Lk, H, 128))
    lens = np.array([Lk, 150], dtype=np.int32)
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Lq, dtype=torch.float32, device="cuda")
    wan.check(wan.wan_xattn_fwd(q, k, v, torch.from_numpy(lens).cuda(), Lk, o, lse, B, grid, H, 128, scale))
    wan.check(wan.wan_get_device_status())
    # no RoPE here: the operands are the bf16 inputs themselves, so the plain oracle is the reference
    o_ref, lse_ref = ref.cross_attention_fwd(f64(qb), f64(kb), f64(vb), lens, scale=scale)
    compare(dev_to_f64(o), o_ref, f"cross O (scale {scale})")
    compare(dev_to_f64(lse), lse_ref, f"cross LSE (scale {scale})")


@pytest.mark.parametrize("scale", SCALES)
def test_backward_at_other_scales(scale):
    grid, B, H = (4, 8, 8), 1, 2             # 256 tokens
    L = grid[0] * grid[1] * grid[2]
    qb, kb, vb, dob = _inputs(B, L, H, 53, (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V, synth.STREAM_DO))
    q, k, v, do = (to_dev(x) for x in (qb, kb, vb, dob))
    tables = wan.rope_tables(grid)
    o, lse = wan.attention_forward(q, k, v, grid, tables=tables, scale=scale)
    dq, dk, dv = wan.attention_backward(q, k, v, o, lse, do, grid, tables=tables, scale=scale)
    wan.check(wan.wan_get_device_status())
    dq_r, dk_r, dv_r = _bwd_bf16_operands(qb, kb, vb, dob, dev_to_f64(o), dev_to_f64(lse), grid, scale)
    f = max(1.0, scale * math.sqrt(128))
    for name, got, want in (("dQ", dq, dq_r), ("dK", dk, dk_r), ("dV", dv, dv_r)):
        compare(dev_to_f64(got), want, f"{name} (scale {scale})", max_abs=MAX_ABS * f, rel_l2=REL_L2 * f)
    if scale < 0.05:
        dq_r, dk_r, dv_r = ref.self_attention_bwd(f64(qb), f64(kb), f64(vb), f64(dob), grid, scale=scale)
        compare(dev_to_f64(dq), dq_r, f"dQ against the plain oracle (scale {scale})")
        compare(dev_to_f64(dk), dk_r, f"dK against the plain oracle (scale {scale})")
        compare(dev_to_f64(dv), dv_r, f"dV against the plain oracle (scale {scale})")
