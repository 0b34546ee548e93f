"""Failure detection without a GPU fault: a producer that withholds one tile
makes the consumers' bounded waits expire; the kernel reports WAN_ERR_TIMEOUT
through the device error word, frees its resources and returns, and the
context stays usable."""
import math

import numpy as np
import pytest

import long_sequence_attention_02_b300 as wan
from long_sequence_attention_02_b300 import synth
from oracle import ref
from tests._util import bits, compare, dev_to_f64, f64, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _tiny():
    grid, B, H = (2, 4, 8), 1, 1
    shape = (B, 64, H, 128)
    return grid, [bits(7, s, shape) for s in (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V)]


def test_withheld_tile_times_out_and_context_survives():
    grid, (qb, kb, vb) = _tiny()
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    assert wan.wan_get_device_status() == wan.WAN_OK
    wan.check(wan.wan_debug_inject_stall(1, 200))
    try:
        o, lse = wan.attention_forward(q, k, v, grid)  # launch itself succeeds
    finally:
        wan.wan_debug_inject_stall(0, 100)
    assert wan.wan_get_device_status() == wan.WAN_ERR_TIMEOUT
    assert wan.wan_get_device_status() == wan.WAN_OK  # the word was cleared
    # the next launch is normal and correct
    o, lse = wan.attention_forward(q, k, v, grid)
    assert wan.wan_get_device_status() == wan.WAN_OK
    o_ref, lse_ref = ref.self_attention_fwd(f64(qb), f64(kb), f64(vb), grid)
    compare(dev_to_f64(o), o_ref, "O after recovery")
    compare(dev_to_f64(lse), lse_ref, "LSE after recovery")


def test_timeout_in_cross_attention():
    grid, (qb, kb, vb) = _tiny()
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    wan.check(wan.wan_debug_inject_stall(1, 100))
    try:
        wan.cross_attention_forward(q, k, v, None, grid)
    finally:
        wan.wan_debug_inject_stall(0, 100)
    assert wan.wan_get_device_status() == wan.WAN_ERR_TIMEOUT
    o, _ = wan.cross_attention_forward(q, k, v, None, grid)
    assert wan.wan_get_device_status() == wan.WAN_OK
    o_ref, _ = ref.cross_attention_fwd(f64(qb), f64(kb), f64(vb), [64])
    compare(dev_to_f64(o), o_ref, "xattn O after recovery")


def test_timeout_in_backward():
    grid, B, H = (2, 8, 16), 1, 1
    shape = (B, 256, H, 128)
    qb, kb, vb, dob = [bits(9, s, shape) for s in (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V,
                                                     synth.STREAM_DO)]
    q, k, v, do = (to_dev(x) for x in (qb, kb, vb, dob))
    o, lse = wan.attention_forward(q, k, v, grid)
    assert wan.wan_get_device_status() == wan.WAN_OK
    wan.check(wan.wan_debug_inject_stall(1, 100))
    try:
        wan.attention_backward(q, k, v, o, lse, do, grid)
    finally:
        wan.wan_debug_inject_stall(0, 100)
    assert wan.wan_get_device_status() == wan.WAN_ERR_TIMEOUT
    dq, dk, dv = wan.attention_backward(q, k, v, o, lse, do, grid)
    assert wan.wan_get_device_status() == wan.WAN_OK
    dq_r, dk_r, dv_r = ref.self_attention_bwd(f64(qb), f64(kb), f64(vb), f64(dob), grid)
    compare(dev_to_f64(dq), dq_r, "dQ after recovery")
    compare(dev_to_f64(dv), dv_r, "dV after recovery")


def test_timeout_in_fp8_forward():
    grid, (qb, kb, vb) = _tiny()
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    wan.check(wan.wan_debug_inject_stall(1, 100))
    try:
        wan.attention_forward_fp8(q, k, v, grid)
    finally:
        wan.wan_debug_inject_stall(0, 100)
    assert wan.wan_get_device_status() == wan.WAN_ERR_TIMEOUT
    o, lse = wan.attention_forward_fp8(q, k, v, grid)
    assert wan.wan_get_device_status() == wan.WAN_OK
    o_ref, lse_ref = ref.self_attention_fwd(f64(qb), f64(kb), f64(vb), grid)
    # the FP8 tolerance (derived in test_fp8_gpu.py): relative L2 0.12 on O, LSE max-abs 0.2
    compare(dev_to_f64(o), o_ref, "fp8 O after recovery", max_abs=0.15 * float(np.abs(o_ref).max()), rel_l2=0.12)
    compare(dev_to_f64(lse), lse_ref, "fp8 LSE after recovery", max_abs=0.2, rel_l2=float("inf"))


@pytest.mark.parametrize("W,c_out", [
    (16, 128),    # 8 x 16 patches: A and B of a K step on one barrier
    (128, 192),   # 1 x 128 strips (N = 192): input and weight rings with producers of their own
    (128, 64),    # two strips per tile (N = 64)
])
def test_timeout_in_conv3d(W, c_out):
    """The VAE Conv3d's input producer withholds one box: the MMA warp's
    bounded wait expires, the weight producer and the epilogue stop on the
    abort flag, TMEM is freed, and the next call is correct."""
    from oracle import vae
    from tests._util import bf16_round

    B, T, H, c_in = 1, 2, 8, 64
    x = bits(11, synth.STREAM_Q, (B, T, H, W, c_in))
    wt = bf16_round(f64(bits(11, synth.STREAM_V, (c_out, 3, 3, 3, c_in))) * 2.0 ** -5)
    xd, wd = to_dev(x), to_dev(wt)
    y = torch.empty(B, T, H, W, c_out, dtype=torch.bfloat16, device="cuda")
    wan.check(wan.wan_debug_inject_stall(1, 100))
    try:
        wan.check(wan.wan_vae_causal_conv3d(xd, None, wd, None, y, None, B, T, H, W, c_in, c_out))
    finally:
        wan.wan_debug_inject_stall(0, 100)
    assert wan.wan_get_device_status() == wan.WAN_ERR_TIMEOUT
    wan.check(wan.wan_vae_causal_conv3d(xd, None, wd, None, y, None, B, T, H, W, c_in, c_out))
    assert wan.wan_get_device_status() == wan.WAN_OK
    y_ref, _ = vae.causal_conv3d(f64(x), f64(wt))
    compare(dev_to_f64(y), y_ref, "conv3d y after recovery")
