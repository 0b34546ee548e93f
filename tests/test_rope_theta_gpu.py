"""The RoPE base theta is an argument of the tables (wan_rope3d_tables): the
forward and backward against the fp64 oracle at theta = 500 (fast angles in
every band) and 1e6 (slow ones), every row."""
import pytest

import long_sequence_attention_02_b300 as wan
from long_sequence_attention_02_b300 import synth
from oracle import ref
from tests._util import bits, compare, dev_to_f64, f64, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _inputs(grid, H, seed, streams):
    L = grid[0] * grid[1] * grid[2]
    return [bits(seed, s, (1, L, H, 128)) for s in streams]


@pytest.mark.parametrize("theta", [500.0, 1.0e6])
def test_forward_at_other_rope_bases(theta):
    grid, H = (4, 16, 16), 2
    qb, kb, vb = _inputs(grid, H, 71, (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V))
    o, lse = wan.attention_forward(to_dev(qb), to_dev(kb), to_dev(vb), grid, theta=theta)
    wan.check(wan.wan_get_device_status())
    o_ref, lse_ref = ref.self_attention_fwd(f64(qb), f64(kb), f64(vb), grid, theta=theta)
    compare(dev_to_f64(o), o_ref, f"O (theta {theta:g})")
    compare(dev_to_f64(lse), lse_ref, f"LSE (theta {theta:g})")


def test_backward_at_another_rope_base():
    grid, H, theta = (4, 8, 8), 2, 500.0
    qb, kb, vb, dob = _inputs(grid, H, 72, (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V, synth.STREAM_DO))
    q, k, v, do = (to_dev(x) for x in (qb, kb, vb, dob))
    tables = wan.rope_tables(grid, theta)
    o, lse = wan.attention_forward(q, k, v, grid, tables=tables)
    dq, dk, dv = wan.attention_backward(q, k, v, o, lse, do, grid, tables=tables)
    wan.check(wan.wan_get_device_status())
    dq_r, dk_r, dv_r = ref.self_attention_bwd(f64(qb), f64(kb), f64(vb), f64(dob), grid, theta=theta)
    compare(dev_to_f64(dq), dq_r, "dQ (theta 500)")
    compare(dev_to_f64(dk), dk_r, "dK (theta 500)")
    compare(dev_to_f64(dv), dv_r, "dV (theta 500)")
