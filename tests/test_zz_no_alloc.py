"""The allocation-free forward entry point, wan_attn_fwd_noalloc.

Some callers cannot allocate device memory: a framework or plugin interface
that gives the library only its input and output buffers, a process whose
device memory is all held by another allocator, or a latency-critical caller
that cannot pay cudaMalloc's implicit device synchronisation. For them the
library keeps a fixed 64 MiB scratch array in device memory and
wan_attn_fwd_noalloc uses it in place of the caller's workspace.

These tests call it through the C ABI twice in a row, on different problems
(so the second call runs over the first call's leftovers in the shared
scratch), and compare each result with the workspace entry point
wan_attn_fwd on the same inputs, within the tolerances of the parity tests.
This file is collected last so that a run that stops at its first failure
has already run every other test.
"""
import math

import pytest

import long_sequence_attention_02_b300 as wan
from long_sequence_attention_02_b300 import synth
from tests._util import bits, compare, dev_to_f64, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _inputs(B, grid, H, seed):
    L = grid[0] * grid[1] * grid[2]
    shape = (B, L, H, 128)
    return [to_dev(bits(seed, s, shape)) for s in (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V)]


def _with_workspace(q, k, v, grid, tables):
    B, L, H, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, H, L, dtype=torch.float32, device=q.device)
    ws_bytes = wan.wan_attn_workspace_size(wan.WAN_OP_FWD, B, grid, H, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    wan.check(wan.wan_attn_fwd(q, k, v, o, lse, B, grid, H, d, tables, 1 / math.sqrt(d), ws, ws_bytes),
              "wan_attn_fwd")
    return o, lse


def _without_workspace(q, k, v, grid, tables):
    B, L, H, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty(B, H, L, dtype=torch.float32, device=q.device)
    wan.check(wan.wan_attn_fwd_noalloc(q, k, v, o, lse, B, grid, H, d, tables, 1 / math.sqrt(d)),
              "wan_attn_fwd_noalloc")
    return o, lse


def test_noalloc_forward_matches_workspace_forward_on_two_calls_in_a_row():
    cases = [
        (2, (4, 16, 16), 4, 41),   # 2 x 1024 tokens x 4 heads (8192 row-heads)
        (1, (5, 13, 17), 3, 42),   # 1105 tokens, ragged tiles, smaller than the first call
    ]
    for B, grid, H, seed in cases:
        q, k, v = _inputs(B, grid, H, seed)
        tables = wan.rope_tables(grid)
        o_ref, lse_ref = _with_workspace(q, k, v, grid, tables)
        o, lse = _without_workspace(q, k, v, grid, tables)
        assert wan.wan_get_device_status() == wan.WAN_OK
        compare(dev_to_f64(o), dev_to_f64(o_ref), f"O, grid {grid}")
        compare(dev_to_f64(lse), dev_to_f64(lse_ref), f"LSE, grid {grid}")


def test_noalloc_rejects_problems_beyond_the_scratch():
    assert wan.NOALLOC_MAX_ROW_HEADS == 262144
    grid, H = (64, 64, 64), 2  # 524,288 row-heads: twice the scratch
    small = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(16, dtype=torch.float32, device="cuda")
    tables = wan.rope_tables(grid)
    rc = wan.wan_attn_fwd_noalloc(small, small, small, small, lse, 1, grid, H, 128, tables, 0.088)
    assert rc == wan.WAN_ERR_INVALID
    # exactly at the limit is accepted by the size check (and runs)
    grid, H = (16, 32, 32), 16  # 16,384 tokens x 16 heads = 262,144 row-heads
    q, k, v = (torch.randn(1, 16384, H, 128, device="cuda").bfloat16() for _ in range(3))
    tables = wan.rope_tables(grid)
    o_ref, lse_ref = _with_workspace(q, k, v, grid, tables)
    o, lse = _without_workspace(q, k, v, grid, tables)
    assert wan.wan_get_device_status() == wan.WAN_OK
    compare(dev_to_f64(o), dev_to_f64(o_ref), "O at the size limit")
    compare(dev_to_f64(lse), dev_to_f64(lse_ref), "LSE at the size limit")


def test_noalloc_call_allocates_no_device_memory():
    """After a first call (which loads the kernels and looks up the scratch's
    address), a call on another problem leaves the device's free memory
    unchanged: the entry point itself allocates nothing."""
    grid_a, grid_b = (2, 8, 16), (3, 9, 10)
    qa, ka, va = _inputs(1, grid_a, 2, 45)
    qb, kb, vb = _inputs(1, grid_b, 3, 46)
    ta, tb = wan.rope_tables(grid_a), wan.rope_tables(grid_b)
    oa, lsea = torch.empty_like(qa), torch.empty(1, 2, 256, dtype=torch.float32, device="cuda")
    ob, lseb = torch.empty_like(qb), torch.empty(1, 3, 270, dtype=torch.float32, device="cuda")
    wan.check(wan.wan_attn_fwd_noalloc(qa, ka, va, oa, lsea, 1, grid_a, 2, 128, ta, 1 / math.sqrt(128)))
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    wan.check(wan.wan_attn_fwd_noalloc(qb, kb, vb, ob, lseb, 1, grid_b, 3, 128, tb, 1 / math.sqrt(128)))
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before, (free_before, free_after)
    assert wan.wan_get_device_status() == wan.WAN_OK
    o_ref, lse_ref = _with_workspace(qb, kb, vb, grid_b, tb)
    compare(dev_to_f64(ob), dev_to_f64(o_ref), "O (no-allocation check)")


def test_noalloc_on_a_side_stream_after_a_default_stream_call():
    """The entry point runs on the caller's stream: a call on a non-default
    stream, ordered after a call on the default stream that used the same
    scratch, gives the workspace path's result."""
    grid1, grid2 = (4, 8, 8), (2, 16, 16)
    q1, k1, v1 = _inputs(1, grid1, 4, 47)
    q2, k2, v2 = _inputs(2, grid2, 2, 48)
    t1, t2 = wan.rope_tables(grid1), wan.rope_tables(grid2)
    o1, lse1 = _without_workspace(q1, k1, v1, grid1, t1)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        o2 = torch.empty_like(q2)
        lse2 = torch.empty(2, 2, 512, dtype=torch.float32, device="cuda")
        wan.check(wan.wan_attn_fwd_noalloc(q2, k2, v2, o2, lse2, 2, grid2, 2, 128, t2, 1 / math.sqrt(128), side),
                  "wan_attn_fwd_noalloc (side stream)")
    side.synchronize()
    assert wan.wan_get_device_status() == wan.WAN_OK
    o1_ref, lse1_ref = _with_workspace(q1, k1, v1, grid1, t1)
    o2_ref, lse2_ref = _with_workspace(q2, k2, v2, grid2, t2)
    compare(dev_to_f64(o1), dev_to_f64(o1_ref), "O (default stream)")
    compare(dev_to_f64(o2), dev_to_f64(o2_ref), "O (side stream)")
    compare(dev_to_f64(lse2), dev_to_f64(lse2_ref), "LSE (side stream)")
