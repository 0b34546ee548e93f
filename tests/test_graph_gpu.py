"""wan_attn_fwd launches work only (no allocation, no synchronisation), so a
call captured once in a CUDA graph replays the same computation on the live
buffers: bit for bit a direct call, also after the inputs are rewritten."""
import math

import pytest

import long_sequence_attention_02_b300 as wan
from long_sequence_attention_02_b300 import synth
from tests._util import bits, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_captured_forward_replays_a_direct_call():
    grid, B, H, d = (3, 7, 9), 2, 3, 128
    L = grid[0] * grid[1] * grid[2]
    shape = (B, L, H, d)
    q, k, v = (to_dev(bits(81, s, shape)) for s in (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V))
    tab = wan.rope_tables(grid)
    wsb = wan.wan_attn_workspace_size(wan.WAN_OP_FWD, B, grid, H, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    o, lse = torch.empty_like(q), torch.empty(B, H, L, device="cuda")

    def call():  # on torch's current stream (the capture stream inside the graph)
        wan.check(wan.wan_attn_fwd(q, k, v, o, lse, B, grid, H, d, tab, 1 / math.sqrt(d), ws, wsb))

    call()
    torch.cuda.synchronize()
    o_direct, lse_direct = o.clone(), lse.clone()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    o.zero_()
    lse.zero_()
    graph.replay()
    torch.cuda.synchronize()
    wan.check(wan.wan_get_device_status())
    assert torch.equal(o, o_direct) and torch.equal(lse, lse_direct)

    # new inputs in the same buffers: the replay computes on them
    for t, s in zip((q, k, v), (synth.STREAM_K, synth.STREAM_V, synth.STREAM_Q)):
        t.copy_(to_dev(bits(82, s, shape)))
    call()
    torch.cuda.synchronize()
    o_direct, lse_direct = o.clone(), lse.clone()
    o.zero_()
    graph.replay()
    torch.cuda.synchronize()
    wan.check(wan.wan_get_device_status())
    assert torch.equal(o, o_direct) and torch.equal(lse, lse_direct)
