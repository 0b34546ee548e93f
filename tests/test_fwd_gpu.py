"""Forward parity: CUDA path (through the C ABI) against the fp64 oracle.

Small grids compare every row; the full-size workloads compare 4096 seeded
(b, h, row) samples that the oracle computes one head at a time.
"""
import math

import numpy as np
import pytest

import long_sequence_attention_02_b300 as wan
from long_sequence_attention_02_b300 import synth
from oracle import ref
from tests._util import MAX_ABS, REL_L2, bits, bf16_round, compare, dev_to_f64, f64, rows_whose_reference_moves, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _self_inputs(B, grid, H, seed):
    L = grid[0] * grid[1] * grid[2]
    shape = (B, L, H, 128)
    return (bits(seed, synth.STREAM_Q, shape), bits(seed, synth.STREAM_K, shape),
            bits(seed, synth.STREAM_V, shape))


def _run_self(qb, kb, vb, grid, canary=True):
    B, L, H, d = qb.shape
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    tables = wan.rope_tables(grid)
    n = B * L * H * d
    pad = 4096
    o_buf = torch.full((n + pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse_buf = torch.full((B * H * L + pad,), 12345.0, dtype=torch.float32, device="cuda")
    o = o_buf[:n].view(B, L, H, d)
    lse = lse_buf[: B * H * L].view(B, H, L)
    ws_bytes = wan.wan_attn_workspace_size(wan.WAN_OP_FWD, B, grid, H, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    wan.check(wan.wan_attn_fwd(q, k, v, o, lse, B, grid, H, d, tables, 1 / math.sqrt(d), ws, ws_bytes))
    wan.check(wan.wan_get_device_status())
    if canary:
        assert torch.isnan(o_buf[n:].float()).all(), "write past the end of O"
        assert (lse_buf[B * H * L:] == 12345.0).all(), "write past the end of LSE"
    return dev_to_f64(o), dev_to_f64(lse)


def test_rope_tables_match_oracle_angles():
    grid = (21, 45, 80)
    t = wan.rope_tables(grid).cpu().numpy()
    F, Hp, Wp = grid
    ang = ref.rope_angles(F, Hp, Wp, 128)
    tt, hh, ww = ref.token_coords(F, Hp, Wp)
    got_t = t[: F * 22 * 2].reshape(F, 22, 2)
    got_h = t[F * 44: F * 44 + Hp * 42].reshape(Hp, 21, 2)
    got_w = t[F * 44 + Hp * 42:].reshape(Wp, 21, 2)
    # token (t, 0, 0) carries the t angles, (0, h, 0) the h angles, (0, 0, w) the w angles
    for f in range(F):
        a = ang[f * Hp * Wp, :22]
        np.testing.assert_array_equal(got_t[f, :, 0], np.cos(a).astype(np.float32))
        np.testing.assert_array_equal(got_t[f, :, 1], np.sin(a).astype(np.float32))
    for h in range(Hp):
        a = ang[h * Wp, 22:43]
        np.testing.assert_allclose(got_h[h, :, 0], np.cos(a), atol=6e-8)
        np.testing.assert_allclose(got_h[h, :, 1], np.sin(a), atol=6e-8)
    for w in range(Wp):
        a = ang[w, 43:]
        np.testing.assert_allclose(got_w[w, :, 0], np.cos(a), atol=6e-8)
        np.testing.assert_allclose(got_w[w, :, 1], np.sin(a), atol=6e-8)


SMALL_GRIDS = [
    (1, (3, 8, 8), 2),     # the tiny workload: 192 tokens
    (1, (2, 4, 4), 1),     # 32 tokens: one partial key tile, one partial query tile
    (2, (4, 8, 8), 3),     # 256 tokens: exactly one CTA of query rows
    (1, (3, 7, 9), 2),     # 189: ragged everywhere
    (1, (8, 16, 16), 2),   # 2048: many key tiles
    (2, (5, 13, 17), 1),   # 1105: ragged, odd extents
    (1, (1, 1, 1), 1),     # a single token
    (3, (1, 1, 129), 5),   # 129 tokens in a 1 x 1 x W grid (t and h angles all 0), B = 3, H = 5
    (1, (257, 1, 1), 2),   # 257 tokens along t only: one row past a 256-row query pair
]


@pytest.mark.parametrize("B,grid,H", SMALL_GRIDS)
def test_self_attention_every_row(B, grid, H):
    qb, kb, vb = _self_inputs(B, grid, H, seed=11)
    o, lse = _run_self(qb, kb, vb, grid)
    o_ref, lse_ref = ref.self_attention_fwd(f64(qb), f64(kb), f64(vb), grid)
    compare(o, o_ref, "O")
    compare(lse, lse_ref, "LSE")


def test_self_attention_zero_queries_give_mean_values():
    B, grid, H = 1, (4, 8, 8), 2
    qb, kb, vb = _self_inputs(B, grid, H, seed=3)
    qb[:] = 0
    o, lse = _run_self(qb, kb, vb, grid)
    mean_v = f64(vb).mean(axis=1, keepdims=True)
    compare(o, np.broadcast_to(mean_v, o.shape), "O(Q=0)")
    np.testing.assert_allclose(lse, math.log(256), atol=1e-5)


def test_self_attention_one_hot_logit():
    B, grid, H = 1, (2, 8, 16), 1
    L = 256
    qb, kb, vb = _self_inputs(B, grid, H, seed=5)
    rng = np.random.default_rng(0)
    u = rng.standard_normal(128)
    u *= 30.0 / np.linalg.norm(u)
    # bf16 bits of u (truncated): the logit of token i0 with itself is ~80,
    # the others are ~N(0, 2.7^2), so row i0 puts all its weight on V[i0]
    ub = (u.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    i0 = 77
    qb[0, i0, 0] = ub
    kb[0, i0, 0] = ub
    o, lse = _run_self(qb, kb, vb, grid)
    o_ref, lse_ref = ref.self_attention_fwd(f64(qb), f64(kb), f64(vb), grid)
    compare(o, o_ref, "O")
    compare(lse, lse_ref, "LSE")
    assert np.abs(o[0, i0, 0] - f64(vb)[0, i0, 0]).max() < 0.05


def test_self_attention_reference_moves():
    """Keys of the first 8 of 16 key tiles scaled by 1/8 and the rest by 2
    (exact in bf16). An item that starts in the small half takes its softmax
    reference there, and the first large tile's row sums exceed the bound, so
    those rows rescale O and l and recompute the tile."""
    B, grid, H = 1, (8, 16, 16), 2
    L = 2048
    qb, kb, vb = _self_inputs(B, grid, H, seed=13)
    kf = f64(kb) * np.where(np.arange(L) // 128 < 8, 0.125, 2.0)[None, :, None, None]
    kb = bf16_round(kf)
    assert np.array_equal(f64(kb), kf)
    assert rows_whose_reference_moves(f64(qb), kf, grid) > 1000
    o, lse = _run_self(qb, kb, vb, grid)
    o_ref, lse_ref = ref.self_attention_fwd(f64(qb), kf, f64(vb), grid)
    compare(o, o_ref, "O")
    compare(lse, lse_ref, "LSE")


def _run_cross(qb, kb, vb, lens, grid):
    B, Lq, H, d = qb.shape
    Lk = kb.shape[1]
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    kv = None if lens is None else torch.from_numpy(np.asarray(lens, dtype=np.int32)).cuda()
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Lq, dtype=torch.float32, device="cuda")
    wan.check(wan.wan_xattn_fwd(q, k, v, kv, Lk, o, lse, B, grid, H, d, 1 / math.sqrt(d)))
    wan.check(wan.wan_get_device_status())
    return dev_to_f64(o), dev_to_f64(lse)


@pytest.mark.parametrize("Lk", [1, 16, 127, 128, 129, 512])
def test_cross_attention_every_row(Lk):
    grid, B, H = (3, 7, 9), 3, 2
    Lq = 189
    qb = bits(21, synth.STREAM_Q, (B, Lq, H, 128))
    kb = bits(21, synth.STREAM_K, (B, Lk, H, 128))
    vb = bits(21, synth.STREAM_V, (B, Lk, H, 128))
    lens = np.array([Lk, max(1, Lk // 2), 0], dtype=np.int32)
    o, lse = _run_cross(qb, kb, vb, lens, grid)
    o_ref, lse_ref = ref.cross_attention_fwd(f64(qb), f64(kb), f64(vb), lens)
    compare(o, o_ref, "O")
    compare(lse, lse_ref, "LSE")
    o2, lse2 = _run_cross(qb, kb, vb, None, grid)
    o2_ref, lse2_ref = ref.cross_attention_fwd(f64(qb), f64(kb), f64(vb), [Lk] * B)
    compare(o2, o2_ref, "O (no lens)")
    compare(lse2, lse2_ref, "LSE (no lens)")


def test_cross_attention_padding_is_ignored_bitwise():
    grid, B, H, Lk = (2, 8, 16), 2, 2, 300
    qb = bits(4, synth.STREAM_Q, (B, 256, H, 128))
    kb = bits(4, synth.STREAM_K, (B, Lk, H, 128))
    vb = bits(4, synth.STREAM_V, (B, Lk, H, 128))
    lens = np.array([130, 257], dtype=np.int32)
    o1, l1 = _run_cross(qb, kb, vb, lens, grid)
    kb2, vb2 = kb.copy(), vb.copy()
    kb2[0, 130:] = 0x4700  # 32768.0
    vb2[0, 130:] = 0xC2F6  # -123.0
    kb2[1, 257:] = 0x4700
    o2, l2 = _run_cross(qb, kb2, vb2, lens, grid)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_cross_attention_out_of_range_lengths_are_clamped():
    grid, B, H, Lk = (1, 4, 8), 2, 1, 40
    qb = bits(8, synth.STREAM_Q, (B, 32, H, 128))
    kb = bits(8, synth.STREAM_K, (B, Lk, H, 128))
    vb = bits(8, synth.STREAM_V, (B, Lk, H, 128))
    o, lse = _run_cross(qb, kb, vb, np.array([-5, 1000], dtype=np.int32), grid)
    o_ref, lse_ref = ref.cross_attention_fwd(f64(qb), f64(kb), f64(vb), [0, Lk])
    compare(o, o_ref, "O")
    compare(lse, lse_ref, "LSE")


def test_non_default_stream_and_lse_optional():
    B, grid, H = 1, (4, 8, 8), 2
    qb, kb, vb = _self_inputs(B, grid, H, seed=2)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
        o, lse = wan.attention_forward(q, k, v, grid, lse=False, stream=s)
    s.synchronize()
    assert lse is None
    o_ref, _ = ref.self_attention_fwd(f64(qb), f64(kb), f64(vb), grid)
    compare(dev_to_f64(o), o_ref, "O")


# ---------------------------------------------------------------------------
# Full-size workloads, 4096 sampled rows


def _sample_rows(seed, B, H, L, n=4096):
    rng = np.random.default_rng(seed)
    flat = rng.choice(B * H * L, size=min(n, B * H * L), replace=False)
    b = flat // (H * L)
    h = (flat // L) % H
    i = flat % L
    return b, h, i


def _head(bits_full, b, h):
    return f64(bits_full[b, :, h, :])


@pytest.mark.parametrize("name", ["wan1.3b_480p_self_fwd", "wan14b_720p_self_fwd"])
def test_self_attention_full_size_sampled(name):
    from long_sequence_attention_02_b300.workloads import WORKLOADS

    w = WORKLOADS[name]
    B, L, H, grid = w.B, w.L, w.H, w.grid
    qb, kb, vb = _self_inputs(B, grid, H, seed=0)
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    o, lse = wan.attention_forward(q, k, v, grid)
    wan.check(wan.wan_get_device_status())
    del q, k, v
    bs, hs, is_ = _sample_rows(1, B, H, L)
    o_rows = dev_to_f64(o[bs, is_, hs])
    lse_rows = dev_to_f64(lse[bs, hs, is_])
    ref_o = np.zeros_like(o_rows)
    ref_l = np.zeros_like(lse_rows)
    for bh in sorted(set(zip(bs.tolist(), hs.tolist()))):
        sel = np.where((bs == bh[0]) & (hs == bh[1]))[0]
        qrows = f64(qb[bh[0], is_[sel], bh[1], :])
        ro, rl = ref.self_attention_fwd_rows(qrows, is_[sel], _head(kb, *bh), _head(vb, *bh), grid)
        ref_o[sel], ref_l[sel] = ro, rl
    compare(o_rows, ref_o, f"{name} O")
    compare(lse_rows, ref_l, f"{name} LSE")


def test_cross_attention_full_size_sampled():
    from long_sequence_attention_02_b300.workloads import WORKLOADS

    w = WORKLOADS["wan14b_720p_cross_fwd"]
    B, Lq, H, Lk = w.B, w.L, w.H, w.Lk
    qb = bits(0, synth.STREAM_Q, (B, Lq, H, 128))
    kb = bits(0, synth.STREAM_K, (B, Lk, H, 128))
    vb = bits(0, synth.STREAM_V, (B, Lk, H, 128))
    lens = synth.kv_lens(0, B)
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    kv = torch.from_numpy(lens).cuda()
    o, lse = wan.cross_attention_forward(q, k, v, kv, w.grid)
    wan.check(wan.wan_get_device_status())
    bs, hs, is_ = _sample_rows(2, B, H, Lq)
    o_rows = dev_to_f64(o[bs, is_, hs])
    lse_rows = dev_to_f64(lse[bs, hs, is_])
    ref_o = np.zeros_like(o_rows)
    ref_l = np.zeros_like(lse_rows)
    for bh in sorted(set(zip(bs.tolist(), hs.tolist()))):
        sel = np.where((bs == bh[0]) & (hs == bh[1]))[0]
        ro, rl = ref.softmax_attention(f64(qb[bh[0], is_[sel], bh[1], :]), _head(kb, *bh), _head(vb, *bh),
                                       1 / math.sqrt(128), lens[bh[0]])
        ref_o[sel], ref_l[sel] = ro, rl
    compare(o_rows, ref_o, "xattn O")
    compare(lse_rows, ref_l, "xattn LSE")
