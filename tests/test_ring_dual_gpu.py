"""Ring-attention steps and decoupled (text + image) cross-attention on the
GPU, through the C ABI, against the fp64 oracle."""
import math

import numpy as np
import pytest

import long_sequence_attention_02_b300 as wan
from long_sequence_attention_02_b300 import synth
from oracle import ref
from tests._util import bits, compare, dev_to_f64, f64, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _ring(qb, kb, vb, grid, q_start, q_len, bounds):
    """Run Ring steps for queries [q_start, q_start+q_len) over the K/V chunks
    given by `bounds`; returns O and LSE of the query chunk."""
    B, L, H, d = qb.shape
    q = to_dev(np.ascontiguousarray(qb[:, q_start:q_start + q_len]))
    tables = wan.rope_tables(grid)
    o = torch.empty(B, q_len, H, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, q_len, dtype=torch.float32, device="cuda")
    ws_bytes = wan.wan_attn_workspace_size(wan.WAN_OP_FWD, B, grid, H, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    for n, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
        k = to_dev(np.ascontiguousarray(kb[:, a:b]))
        v = to_dev(np.ascontiguousarray(vb[:, a:b]))
        wan.check(wan.wan_attn_fwd_ring_step(q, k, v, o, lse, B, grid, H, d, tables, 1 / math.sqrt(d), q_start,
                                             q_len, a, b - a, 1 if n > 0 else 0, ws, ws_bytes), "ring step")
    wan.check(wan.wan_get_device_status())
    return dev_to_f64(o), dev_to_f64(lse)


RING_CASES = [
    (2, (3, 7, 9), 2, 17, 150, [0, 60, 61, 189]),          # ragged chunks, a 1-key chunk
    (1, (4, 16, 16), 2, 300, 700, [0, 256, 756, 1024]),    # several query and key tiles per step
    (1, (2, 8, 16), 1, 0, 256, [0, 256]),                   # one step over everything
]


@pytest.mark.parametrize("B,grid,H,q_start,q_len,bounds", RING_CASES)
def test_ring_steps_match_full_attention(B, grid, H, q_start, q_len, bounds):
    L = grid[0] * grid[1] * grid[2]
    shape = (B, L, H, 128)
    qb, kb, vb = (bits(31, s, shape) for s in (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V))
    o, lse = _ring(qb, kb, vb, grid, q_start, q_len, bounds)
    o_ref, lse_ref = ref.self_attention_fwd(f64(qb), f64(kb), f64(vb), grid)
    compare(o, o_ref[:, q_start:q_start + q_len], "O (ring)")
    compare(lse, lse_ref[:, :, q_start:q_start + q_len], "LSE (ring)")


def test_ring_single_step_equals_forward_bitwise():
    B, grid, H = 1, (4, 8, 8), 2
    L = 256
    shape = (B, L, H, 128)
    qb, kb, vb = (bits(32, s, shape) for s in (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V))
    o_r, lse_r = _ring(qb, kb, vb, grid, 0, L, [0, L])
    o_f, lse_f = wan.attention_forward(to_dev(qb), to_dev(kb), to_dev(vb), grid)
    wan.check(wan.wan_get_device_status())
    assert np.array_equal(o_r, dev_to_f64(o_f)) and np.array_equal(lse_r, dev_to_f64(lse_f))


def test_ring_step_chunk_matches_oracle_chunk():
    # one non-accumulating step is the oracle's chunk attention at grid positions
    B, grid, H = 1, (3, 8, 8), 1
    L = 192
    shape = (B, L, H, 128)
    qb, kb, vb = (bits(33, s, shape) for s in (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V))
    o, lse = _ring(qb, kb, vb, grid, 64, 100, [130, 192])
    o_ref, lse_ref = ref.self_attention_fwd_chunk(f64(qb[0, 64:164, 0]), 64, f64(kb[0, 130:192, 0]),
                                                  f64(vb[0, 130:192, 0]), 130, grid)
    compare(o[0, :, 0], o_ref, "O (chunk)")
    compare(lse[0, 0], lse_ref, "LSE (chunk)")


def test_ring_step_rejects_bad_ranges():
    B, grid, H = 1, (2, 4, 4), 1
    t = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(64, dtype=torch.float32, device="cuda")
    tables = wan.rope_tables(grid)
    ws = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    for qs, ql, ks, kl, acc in [(-1, 4, 0, 4, 0), (0, 33, 0, 4, 0), (0, 4, 30, 4, 0), (0, 0, 0, 4, 0),
                                (0, 4, 0, 4, 2)]:
        rc = wan.wan_attn_fwd_ring_step(t, t, t, t, lse, B, grid, H, 128, tables, 0.088, qs, ql, ks, kl, acc, ws,
                                        ws.numel())
        assert rc == wan.WAN_ERR_INVALID, (qs, ql, ks, kl, acc)


@pytest.mark.parametrize("lens_txt,Lk_txt,lens_img,Lk_img", [
    ([77, 30, 0], 77, None, 257),
    ([77, 1, 64], 77, [257, 0, 100], 257),
    (None, 512, [130, 131, 129], 160),
])
def test_decoupled_cross_attention(lens_txt, Lk_txt, lens_img, Lk_img):
    grid, B, H = (3, 7, 9), 3, 2
    Lq = 189
    qb = bits(41, synth.STREAM_Q, (B, Lq, H, 128))
    ktb = bits(41, synth.STREAM_K, (B, Lk_txt, H, 128))
    vtb = bits(41, synth.STREAM_V, (B, Lk_txt, H, 128))
    kib = bits(42, synth.STREAM_K, (B, Lk_img, H, 128))
    vib = bits(42, synth.STREAM_V, (B, Lk_img, H, 128))
    dev_lens = lambda x: None if x is None else torch.tensor(x, dtype=torch.int32, device="cuda")  # noqa: E731
    q = to_dev(qb)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Lq, dtype=torch.float32, device="cuda")
    wan.check(wan.wan_xattn_fwd_dual(q, to_dev(ktb), to_dev(vtb), dev_lens(lens_txt), Lk_txt, to_dev(kib),
                                     to_dev(vib), dev_lens(lens_img), Lk_img, o, lse, B, grid, H, 128,
                                     1 / math.sqrt(128)), "dual")
    wan.check(wan.wan_get_device_status())
    lt = [Lk_txt] * B if lens_txt is None else lens_txt
    li = [Lk_img] * B if lens_img is None else lens_img
    o_ref, lse_ref = ref.decoupled_cross_attention_fwd(f64(qb), f64(ktb), f64(vtb), lt, f64(kib), f64(vib), li)
    compare(dev_to_f64(o), o_ref, "O (text + image)")
    compare(dev_to_f64(lse), lse_ref, "LSE (text path)")


@pytest.mark.parametrize("lens_txt,lens_img", [([300, 512], [257, 129]), ([512, 17], [0, 200])])
def test_decoupled_cross_attention_many_items_every_row(lens_txt, lens_img):
    """More work items than CTAs (2 batch items x 20 heads x 24 pairs of
    query tiles = 960 items on 148 SMs): each CTA walks about six items, so
    every Q buffer, O staging area and old-O load of the summed path is
    reused several times; every row is compared. The second case has a batch
    item with no image key (its items are skipped by the summed path)."""
    grid, B, H = (6, 25, 40), 2, 20
    Lq, Lt, Li = 6000, 512, 257
    qb = bits(43, synth.STREAM_Q, (B, Lq, H, 128))
    ktb, vtb = bits(43, synth.STREAM_K, (B, Lt, H, 128)), bits(43, synth.STREAM_V, (B, Lt, H, 128))
    kib, vib = bits(44, synth.STREAM_K, (B, Li, H, 128)), bits(44, synth.STREAM_V, (B, Li, H, 128))
    q = to_dev(qb)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Lq, dtype=torch.float32, device="cuda")
    lt = torch.tensor(lens_txt, dtype=torch.int32, device="cuda")
    li = torch.tensor(lens_img, dtype=torch.int32, device="cuda")
    wan.check(wan.wan_xattn_fwd_dual(q, to_dev(ktb), to_dev(vtb), lt, Lt, to_dev(kib), to_dev(vib), li, Li, o, lse,
                                     B, grid, H, 128, 1 / math.sqrt(128)), "dual")
    wan.check(wan.wan_get_device_status())
    o_ref, lse_ref = ref.decoupled_cross_attention_fwd(f64(qb), f64(ktb), f64(vtb), lens_txt, f64(kib), f64(vib),
                                                       lens_img)
    compare(dev_to_f64(o), o_ref, "O (text + image, many items)")
    compare(dev_to_f64(lse), lse_ref, "LSE (text path, many items)")


# ---------------------------------------------------------------------------
# Full-size cases on 4096 seeded sampled rows


def _sample(seed, B, H, L, n=4096):
    rng = np.random.default_rng(seed)
    flat = rng.choice(B * H * L, size=min(n, B * H * L), replace=False)
    return flat // (H * L), (flat // L) % H, flat % L


def test_ring_steps_480p_sampled():
    """The 32,760-token, 12-head grid: the middle third of the queries over
    three K/V chunks (one of them ragged), against the oracle's full rows."""
    from long_sequence_attention_02_b300.workloads import WORKLOADS

    w = WORKLOADS["wan1.3b_480p_self_fwd"]
    B, L, H, grid = w.B, w.L, w.H, w.grid
    shape = (B, L, H, 128)
    qb, kb, vb = (bits(5, s, shape) for s in (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V))
    q_start, q_len = 10920, 10920
    o, lse = _ring(qb, kb, vb, grid, q_start, q_len, [0, 12000, 12001, L])
    bs, hs, is_ = _sample(6, B, H, q_len)
    o_rows, lse_rows = o[bs, is_, hs], lse[bs, hs, is_]
    r_o, r_l = np.zeros_like(o_rows), np.zeros_like(lse_rows)
    for bh in sorted(set(zip(bs.tolist(), hs.tolist()))):
        sel = np.where((bs == bh[0]) & (hs == bh[1]))[0]
        tok = q_start + is_[sel]
        r_o[sel], r_l[sel] = ref.self_attention_fwd_rows(f64(qb[bh[0], tok, bh[1]]), tok, f64(kb[bh[0], :, bh[1]]),
                                                         f64(vb[bh[0], :, bh[1]]), grid)
    compare(o_rows, r_o, "ring O (480p)")
    compare(lse_rows, r_l, "ring LSE (480p)")


def test_decoupled_cross_attention_full_size_sampled():
    """2 x 75,600 video queries, 40 heads; 512 text keys (seeded lengths) and
    257 image keys."""
    from long_sequence_attention_02_b300.workloads import WORKLOADS

    w = WORKLOADS["wan14b_720p_cross_fwd"]
    B, Lq, H, Lt, Li = w.B, w.L, w.H, w.Lk, 257
    qb = bits(7, synth.STREAM_Q, (B, Lq, H, 128))
    ktb, vtb = bits(7, synth.STREAM_K, (B, Lt, H, 128)), bits(7, synth.STREAM_V, (B, Lt, H, 128))
    kib, vib = bits(8, synth.STREAM_K, (B, Li, H, 128)), bits(8, synth.STREAM_V, (B, Li, H, 128))
    lens = synth.kv_lens(7, B)
    q = to_dev(qb)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Lq, dtype=torch.float32, device="cuda")
    wan.check(wan.wan_xattn_fwd_dual(q, to_dev(ktb), to_dev(vtb), torch.from_numpy(lens).cuda(), Lt, to_dev(kib),
                                     to_dev(vib), None, Li, o, lse, B, w.grid, H, 128, 1 / math.sqrt(128)), "dual")
    wan.check(wan.wan_get_device_status())
    bs, hs, is_ = _sample(9, B, H, Lq)
    o_rows, lse_rows = dev_to_f64(o[bs, is_, hs]), dev_to_f64(lse[bs, hs, is_])
    r_o, r_l = np.zeros_like(o_rows), np.zeros_like(lse_rows)
    sc = 1 / math.sqrt(128)
    for bh in sorted(set(zip(bs.tolist(), hs.tolist()))):
        b, h = bh
        sel = np.where((bs == b) & (hs == h))[0]
        qr = f64(qb[b, is_[sel], h])
        o1, l1 = ref.softmax_attention(qr, f64(ktb[b, :, h]), f64(vtb[b, :, h]), sc, lens[b])
        o2, _ = ref.softmax_attention(qr, f64(kib[b, :, h]), f64(vib[b, :, h]), sc, Li)
        r_o[sel], r_l[sel] = o1 + o2, l1
    compare(o_rows, r_o, "dual O (full size)")
    compare(lse_rows, r_l, "dual LSE (full size)")
