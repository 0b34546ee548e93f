"""Backward parity: dQ, dK, dV of the CUDA path against the fp64 oracle.

The CUDA backward consumes the CUDA forward's O and LSE (as a training step
does); the oracle recomputes everything from Q, K, V and dO alone.
"""
import math

import numpy as np
import pytest

import long_sequence_attention_02_b300 as wan
from long_sequence_attention_02_b300 import synth
from oracle import ref
from tests._util import bits, compare, dev_to_f64, f64, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _inputs(B, grid, H, seed):
    L = grid[0] * grid[1] * grid[2]
    shape = (B, L, H, 128)
    return [bits(seed, s, shape) for s in (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V, synth.STREAM_DO)]


def _run(qb, kb, vb, dob, grid):
    q, k, v, do = (to_dev(x) for x in (qb, kb, vb, dob))
    tables = wan.rope_tables(grid)
    o, lse = wan.attention_forward(q, k, v, grid, tables=tables)
    dq, dk, dv = wan.attention_backward(q, k, v, o, lse, do, grid, tables=tables)
    wan.check(wan.wan_get_device_status())
    return o, lse, dq, dk, dv


SMALL = [
    (1, (2, 4, 4), 1),     # 32 tokens: one partial tile of keys and of queries
    (1, (3, 8, 8), 2),     # the tiny workload
    (1, (3, 7, 9), 2),     # 189: ragged
    (2, (4, 8, 8), 1),     # 256: two full tiles, B = 2
    (1, (8, 16, 16), 2),   # 2048: many tiles both ways
    (2, (5, 13, 17), 1),   # 1105: ragged, odd extents
    (1, (2, 4, 5), 72),    # 40 tokens, 72 heads: the row pass takes its heads in two passes (64 + 8)
    (1, (1, 1, 1), 2),     # a single token
    (3, (1, 1, 129), 3),   # 129 tokens in a 1 x 1 x W grid, B = 3: one row past a key tile
]


@pytest.mark.parametrize("B,grid,H", SMALL)
def test_backward_every_row(B, grid, H):
    qb, kb, vb, dob = _inputs(B, grid, H, seed=13)
    _, _, dq, dk, dv = _run(qb, kb, vb, dob, grid)
    dq_r, dk_r, dv_r = ref.self_attention_bwd(f64(qb), f64(kb), f64(vb), f64(dob), grid)
    compare(dev_to_f64(dq), dq_r, "dQ")
    compare(dev_to_f64(dk), dk_r, "dK")
    compare(dev_to_f64(dv), dv_r, "dV")


def test_backward_sum_identities():
    B, grid, H = 1, (4, 16, 16), 3
    qb, kb, vb, dob = _inputs(B, grid, H, seed=5)
    _, _, dq, dk, dv = _run(qb, kb, vb, dob, grid)
    # softmax rows sum to one: sum_j dV_j = sum_i dO_i
    got = dev_to_f64(dv).sum(axis=1)
    want = f64(dob).sum(axis=1)
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 5e-3
    # rows of dS sum to zero: the rotated key gradients sum to zero
    ang = ref.rope_angles(*grid, 128)
    dkf = dev_to_f64(dk)
    for h in range(H):
        dkr = ref.rope_rotate(dkf[0, :, h], ang)
        assert np.abs(dkr.sum(axis=0)).max() < 2e-2 * np.abs(dkr).sum(axis=0).max() + 1e-3


def test_backward_exhaustive_16x32x32():
    B, grid, H = 1, (16, 32, 32), 1
    qb, kb, vb, dob = _inputs(B, grid, H, seed=17)
    _, _, dq, dk, dv = _run(qb, kb, vb, dob, grid)
    dq_r, dk_r, dv_r = ref.self_attention_bwd(f64(qb), f64(kb), f64(vb), f64(dob), grid)
    compare(dev_to_f64(dq), dq_r, "dQ")
    compare(dev_to_f64(dk), dk_r, "dK")
    compare(dev_to_f64(dv), dv_r, "dV")


@pytest.fixture(scope="module")
def full_step():
    """The 64x64x64 grid, H = 12 training step (forward, then backward on the
    forward's O and LSE), run once for the full-size tests below."""
    from long_sequence_attention_02_b300.workloads import WORKLOADS

    w = WORKLOADS["train_64x64x64_fwd_bwd"]
    qb, kb, vb, dob = _inputs(w.B, w.grid, w.H, seed=0)
    out = _run(qb, kb, vb, dob, w.grid)
    yield w, (qb, kb, vb, dob), out
    del out
    torch.cuda.empty_cache()


def test_training_step_full_size_sampled(full_step):
    """O, LSE and dQ on 4096 sampled rows against the oracle; dK and dV
    through the exact sum identities on every head."""
    w, (qb, kb, vb, dob), (o, lse, dq, dk, dv) = full_step
    B, L, H, grid = w.B, w.L, w.H, w.grid
    rng = np.random.default_rng(3)
    flat = rng.choice(B * H * L, size=4096, replace=False)
    bs, hs, is_ = flat // (H * L), (flat // L) % H, flat % L
    o_rows = dev_to_f64(o[bs, is_, hs])
    lse_rows = dev_to_f64(lse[bs, hs, is_])
    dq_rows = dev_to_f64(dq[bs, is_, hs])
    r_o, r_l, r_dq = np.zeros_like(o_rows), np.zeros_like(lse_rows), np.zeros_like(dq_rows)
    for bh in sorted(set(zip(bs.tolist(), hs.tolist()))):
        sel = np.where((bs == bh[0]) & (hs == bh[1]))[0]
        kh, vh = f64(kb[bh[0], :, bh[1]]), f64(vb[bh[0], :, bh[1]])
        qrows, dorows = f64(qb[bh[0], is_[sel], bh[1]]), f64(dob[bh[0], is_[sel], bh[1]])
        r_o[sel], r_l[sel] = ref.self_attention_fwd_rows(qrows, is_[sel], kh, vh, grid)
        r_dq[sel] = ref.self_attention_bwd_dq_rows(qrows, dorows, is_[sel], kh, vh, grid, block=128)
    compare(o_rows, r_o, "O")
    compare(lse_rows, r_l, "LSE")
    compare(dq_rows, r_dq, "dQ")
    got = dv.float().sum(dim=1).double().cpu().numpy()
    want = f64(dob).sum(axis=1)
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 5e-3
    ang = ref.rope_angles(*grid, 128)
    for h in range(H):
        dkr = ref.rope_rotate(dev_to_f64(dk[0, :, h]), ang)
        col = dkr.sum(axis=0)
        assert np.abs(col).max() < 2e-2 * np.abs(dkr).sum(axis=0).max() + 1e-3


def test_training_step_full_size_key_rows(full_step):
    """dK and dV element by element on 4096 seeded key rows of one seeded head
    of the 262,144-token step. Each key row needs the LSE and D of all
    262,144 queries of its head, so the oracle runs that head's whole forward
    (in blocks of query rows spread over the host's cores) and then the
    selected key columns of the backward."""
    import os
    from concurrent.futures import ThreadPoolExecutor

    from tests._util import blas_single_threaded

    w, (qb, kb, vb, dob), (_, _, _, dk, dv) = full_step
    B, L, H, grid = w.B, w.L, w.H, w.grid
    rng = np.random.default_rng(29)
    b, h = int(rng.integers(B)), int(rng.integers(H))
    keys = np.sort(rng.choice(L, size=4096, replace=False))
    heads = [f64(x[b, :, h]) for x in (qb, kb, vb, dob)]
    workers = max(1, min(len(os.sched_getaffinity(0)), 32))
    with blas_single_threaded(), ThreadPoolExecutor(workers) as ex:
        dk_r, dv_r = ref.self_attention_bwd_dkdv_rows(*heads, keys, grid, block=64, row_map=ex.map)
    compare(dev_to_f64(dk[b, keys, h]), dk_r, f"dK (head {h}, 4096 key rows)")
    compare(dev_to_f64(dv[b, keys, h]), dv_r, f"dV (head {h}, 4096 key rows)")
