"""FP8 (e4m3) self-attention forward against the fp64 oracle.

Tolerance (no precision is stated for FP8, so it is derived here). e4m3 keeps 3 mantissa bits:
- Rounding to nearest gives a relative error of at most 2^-4, RMS u = 2^-4/sqrt(3) ~ 0.036, on
  every quantised element: Q_rot, K_rot, V (each scaled by its per-head amax) and P.
- Relative L2 of O. With N(0,1) inputs a logit sums 128 products, each with relative error
  ~sqrt(2) u. After the 1/sqrt(128) scale the logit error is ~1.4 u ~ 0.05, which is also the
  relative error it puts on p. O is a softmax average of nearly independent rows, so its relative
  error is about the per-term one: sqrt(0.05^2 + u^2 + u^2) ~ 0.07. Bound: 0.12.
- Max-abs of O. A row that attends to one key returns that key's V row, carrying up to 2^-4 from
  V's rounding and 2^-4 from P's (l sums the unrounded p). That is ~0.125 of the output's
  magnitude. Bound: 0.15 * max|O_ref|.
- LSE. It uses the fp32 probabilities, so it carries only the logit error: a p-weighted mean of
  errors whose RMS is ~0.05 for N(0,1) inputs. A row with one key (or one dominant key) keeps
  that error whole, with no averaging. Bound: 4 RMS = 0.2.
"""
import math

import numpy as np
import pytest

import long_sequence_attention_02_b300 as wan
from long_sequence_attention_02_b300 import synth
from oracle import ref
from tests._util import bf16_round, bits, compare, dev_to_f64, f64, rows_whose_reference_moves, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

FP8_REL_L2 = 0.12
FP8_MAX_ABS_FRACTION = 0.15  # of max |O_ref|
FP8_LSE_MAX_ABS = 0.2


def compare_fp8(o, o_ref, lse, lse_ref, name):
    compare(o, o_ref, f"O ({name})", max_abs=FP8_MAX_ABS_FRACTION * float(np.abs(o_ref).max()), rel_l2=FP8_REL_L2)
    # LSE is judged by its absolute error: with one key it is a single logit, which can be near 0.
    compare(lse, lse_ref, f"LSE ({name})", max_abs=FP8_LSE_MAX_ABS, rel_l2=float("inf"))


def _inputs(B, grid, H, seed):
    L = grid[0] * grid[1] * grid[2]
    shape = (B, L, H, 128)
    return [bits(seed, s, shape) for s in (synth.STREAM_Q, synth.STREAM_K, synth.STREAM_V)]


def _run(qb, kb, vb, grid):
    o, lse = wan.attention_forward_fp8(to_dev(qb), to_dev(kb), to_dev(vb), grid)
    wan.check(wan.wan_get_device_status())
    return dev_to_f64(o), dev_to_f64(lse)


@pytest.mark.parametrize("B,grid,H", [
    (1, (3, 8, 8), 2),     # 192 tokens
    (1, (3, 7, 9), 2),     # 189: ragged key and query tiles
    (2, (4, 8, 8), 3),     # 256, B = 2
    (1, (8, 16, 16), 2),   # 2048: many key tiles
    (1, (1, 1, 1), 1),     # a single token
])
def test_fp8_every_row(B, grid, H):
    qb, kb, vb = _inputs(B, grid, H, seed=51)
    o, lse = _run(qb, kb, vb, grid)
    o_ref, lse_ref = ref.self_attention_fwd(f64(qb), f64(kb), f64(vb), grid)
    compare_fp8(o, o_ref, lse, lse_ref, "fp8")


def test_fp8_zero_queries_give_mean_values():
    B, grid, H = 1, (4, 8, 8), 2
    qb, kb, vb = _inputs(B, grid, H, seed=52)
    qb[:] = 0
    o, lse = _run(qb, kb, vb, grid)
    mean_v = f64(vb).mean(axis=1, keepdims=True)
    mean_v = np.broadcast_to(mean_v, o.shape)
    compare(o, mean_v, "O(Q=0, fp8)", max_abs=FP8_MAX_ABS_FRACTION * float(np.abs(mean_v).max()), rel_l2=FP8_REL_L2)
    np.testing.assert_allclose(lse, math.log(256), atol=1e-4)


def test_fp8_reference_moves():
    """Keys of the first 8 of 16 key tiles scaled by 1/16 and the rest by 1.5:
    items that start in the small half move their softmax reference at the
    first large tile (row sums of P above the bound), rescale O and l and
    recompute that tile. The larger logits stay within the derived tolerance
    (logit error ~0.05 per unit of logit spread)."""
    B, grid, H = 1, (8, 16, 16), 2
    L = 2048
    qb, kb, vb = _inputs(B, grid, H, seed=54)
    kb = bf16_round(f64(kb) * np.where(np.arange(L) // 128 < 8, 0.0625, 1.5)[None, :, None, None])
    assert rows_whose_reference_moves(f64(qb), f64(kb), grid) > 300
    o, lse = _run(qb, kb, vb, grid)
    o_ref, lse_ref = ref.self_attention_fwd(f64(qb), f64(kb), f64(vb), grid)
    compare_fp8(o, o_ref, lse, lse_ref, "fp8, moving reference")


def test_fp8_tracks_the_bf16_path():
    B, grid, H = 1, (4, 16, 16), 2
    qb, kb, vb = _inputs(B, grid, H, seed=53)
    o8, lse8 = _run(qb, kb, vb, grid)
    o16, lse16 = wan.attention_forward(to_dev(qb), to_dev(kb), to_dev(vb), grid)
    compare_fp8(o8, dev_to_f64(o16), lse8, dev_to_f64(lse16), "fp8 vs bf16")


def test_fp8_full_size_sampled():
    """The 75,600-token, 40-head workload on 4096 seeded sampled rows."""
    from long_sequence_attention_02_b300.workloads import WORKLOADS

    w = WORKLOADS["wan14b_720p_self_fwd"]
    B, L, H, grid = w.B, w.L, w.H, w.grid
    qb, kb, vb = _inputs(B, grid, H, seed=0)
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    o, lse = wan.attention_forward_fp8(q, k, v, grid)
    wan.check(wan.wan_get_device_status())
    del q, k, v
    rng = np.random.default_rng(11)
    flat = rng.choice(B * H * L, size=4096, replace=False)
    bs, hs, is_ = flat // (H * L), (flat // L) % H, flat % L
    o_rows, lse_rows = dev_to_f64(o[bs, is_, hs]), dev_to_f64(lse[bs, hs, is_])
    r_o, r_l = np.zeros_like(o_rows), np.zeros_like(lse_rows)
    for bh in sorted(set(zip(bs.tolist(), hs.tolist()))):
        sel = np.where((bs == bh[0]) & (hs == bh[1]))[0]
        r_o[sel], r_l[sel] = ref.self_attention_fwd_rows(f64(qb[bh[0], is_[sel], bh[1]]), is_[sel],
                                                         f64(kb[bh[0], :, bh[1]]), f64(vb[bh[0], :, bh[1]]), grid)
    compare_fp8(o_rows, r_o, lse_rows, r_l, "fp8, 75,600 tokens")
