"""Shared helpers of the test suite: seeded inputs, conversions, comparison."""
import math

import numpy as np

from long_sequence_attention_02_b300 import synth

# Tolerances of the workload (bf16 inputs, fp32 accumulation, fp64 oracle).
MAX_ABS = 2e-2
REL_L2 = 5e-3


def bits(seed, stream, shape):
    return synth.normal_bf16(seed, stream, shape)


def to_dev(b):
    import torch

    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()


def dev_to_f64(t):
    import torch

    x = t.detach()
    if x.dtype == torch.bfloat16:
        x = x.float()
    return x.cpu().numpy().astype(np.float64)


def f64(b):
    return synth.bf16_bits_to_f64(b)


def compare(got, ref, name, max_abs=MAX_ABS, rel_l2=REL_L2):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    fin = np.isfinite(ref)
    # -inf entries (empty rows) must match exactly
    assert np.array_equal(np.isfinite(got), fin), f"{name}: finiteness differs"
    assert np.all(got[~fin] == ref[~fin]), f"{name}: non-finite values differ"
    g, r = got[fin], ref[fin]
    err = np.abs(g - r)
    mx = float(err.max()) if err.size else 0.0
    nrm = float(np.linalg.norm(r))
    rl2 = float(np.linalg.norm(g - r) / nrm) if nrm > 0 else float(np.linalg.norm(g - r))
    assert mx <= max_abs, f"{name}: max-abs {mx:.3e} > {max_abs}"
    assert rl2 <= rel_l2, f"{name}: rel-L2 {rl2:.3e} > {rel_l2}"
    return mx, rl2


def scale_of(d=128):
    return 1.0 / math.sqrt(d)
