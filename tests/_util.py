"""Shared helpers of the test suite: seeded inputs, conversions, comparison."""
import contextlib
import ctypes
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


def bf16_round(x):
    """bf16 bits of float values, rounded to nearest even (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def rows_whose_reference_moves(qf, kf, grid, bound=256.0):
    """How many query rows of a self-attention forward move their softmax
    reference at least once, following the kernels' schedule: an item is 256
    query rows of one (b, h); it visits its 128-key tiles cyclically from tile
    qp * n_tiles // n_qpairs; the first tile visited sets the reference to its
    row maximum, and a later tile whose row sum of 2^(x - m) exceeds `bound`
    moves it to that tile's maximum. Lets a test check that its inputs really
    take that path."""
    from oracle import ref

    B, L, H, d = qf.shape
    ang = ref.rope_angles(*grid, d)
    n_tiles = (L + 127) // 128
    n_qpairs = (L + 255) // 256
    c = scale_of(d) * math.log2(math.e)
    moved_rows = 0
    for b in range(B):
        for h in range(H):
            x = (ref.rope_rotate(qf[b, :, h], ang) @ ref.rope_rotate(kf[b, :, h], ang).T) * c
            for qp in range(n_qpairs):
                xs = x[256 * qp:256 * (qp + 1)]
                start = qp * n_tiles // n_qpairs
                order = [(start + j) % n_tiles for j in range(n_tiles)]
                m = xs[:, 128 * order[0]:128 * (order[0] + 1)].max(axis=1)
                moved = np.zeros(len(xs), dtype=bool)
                for t in order[1:]:
                    blk = xs[:, 128 * t:128 * (t + 1)]
                    need = np.exp2(blk - m[:, None]).sum(axis=1) > bound
                    m = np.where(need, np.maximum(m, blk.max(axis=1)), m)
                    moved |= need
                moved_rows += int(moved.sum())
    return moved_rows


@contextlib.contextmanager
def blas_single_threaded():
    """Run numpy's BLAS on one thread inside the block, so that a pool of
    Python threads, each in its own BLAS call, spreads over the cores without
    oversubscribing them. Uses threadpoolctl when installed, else the loaded
    OpenBLAS's own set_num_threads; if neither is found, BLAS is left as is
    (the result is the same, only slower)."""
    try:
        from threadpoolctl import threadpool_limits
    except ImportError:
        threadpool_limits = None
    if threadpool_limits is not None:
        with threadpool_limits(limits=1, user_api="blas"):
            yield
        return
    setter = getter = None
    try:
        with open("/proc/self/maps") as f:
            paths = sorted({ln.split()[-1] for ln in f if "openblas" in ln.lower() and ln.split()[-1].startswith("/")})
        for path in paths:
            lib = ctypes.CDLL(path)
            for suffix in ("64_", ""):
                for prefix in ("scipy_openblas", "openblas"):
                    if hasattr(lib, f"{prefix}_set_num_threads{suffix}"):
                        setter = getattr(lib, f"{prefix}_set_num_threads{suffix}")
                        getter = getattr(lib, f"{prefix}_get_num_threads{suffix}")
                        break
                if setter:
                    break
            if setter:
                break
    except OSError:
        setter = None
    if setter is None:
        yield
        return
    before = int(getter())
    setter(1)
    try:
        yield
    finally:
        setter(before)
