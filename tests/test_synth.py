"""The seeded input generator (host only, no GPU)."""
import numpy as np
import pytest

from long_sequence_attention_02_b300 import synth


def test_splitmix64_published_outputs():
    # SplitMix64 started from state 0: the first three outputs as published
    # with the reference implementation of the generator.
    out = synth.raw_stream(0, 3)
    assert [int(x) for x in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


@pytest.mark.parametrize("seed,stream,offset", [(0, 1, 0), (1, 2, 12345), (2, 4, 7)])
def test_c_generator_matches_numpy_statement(seed, stream, offset):
    n = 50_000
    a = synth.normal_bf16(seed, stream, (n,), offset=offset)
    b = synth.normal_bf16_numpy(seed, stream, n, offset=offset)
    assert np.array_equal(a, b)


def test_indexed_draw_matches_contiguous():
    a = synth.normal_bf16(3, synth.STREAM_K, (4, 1000))
    idx = np.array([5, 999, 1000, 3999, 2048], dtype=np.uint64)
    b = synth.normal_bf16_at(3, synth.STREAM_K, idx)
    assert np.array_equal(a.reshape(-1)[idx.astype(np.int64)], b)


def test_normal_statistics():
    x = synth.bf16_bits_to_f64(synth.normal_bf16(0, synth.STREAM_Q, (1 << 20,)))
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    # fourth moment of N(0,1) is 3
    assert abs(np.mean(x ** 4) - 3.0) < 0.05
    assert np.all(np.isfinite(x))


def test_streams_and_seeds_differ():
    a = synth.normal_bf16(0, synth.STREAM_Q, (4096,))
    b = synth.normal_bf16(0, synth.STREAM_K, (4096,))
    c = synth.normal_bf16(1, synth.STREAM_Q, (4096,))
    assert not np.array_equal(a, b) and not np.array_equal(a, c)


def test_bf16_widening_exact():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x4049, 0x7F7F], dtype=np.uint16)
    x = synth.bf16_bits_to_f64(bits)
    assert x[0] == 1.0 and x[1] == -1.0 and x[2] == 0.0
    assert x[3] == 3.140625
    assert x[4] == float.fromhex("0x1.fep127")


def test_kv_lens_range():
    lens = synth.kv_lens(0, 10000)
    assert lens.min() >= 16 and lens.max() <= 512
    assert lens.dtype == np.int32
    assert abs(lens.mean() - 264) < 5
