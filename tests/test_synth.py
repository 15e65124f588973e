"""The seeded generator is deterministic, stream-separated and has the
requested distributions."""
import numpy as np
import pytest
import torch

from memory_bound_decode_qk_gb300 import synth


def test_deterministic_and_stream_separated():
    a = synth.normal(0, 1, 1000)
    b = synth.normal(0, 1, 1000)
    c = synth.normal(0, 2, 1000)
    d = synth.normal(1, 1, 1000)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)
    # a prefix of a longer draw is the shorter draw (counter-based)
    assert np.array_equal(synth.normal(0, 1, 10), a[:10])


def test_known_first_draws():
    # SplitMix64 is fully specified: the first draws never change
    b = synth.raw_bits(0, 1, 3)
    assert b.dtype == np.uint64 and len(set(b.tolist())) == 3
    assert np.array_equal(b, synth.raw_bits(0, 1, 3))


def test_moments():
    z = synth.normal(3, 7, 200000, mean=1.0, std=0.5)
    assert abs(z.mean() - 1.0) < 0.01 and abs(z.std() - 0.5) < 0.01
    u = synth.uniform(3, 8, 200000)
    assert u.min() > 0 and u.max() < 1 and abs(u.mean() - 0.5) < 0.01


def test_outlier_fraction():
    x = np.ones(1_000_000)
    y = synth.with_outliers(x, 0, 31, 0.001, 20.0)
    frac = np.count_nonzero(y == 20.0) / y.size
    assert 0.0008 < frac < 0.0012


def test_positions_recipes():
    inp = synth.qk_inputs(0, torch.float32, 4, 8, 2, 128, 128, theta=1e6, cache_len=4096,
                          positions="cfg_out_of_cache")
    p = inp["positions"].numpy()
    assert p[-1] == 4096 and np.all((p[:3] >= 0) & (p[:3] < 4096))
    inp = synth.qk_inputs(0, torch.bfloat16, 16, 2, 1, 256, 64, theta=1e7, cache_len=32768,
                          positions="offset")
    p = inp["positions"].numpy()
    assert np.array_equal(np.diff(p), np.ones(15)) and p[0] >= 0 and p[-1] < 32768
    assert inp["cos"].shape == (32768, 32) and inp["cos"].dtype == torch.float32


def test_rope_cache_rows():
    cos, sin = synth.rope_cache(1e4, 8, 3)
    assert torch.equal(cos[0], torch.ones(4)) and torch.equal(sin[0], torch.zeros(4))
    np.testing.assert_allclose(cos[2, 1].item(), np.cos(2 * 1e4 ** (-2 / 8)), rtol=1e-7)


def test_block_positions():
    # B sequences of W consecutive positions, each inside the cache, ordered [B][W]
    p = synth.block_positions(0, 16, 5, 32768)
    assert p.shape == (80,) and p.dtype == np.int64
    blocks = p.reshape(5, 16)
    assert np.all(np.diff(blocks, axis=1) == 1)
    assert blocks[:, 0].min() >= 0 and blocks[:, -1].max() < 32768
    assert len(set(blocks[:, 0].tolist())) > 1
    # W equal to the cache length leaves a single start, 0
    assert np.array_equal(synth.block_positions(3, 8, 2, 8), np.tile(np.arange(8), 2))
    inp = synth.qk_inputs(0, torch.bfloat16, 48, 2, 2, 128, 128, theta=1e6, cache_len=4096,
                          positions="blocks:16")
    assert np.array_equal(inp["positions"].numpy(), synth.block_positions(0, 16, 3, 4096))
    with pytest.raises(ValueError):
        synth.qk_inputs(0, torch.bfloat16, 50, 2, 2, 128, 128, theta=1e6, cache_len=4096,
                        positions="blocks:16")
