"""Pins of the oracle's number formats against independent references.

The oracle rounds and decodes binary32, binary16, bfloat16 and E4M3 "fn"
from the formats' definitions.  These tests check it against numpy's and
torch's own conversions, against hand-derived points (tests/golden), and
exhaustively over every bit pattern where that is cheap.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        if line.startswith("#") or not line.strip():
            continue
        v, b = line.split()[:2]
        rows.append((float(v), int(b, 16)))
    return rows


def test_e4m3_golden_points():
    # hand-derived from the OCP OFP8 definition (see the file header)
    for v, code in _golden("e4m3_points.txt"):
        got = oracle.quantize(np.array([v]), 1.0)[0]
        assert got == code, (v, hex(got), hex(code))


def test_bf16_golden_points():
    for v, bits in _golden("bf16_points.txt"):
        assert oracle.bits_of(oracle.round_to(v, oracle.BF16), oracle.BF16) == bits, v


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode(codes, oracle.E4M3)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])
    # NaN exactly at S.1111.111
    assert set(np.flatnonzero(np.isnan(got))) == {0x7F, 0xFF}


def test_e4m3_encode_round_trip_all_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = oracle.decode(codes, oracle.E4M3)
    back = oracle.quantize(vals, 1.0)
    # +0 and -0 both exist; every other code maps back to itself
    assert np.array_equal(back, codes)


def test_e4m3_encode_vs_torch_random_and_midpoints():
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(20000) * 50,
        rng.standard_normal(20000) * 0.01,
        rng.uniform(-448, 448, 20000),
    ]).astype(np.float32)
    # every midpoint between adjacent finite positive codes (fp32-exact)
    pos = np.sort(oracle.decode(np.arange(0, 0x7F, dtype=np.uint8), oracle.E4M3))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.quantize(v.astype(np.float64), 1.0)
    assert np.array_equal(got, ref)


def test_e4m3_saturates_instead_of_nan():
    v = np.array([448.0, 449.0, 500.0, 1e9, -1e9, np.inf, -np.inf])
    got = oracle.quantize(v, 1.0)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE]


def test_bf16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32)
    ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = oracle.decode(bits.astype(np.uint16), oracle.BF16)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


def test_f16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.decode(bits, oracle.F16)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])


def _bf16_midpoints(rng, n):
    # random bf16 values plus half a bf16 spacing: fp32-exact rounding midpoints
    b = rng.integers(0, 0x7F7F, n).astype(np.uint32)
    base = (b << 16).view(np.float32).astype(np.float64)
    half = ((b + 1) << 16).view(np.float32).astype(np.float64) - base
    return base + half / 2


def test_bf16_round_vs_torch():
    rng = np.random.default_rng(11)
    v = np.concatenate([
        rng.standard_normal(50000).astype(np.float32).astype(np.float64),
        (rng.standard_normal(5000) * 1e-39).astype(np.float32).astype(np.float64),
        _bf16_midpoints(rng, 20000),
    ])
    v = np.concatenate([v, -v])
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    got = oracle.encode(v, oracle.BF16)
    assert np.array_equal(got, ref.view(np.uint16))


def test_f16_round_vs_numpy():
    rng = np.random.default_rng(12)
    v = np.concatenate([
        rng.standard_normal(50000),
        rng.standard_normal(5000) * 1e-6,           # subnormal range
        rng.standard_normal(5000) * 3e4,            # near overflow
        np.array([65504.0, 65519.99, 65520.0, 70000.0, 2.0 ** -25, 3 * 2.0 ** -26]),
    ])
    ref = v.astype(np.float16).view(np.uint16)
    got = oracle.encode(v, oracle.F16)
    assert np.array_equal(got, ref)


def test_f32_round_vs_numpy():
    rng = np.random.default_rng(13)
    v = np.concatenate([rng.standard_normal(50000) * 10.0 ** rng.integers(-40, 38, 50000),
                        np.array([3.5e38, 1e-46])])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float32)
    got = oracle.encode(v, oracle.F32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("fmt", [oracle.F16, oracle.BF16, oracle.E4M3])
def test_rounding_is_monotone(fmt):
    rng = np.random.default_rng(14)
    v = np.sort(rng.standard_normal(100000) * 4)
    if fmt == oracle.E4M3:
        r = oracle.decode(oracle.quantize(v, 1.0), fmt)
    else:
        r = oracle.decode(oracle.encode(v, fmt), fmt)
    assert np.all(np.diff(r) >= 0)


def test_fp8_decision_taken_in_fp32():
    # The static-scale epilogue quantizes the fp32 result: y (fp32) times the
    # inverse scale (fp32), rounded to fp32, then converted to E4M3.  Values are
    # placed next to E4M3 rounding midpoints so that a decision taken in fp64
    # would differ; torch's fp32 multiply + float8 cast is the reference.
    inv = np.float32(448.0 / 6.3)
    pos = np.sort(oracle.decode(np.arange(0, 0x7F, dtype=np.uint8), oracle.E4M3))
    mids = (pos[:-1] + pos[1:]) / 2
    rng = np.random.default_rng(15)
    v = []
    for mid in mids:
        target = mid / np.float64(inv)
        base = np.float32(target)
        for k in range(-3, 4):
            v.append(np.nextafter(base, np.float32(np.inf * np.sign(k))) if k else base)
    v = np.array(v, np.float32)
    v = np.concatenate([v, -v, (rng.standard_normal(20000) * 3).astype(np.float32)])
    ref = (torch.from_numpy(v) * torch.tensor(inv)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    ref = ref.view(torch.uint8).numpy()
    got = oracle.quantize(v.astype(np.float64), float(inv))
    assert np.array_equal(got, ref)
    # the set must contain cases where the fp64 product rounds differently
    exact = oracle.encode(v.astype(np.float64) * np.float64(inv), oracle.E4M3)
    assert np.count_nonzero(exact != got) > 0
