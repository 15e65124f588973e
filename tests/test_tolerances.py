"""Pins of the parity acceptance rules: the oracle's tie diagnostics and the bands.

A GPU output passes the strict check when it is a correct rounding of a value
within a band of the oracle's exact value, or of the interval the oracle
reports where an intermediate rounding sat near a tie.  These tests fix that
machinery from outside the oracle, so that a band made wider than its error
analysis allows fails here:
  * the near-tie decision at values placed at known distances from a rounding
    midpoint, and the candidate it offers;
  * the prologue's tie interval on a head built so that its normalized value
    lands at a chosen distance from a midpoint;
  * the magnitude (error scale) diagnostics on hand-worked rows;
  * every band against its fp32 error analysis, and against planted slips: a
    slip of half the band is accepted, one of four bands is caught.
The strength control of the ninfer text-profile pull request ("Output") is the
standard: a tolerance must not hide a slip the comparison exists to find.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import f32_ok, storage, strict_ok
from memory_bound_decode_qk_gb300 import synth
from tolerances import (ETA_NORM, GATE_BAND, REL_F32, U, gate_error_coefficients, gate_eta,
                        rms_norm_error_u)

# a bf16 rounding midpoint near 1: 258/256 and 260/256 are neighbours in bf16
M_BF16 = 259.0 / 256.0
# an fp16 midpoint near 1: 1 + 2^-11 lies between 1 and 1 + 2^-10
M_F16 = 1.0 + 2.0 ** -11


# ---------------------------------------------------------------- near-tie decision

# (format, midpoint, neighbour below, neighbour above, the even one of the two):
# 260/256 = 65/64 has the even bf16 significand, 1 the even fp16 one
@pytest.mark.parametrize("fmt,M,down,up,even", [
    (oracle.BF16, M_BF16, 258 / 256, 260 / 256, 260 / 256),
    (oracle.F16, M_F16, 1.0, 1.0 + 2.0 ** -10, 1.0)])
def test_near_tie_band_is_eta_wide(fmt, M, down, up, even):
    eta = 2.0 ** -18
    # inside the band on either side: flagged, and the other neighbour offered
    for rel, own, other in ((-2.0 ** -19, down, up), (2.0 ** -19, up, down),
                            (-2.0 ** -20, down, up), (2.0 ** -20, up, down)):
        v = M * (1.0 + rel)
        assert oracle.round_to(v, fmt) == own
        assert oracle.near_tie(v, fmt, eta) == (True, other)
        assert oracle.near_tie(-v, fmt, eta) == (True, -other)
    # twice the band away on either side: not flagged
    for rel in (-2.0 ** -17, 2.0 ** -17, -2.0 ** -16, 2.0 ** -12):
        flagged, other = oracle.near_tie(M * (1.0 + rel), fmt, eta)
        assert not flagged and other == oracle.round_to(M * (1.0 + rel), fmt)
    # the exact midpoint rounds to even and offers the odd neighbour
    assert oracle.round_to(M, fmt) == even
    assert oracle.near_tie(M, fmt, eta) == (True, down if even == up else up)
    # the band scales with eta: 2^-17 away is inside a band of 2^-16
    assert oracle.near_tie(M * (1 + 2.0 ** -17), fmt, 2.0 ** -16)[0]
    # representable values and values far from any midpoint are never flagged
    assert not oracle.near_tie(down, fmt, eta)[0]
    assert not oracle.near_tie((down + M) / 2, fmt, eta)[0]


def test_near_tie_never_applies_to_fp32_intermediates():
    # fp32 heads round the normalized value exactly like the GPU: no interval
    inp = synth.qk_inputs(3, torch.float32, 8, 4, 2, 64, 64, theta=1e4, cache_len=16,
                          positions="arange")
    r = oracle.qk_norm_rope(*(storage(inp[n]) for n in ("q", "k", "wq", "wk")), oracle.F32, 64,
                            oracle.ROTATE_HALF, inp["positions"].numpy(), storage(inp["cos"]),
                            storage(inp["sin"]), 1e-6, 1, eta=2.0 ** -10)
    assert np.array_equal(r.q_lo, r.q_hi) and np.array_equal(r.k_lo, r.k_hi)


# ---------------------------------------------------------------- the prologue's tie interval

def _head_at(eps, out_fmt=None, rotary=2):
    """One bf16 head [1, 1] of length 2 whose channel 0 normalizes to
    (259/256) / sqrt(1 + eps): x = (1, 1) gives mean(x^2) = 1, and the offset
    weight 3/256 gives 1 + w = 259/256, the bf16 midpoint.  Position 0 of a
    one-row cache (cos 1, sin 0) rotates by the identity."""
    bf = lambda a: storage(torch.tensor(a, dtype=torch.bfloat16))
    x = bf([[[1.0, 1.0]]])
    w = bf([3.0 / 256.0, 0.0])
    cos = np.ones((1, 1), np.float32)
    sin = np.zeros((1, 1), np.float32)
    return oracle.qk_norm_rope(x, x, w, w, oracle.BF16, rotary, oracle.ROTATE_HALF,
                               np.zeros(1, np.int64), cos, sin, eps, 1,
                               out_fmt=out_fmt, inv_scale=1.0, eta=ETA_NORM)


@pytest.mark.parametrize("out_fmt,rotary", [(None, 2), (oracle.E4M3, 0)])
def test_prologue_tie_interval_follows_the_band(out_fmt, rotary):
    # eps = 2^-18: n0 = M (1 - 2^-19 + ...), inside the band of 2^-18
    near = 1.0 - 1.0 / math.sqrt(1.0 + 2.0 ** -18)
    assert 0.9 * 2.0 ** -19 < near < 1.1 * 2.0 ** -19
    r = _head_at(2.0 ** -18, out_fmt, rotary)
    assert r.q_lo[0, 0, 0] == 258 / 256 and r.q_hi[0, 0, 0] == 260 / 256
    # channel 1 normalizes to 1 - 2^-19: far from the midpoint below 1
    assert r.q_lo[0, 0, 1] == r.q_hi[0, 0, 1] == 1.0
    # eps = 2^-16: n0 = M (1 - 2^-17 + ...), twice the band away: no interval
    r = _head_at(2.0 ** -16, out_fmt, rotary)
    assert r.q_lo[0, 0, 0] == r.q_hi[0, 0, 0] == 258 / 256


# ---------------------------------------------------------------- magnitude diagnostics

def test_layernorm_magnitude_on_a_hand_worked_row():
    # x = (1, 2, 3, 6): mean 3, mean |x| 3, biased variance 3.5, r = 1/sqrt(3.5)
    x = np.array([[1.0, 2.0, 3.0, 6.0]], np.float32)
    g = np.array([1.0, -2.0, 0.5, 1.0], np.float32)
    b = np.array([0.0, 0.25, -1.0, 0.0], np.float32)
    _, pre, mag = oracle.layernorm(x, g, b, oracle.F32, 0.0)
    r = 1.0 / math.sqrt(3.5)
    np.testing.assert_allclose(pre[0], [-2 * r, 2 * r + 0.25, -1.0, 3 * r], rtol=1e-15)
    # (|x_i| + |mu| + mean|x|) r |gamma_i| + |beta_i|
    np.testing.assert_allclose(mag[0], [7 * r, 16 * r + 0.25, 4.5 * r + 1.0, 12 * r],
                               rtol=1e-15)
    # no affine: (|x_i| + 6) r
    _, _, mag = oracle.layernorm(x, None, None, oracle.F32, 0.0)
    np.testing.assert_allclose(mag[0], np.array([7, 8, 9, 12]) * r, rtol=1e-15)


def test_prologue_magnitude_is_the_pair_norm():
    # fp32 head (3, 4): r = 1/sqrt(12.5) and n = (3, 4) r has norm sqrt(2)
    x = np.array([[[3.0, 4.0]]], np.float32)
    c, s = np.float32(0.6), np.float32(0.8)
    cos, sin = np.array([[c]], np.float32), np.array([[s]], np.float32)
    r = oracle.qk_norm_rope(x, x, None, None, oracle.F32, 2, oracle.ROTATE_HALF,
                            np.zeros(1, np.int64), cos, sin, 0.0, 0)
    m = np.float32(np.array([3.0, 4.0]) / math.sqrt(12.5)).astype(np.float64)
    want = math.hypot(m[0], m[1]) * math.hypot(float(c), float(s))
    np.testing.assert_allclose(r.q_mag[0, 0], [want, want], rtol=1e-15)
    # without rotation each channel's scale is its own magnitude
    r = oracle.qk_norm_rope(x, x, None, None, oracle.F32, 0, oracle.ROTATE_HALF,
                            np.zeros(1, np.int64), None, None, 0.0, 0)
    np.testing.assert_allclose(r.q_mag[0, 0], np.array([3.0, 4.0]) / math.sqrt(12.5),
                               rtol=1e-15)
    # standalone rotation: the pair norm of (3, 4) is 5 times |(c, s)|
    out, pre, mag = oracle.rope(x, oracle.F32, 2, oracle.ROTATE_HALF, np.zeros(1, np.int64),
                                cos, sin, diagnostics=True)
    np.testing.assert_allclose(mag[0, 0], [5 * math.hypot(float(c), float(s))] * 2, rtol=1e-15)


# ---------------------------------------------------------------- bands vs their analysis

def test_norm_band_covers_its_error_bound_with_at_most_twice_the_margin():
    bound = rms_norm_error_u()
    assert bound * U <= ETA_NORM <= 2 * bound * U
    # the LayerNorm mean adds at most as many terms as the sum of squares, and
    # its error is carried by the magnitude scale (|x| + |mu| + mean|x|) r |gamma|
    assert rms_norm_error_u() < ETA_NORM / U


@pytest.mark.parametrize("act", [oracle.SILU, oracle.GELU_TANH])
def test_gate_band_covers_its_error_bound_with_at_most_twice_the_margin(act):
    c0, c1 = gate_error_coefficients(act)
    b0, b1 = GATE_BAND[act]
    assert c0 <= b0 <= 2 * c0 and c1 <= b1 <= 2 * c1


# ---------------------------------------------------------------- planted slips

def _slip(pre, rel_or_abs, fmt, inv=1.0):
    """Round (or quantize) the slipped exact values like an output."""
    if fmt == oracle.E4M3:
        return oracle.quantize(pre + rel_or_abs, inv)
    return oracle.encode(pre + rel_or_abs, fmt)


def _norm_case(fmt):
    inp = synth.rows_inputs(0, {oracle.BF16: torch.bfloat16, oracle.F16: torch.float16,
                                oracle.F32: torch.float32}[fmt], 64, 2560)
    _, pre = oracle.rmsnorm(storage(inp["x"]), storage(inp["w"]), fmt, 1e-6)
    return pre


@pytest.mark.parametrize("fmt", [oracle.BF16, oracle.F16])
def test_norm_band_accepts_half_a_band_and_catches_four(fmt):
    pre = _norm_case(fmt)
    mag = np.abs(pre)
    ok = strict_ok(_slip(pre, 0.5 * ETA_NORM * mag, fmt), pre, pre, mag, fmt, ETA_NORM)
    assert ok.all()
    ok = strict_ok(_slip(pre, 4 * ETA_NORM * mag, fmt), pre, pre, mag, fmt, ETA_NORM)
    assert np.count_nonzero(~ok) >= 20


def test_fp8_band_accepts_half_a_band_and_catches_four():
    inp = synth.rows_inputs(0, torch.bfloat16, 512, 2048, outlier_frac=0.001)
    _, pre = oracle.rmsnorm(storage(inp["x"]), None, oracle.BF16, 1e-6)
    inv = float(np.float32(448.0) / np.float32(np.abs(pre).max()))
    mag = np.abs(pre)
    ok = strict_ok(_slip(pre, 0.5 * ETA_NORM * mag, oracle.E4M3, inv), pre, pre, mag,
                   oracle.E4M3, ETA_NORM, inv_scale=inv)
    assert ok.all()
    ok = strict_ok(_slip(pre, 4 * ETA_NORM * mag, oracle.E4M3, inv), pre, pre, mag,
                   oracle.E4M3, ETA_NORM, inv_scale=inv)
    assert np.count_nonzero(~ok) >= 5


def test_fp32_bar_accepts_half_and_catches_four():
    pre = _norm_case(oracle.F32)
    mag = np.abs(pre)
    ok = f32_ok(np.float32(pre * (1 + 0.5 * REL_F32)), pre, mag, REL_F32)
    assert ok.all()
    ok = f32_ok(np.float32(pre * (1 + 4 * REL_F32)), pre, mag, REL_F32)
    assert np.count_nonzero(~ok) > 0.9 * pre.size


@pytest.mark.parametrize("act", [oracle.SILU, oracle.GELU_TANH])
def test_gate_band_accepts_half_a_band_and_catches_four(act):
    inp = synth.glu_inputs(0, torch.bfloat16, 64, 9728, std=2.0)
    gu = storage(inp["gate_up"])
    _, pre = oracle.glu_act(gu, oracle.BF16, act)
    eta = gate_eta(oracle.decode(gu, oracle.BF16)[:, :9728], act)
    mag = np.abs(pre)
    ok = strict_ok(_slip(pre, 0.5 * eta * mag, oracle.BF16), pre, pre, mag, oracle.BF16, eta)
    assert ok.all()
    ok = strict_ok(_slip(pre, 4 * eta * mag, oracle.BF16), pre, pre, mag, oracle.BF16, eta)
    assert np.count_nonzero(~ok) >= 20


def test_layernorm_band_accepts_half_a_band_and_catches_four():
    # the slip is sized by the magnitude scale written out here, not the
    # oracle's, so that an inflated oracle scale cannot hide it
    x = synth.to_dtype(synth.normal(0, 41, 256 * 1152, 0.7, 2.0), torch.bfloat16).view(256, 1152)
    g = synth.to_dtype(synth.normal(0, 42, 1152, 1.0, 0.1), torch.bfloat16)
    b = synth.to_dtype(synth.normal(0, 43, 1152, 0.0, 0.1), torch.bfloat16)
    _, pre, mag = oracle.layernorm(storage(x), storage(g), storage(b), oracle.BF16, 1e-5)
    xv, gv, bv = (t.double().numpy() for t in (x, g, b))
    mu = xv.mean(axis=1, keepdims=True)
    r = 1.0 / np.sqrt(((xv - mu) ** 2).mean(axis=1, keepdims=True) + np.float32(1e-5))
    scale = (np.abs(xv) + np.abs(mu) + np.abs(xv).mean(axis=1, keepdims=True)) * r * np.abs(gv) \
        + np.abs(bv)
    np.testing.assert_allclose(mag, scale, rtol=1e-12)
    ok = strict_ok(_slip(pre, 0.5 * ETA_NORM * scale, oracle.BF16), pre, pre, mag, oracle.BF16,
                   ETA_NORM)
    assert ok.all()
    ok = strict_ok(_slip(pre, 4 * ETA_NORM * scale, oracle.BF16), pre, pre, mag, oracle.BF16,
                   ETA_NORM)
    assert np.count_nonzero(~ok) >= 20


def test_prologue_interval_catches_four_bands():
    # the rotated channels use the oracle's tie interval [lo, hi]: a slip of
    # four bands of the pair norm past it is still caught
    inp = synth.qk_inputs(0, torch.bfloat16, 256, 16, 2, 256, 64, theta=1e7, cache_len=32768,
                          positions="offset", w_std=0.05)
    r = oracle.qk_norm_rope(*(storage(inp[n]) for n in ("q", "k", "wq", "wk")), oracle.BF16, 64,
                            oracle.ROTATE_HALF, inp["positions"].numpy(), storage(inp["cos"]),
                            storage(inp["sin"]), 1e-6, 1, eta=ETA_NORM)
    rot = (slice(None), slice(None), slice(0, 64))
    lo, hi, mag, pre = r.q_lo[rot], r.q_hi[rot], r.q_mag[rot], r.q_pre[rot]
    ok = strict_ok(_slip(pre, 0.5 * ETA_NORM * mag, oracle.BF16), lo, hi, mag, oracle.BF16,
                   ETA_NORM)
    assert ok.all()
    ok = strict_ok(_slip(hi, 4 * ETA_NORM * mag, oracle.BF16), lo, hi, mag, oracle.BF16, ETA_NORM)
    assert np.count_nonzero(~ok) >= 20
