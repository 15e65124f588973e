"""Pins of the oracle's operators against what the pages and mathematics fix.

Each operator is checked against at least one reference that does not share
its code: a torch CPU library routine in fp64, a closed form, an exact
identity, brute force by complex multiplication, or an eager torch add.  The
checks are chosen so that a plausible slip fails one of them.  Examples: eps
outside the root, mean taken as a sum, a wrong rotation sign, swapped pair
indices, a missed intermediate rounding, gate and up halves swapped.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from helpers import storage
from memory_bound_decode_qk_gb300 import synth

DT = [torch.float32, torch.float16, torch.bfloat16]
FMT = {torch.float32: oracle.F32, torch.float16: oracle.F16, torch.bfloat16: oracle.BF16}


def E32(v):
    # the operators take eps as binary32, as the C ABI does
    return float(np.float32(v))


def dec(t):
    return oracle.decode(storage(t), FMT[t.dtype])


# ----------------------------------------------------------------- RMSNorm

@pytest.mark.parametrize("dtype", DT)
@pytest.mark.parametrize("offset", [0, 1])
def test_rmsnorm_vs_torch_fp64(dtype, offset):
    inp = synth.rows_inputs(3, dtype, 7, 37, w_mean=0.0 if offset else 1.0, w_std=0.3,
                            residual=False)
    out, pre = oracle.rmsnorm(storage(inp["x"]), storage(inp["w"]), FMT[dtype], 1e-5, offset)
    x64 = torch.from_numpy(dec(inp["x"]))
    w64 = torch.from_numpy(dec(inp["w"])) + offset
    ref = F.rms_norm(x64, (37,), weight=w64, eps=E32(1e-5)).numpy()
    np.testing.assert_allclose(pre, ref, rtol=1e-13, atol=0)
    # one rounding of the exact value
    assert np.array_equal(out, oracle.encode(pre, FMT[dtype]))


def test_rmsnorm_no_weight_vs_torch():
    inp = synth.rows_inputs(4, torch.bfloat16, 5, 2048, residual=False)
    _, pre = oracle.rmsnorm(storage(inp["x"]), None, oracle.BF16, 1e-6)
    ref = F.rms_norm(torch.from_numpy(dec(inp["x"])), (2048,), eps=E32(1e-6)).numpy()
    np.testing.assert_allclose(pre, ref, rtol=1e-13)


def test_rmsnorm_unit_weight_has_rms_one():
    # closed form: with unit weight, rms(y) = sqrt(ms / (ms + eps))
    inp = synth.rows_inputs(5, torch.float32, 4, 1024, residual=False)
    x = dec(inp["x"])
    eps = 1e-2
    _, pre = oracle.rmsnorm(storage(inp["x"]), None, oracle.F32, eps)
    ms = np.mean(x * x, axis=1)
    eps = E32(eps)
    np.testing.assert_allclose(np.sqrt(np.mean(pre * pre, axis=1)), np.sqrt(ms / (ms + eps)),
                               rtol=1e-13)


def test_rmsnorm_constant_row_closed_form():
    # x = c * 1 gives y = c / sqrt(c^2 + eps) * w
    c, eps, H = 0.75, 1e-3, 16
    x = torch.full((1, H), c, dtype=torch.float32)
    w = torch.linspace(-2, 2, H, dtype=torch.float32)
    _, pre = oracle.rmsnorm(storage(x), storage(w), oracle.F32, eps)
    ref = c / math.sqrt(c * c + E32(eps)) * w.double().numpy()
    np.testing.assert_allclose(pre[0], ref, rtol=1e-14)


def test_rmsnorm_worked_example_bf16():
    # x = [3, 4], eps = 0: mean square 12.5, y = [3, 4] / sqrt(12.5)
    # = [0.8485281374, 1.1313708499]; bf16: 0.8485 * 256 = 217.2 -> 217/256,
    # 1.1314 * 128 = 144.8 -> 145/128.
    x = torch.tensor([[3.0, 4.0]], dtype=torch.bfloat16)
    out, pre = oracle.rmsnorm(storage(x), None, oracle.BF16, 0.0)
    np.testing.assert_allclose(pre[0], [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rtol=1e-15)
    assert list(oracle.decode(out, oracle.BF16)[0]) == [217 / 256, 145 / 128]


@pytest.mark.parametrize("dtype", DT)
def test_offset_zero_equals_direct_one(dtype):
    # the Gemma form 1 + w at w = 0 is bit-identical to the Llama form at w = 1
    inp = synth.rows_inputs(6, dtype, 9, 300, residual=False)
    zero = torch.zeros(300, dtype=dtype)
    one = torch.ones(300, dtype=dtype)
    a, _ = oracle.rmsnorm(storage(inp["x"]), storage(zero), FMT[dtype], 1e-6, 1)
    b, _ = oracle.rmsnorm(storage(inp["x"]), storage(one), FMT[dtype], 1e-6, 0)
    c, _ = oracle.rmsnorm(storage(inp["x"]), None, FMT[dtype], 1e-6, 0)
    assert np.array_equal(a, b) and np.array_equal(a, c)


def test_rmsnorm_scale_invariance():
    inp = synth.rows_inputs(7, torch.float32, 3, 64, residual=False)
    x = inp["x"]
    _, p1 = oracle.rmsnorm(storage(x), storage(inp["w"]), oracle.F32, 0.0)
    _, p2 = oracle.rmsnorm(storage(x * 8.0), storage(inp["w"]), oracle.F32, 0.0)
    np.testing.assert_allclose(p1, p2, rtol=1e-14)


# ----------------------------------------------------------------- residual add

@pytest.mark.parametrize("dtype", DT)
def test_residual_sum_bit_identical_to_eager_add(dtype):
    inp = synth.rows_inputs(8, dtype, 6, 333)
    # include large-exponent-gap pairs to exercise the fp32 add before rounding
    x = inp["x"].clone()
    x[0, :10] = x[0, :10] * 1e4
    _, res, _ = oracle.add_rmsnorm(storage(x), storage(inp["residual"]), storage(inp["w"]),
                                   FMT[dtype], 1e-6)
    eager = x + inp["residual"]
    assert np.array_equal(res, storage(eager))


@pytest.mark.parametrize("dtype", DT)
def test_add_rmsnorm_normalizes_the_rounded_sum(dtype):
    inp = synth.rows_inputs(9, dtype, 5, 256)
    out, res, pre = oracle.add_rmsnorm(storage(inp["x"]), storage(inp["residual"]),
                                       storage(inp["w"]), FMT[dtype], 1e-6, 0)
    s64 = torch.from_numpy(oracle.decode(res, FMT[dtype]))
    ref = F.rms_norm(s64, (256,), weight=torch.from_numpy(dec(inp["w"])), eps=E32(1e-6)).numpy()
    np.testing.assert_allclose(pre, ref, rtol=1e-13)
    out2, _ = oracle.rmsnorm(res, storage(inp["w"]), FMT[dtype], 1e-6, 0)
    assert np.array_equal(out, out2)


# ----------------------------------------------------------------- gates

def _gate_up(g, u):
    return torch.cat([torch.as_tensor(g), torch.as_tensor(u)], dim=1)


@pytest.mark.parametrize("act", [oracle.SILU, oracle.GELU_TANH])
def test_gates_vs_torch_fp64(act):
    inp = synth.glu_inputs(10, torch.float32, 8, 500, std=2.0)
    gu = inp["gate_up"]
    _, pre = oracle.glu_act(storage(gu), oracle.F32, act)
    g = gu[:, :500].double()
    u = gu[:, 500:].double()
    ref = F.silu(g) if act == oracle.SILU else F.gelu(g, approximate="tanh")
    ref = (ref * u).numpy()
    # torch's tanh form cancels for very negative g: compare where it is well conditioned
    ok = g.numpy() > -3.0
    np.testing.assert_allclose(pre[ok], ref[ok], rtol=1e-12, atol=1e-300)


@pytest.mark.parametrize("act", [oracle.SILU, oracle.GELU_TANH])
def test_gate_odd_part_identity(act):
    # act(x) - act(-x) = x for both gates (z is odd in x for the tanh form)
    g = torch.linspace(-12, 12, 2001, dtype=torch.float64).float().view(1, -1)
    u = torch.ones_like(g)
    _, p_pos = oracle.glu_act(storage(_gate_up(g, u)), oracle.F32, act)
    _, p_neg = oracle.glu_act(storage(_gate_up(-g, u)), oracle.F32, act)
    np.testing.assert_allclose(p_pos - p_neg, g.double().numpy(), rtol=1e-14, atol=1e-14)


@pytest.mark.parametrize("act", [oracle.SILU, oracle.GELU_TANH])
def test_gate_limits_and_order(act):
    g = torch.tensor([[0.0, 30.0, 3.0]], dtype=torch.float32)
    u = torch.tensor([[5.0, 2.0, 1.0]], dtype=torch.float32)
    _, p = oracle.glu_act(storage(_gate_up(g, u)), oracle.F32, act)
    assert p[0, 0] == 0.0                              # act(0) = 0
    np.testing.assert_allclose(p[0, 1], 60.0, rtol=1e-12)  # act(g) -> g for large g
    # gate is the first half: swapping the halves changes the result
    _, q = oracle.glu_act(storage(_gate_up(u, g)), oracle.F32, act)
    assert q[0, 2] != p[0, 2]


def test_gelu_identity_matches_tanh_form_where_well_conditioned():
    g = np.linspace(-3.0, 6.0, 901)
    z = math.sqrt(2 / math.pi) * (g + 0.044715 * g ** 3)
    tanh_form = 0.5 * g * (1 + np.tanh(z))
    x = torch.from_numpy(g.astype(np.float32)).view(1, -1)
    _, p = oracle.glu_act(storage(_gate_up(x, torch.ones_like(x))), oracle.F32, oracle.GELU_TANH)
    g32 = x.double().numpy()[0]
    z32 = math.sqrt(2 / math.pi) * (g32 + 0.044715 * g32 ** 3)
    np.testing.assert_allclose(p[0], 0.5 * g32 * (1 + np.tanh(z32)), rtol=1e-12, atol=1e-15)
    assert tanh_form.shape == p[0].shape


def test_gelu_far_negative_is_not_cancelled():
    # exact value 0.5 g (1 + tanh z) = g e^{2z} / (1 + e^{2z}); at g = -8 it is
    # about -8 e^{-49}, nonzero; a cancelling 1 + tanh(z) would give 0
    x = torch.tensor([[-8.0]], dtype=torch.float32)
    _, p = oracle.glu_act(storage(_gate_up(x, torch.ones_like(x))), oracle.F32, oracle.GELU_TANH)
    z = math.sqrt(2 / math.pi) * (-8 + 0.044715 * -512)
    np.testing.assert_allclose(p[0, 0], -8 * math.exp(2 * z) / (1 + math.exp(2 * z)), rtol=1e-12)
    assert p[0, 0] < 0


# ----------------------------------------------------------------- rotary / prologue

def _qk(dtype, T=3, Hq=4, Hk=2, D=64, rho=64, layout=oracle.ROTATE_HALF, positions="arange",
        cache_len=64, theta=1e4, offset=1, seed=21, w_mean=0.0, w_std=0.1):
    inp = synth.qk_inputs(seed, dtype, T, Hq, Hk, D, rho, theta=theta, cache_len=cache_len,
                          positions=positions, w_mean=w_mean, w_std=w_std)
    r = oracle.qk_norm_rope(storage(inp["q"]), storage(inp["k"]), storage(inp["wq"]),
                            storage(inp["wk"]), FMT[dtype], rho, layout,
                            inp["positions"].numpy(), storage(inp["cos"]) if rho else None,
                            storage(inp["sin"]) if rho else None, 1e-6, offset)
    return inp, r


def _heads_norm(inp, dtype, offset):
    """Per-head RMSNorm through the row operator (q rows use wq, k rows wk)."""
    T, Hq, D = inp["q"].shape
    Hk = inp["k"].shape[1]
    qn, qpre = oracle.rmsnorm(storage(inp["q"]).reshape(T * Hq, D), storage(inp["wq"]),
                              FMT[dtype], 1e-6, offset)
    kn, kpre = oracle.rmsnorm(storage(inp["k"]).reshape(T * Hk, D), storage(inp["wk"]),
                              FMT[dtype], 1e-6, offset)
    return qn.reshape(T, Hq, D), kn.reshape(T, Hk, D), qpre.reshape(T, Hq, D), kpre.reshape(T, Hk, D)


@pytest.mark.parametrize("layout", [oracle.ROTATE_HALF, oracle.INTERLEAVED])
def test_rotation_vs_complex_multiplication(layout):
    # RoFormer: pair (a, b) as a + ib times e^{i angle} = c + i s
    T, H, D, rho = 4, 3, 32, 24
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal((T, H, D)).astype(np.float32))
    cos, sin = synth.rope_cache(1e4, rho, 50)
    pos = np.array([0, 7, 49, 13])
    out = oracle.rope(storage(x), oracle.F32, rho, layout, pos, storage(cos), storage(sin))
    xv = x.double().numpy()
    half = rho // 2
    if layout == oracle.ROTATE_HALF:
        ia, ib = np.arange(half), np.arange(half) + half
    else:
        ia, ib = 2 * np.arange(half), 2 * np.arange(half) + 1
    z = xv[:, :, ia] + 1j * xv[:, :, ib]
    e = cos.double().numpy()[pos][:, None, :] + 1j * sin.double().numpy()[pos][:, None, :]
    zr = z * e
    ref = xv.copy()
    ref[:, :, ia] = zr.real
    ref[:, :, ib] = zr.imag
    got = out.astype(np.float64)
    np.testing.assert_allclose(got, ref.astype(np.float32).astype(np.float64), rtol=2 ** -23,
                               atol=1e-30)
    # channels past rotary_dim pass through untouched
    assert np.array_equal(out[:, :, rho:], storage(x)[:, :, rho:])


@pytest.mark.parametrize("dtype", DT)
@pytest.mark.parametrize("layout", [oracle.ROTATE_HALF, oracle.INTERLEAVED])
def test_fused_equals_norm_round_rope(dtype, layout):
    # the ninfer text profile's contract: fused == rmsnorm -> rmsnorm -> rope
    # from the rounded normalized value, bit for bit
    inp, r = _qk(dtype, T=5, Hq=3, Hk=2, D=64, rho=32, layout=layout,
                 positions=np.array([0, 5, 63, 64, -1]), cache_len=64)
    qn, kn, _, _ = _heads_norm(inp, dtype, 1)
    pos = inp["positions"].numpy()
    cs, sn = storage(inp["cos"]), storage(inp["sin"])
    qref = oracle.rope(qn, FMT[dtype], 32, layout, pos, cs, sn)
    kref = oracle.rope(kn, FMT[dtype], 32, layout, pos, cs, sn)
    assert np.array_equal(r.q_out, qref) and np.array_equal(r.k_out, kref)


@pytest.mark.parametrize("dtype", DT)
def test_position_zero_is_identity(dtype):
    inp, r = _qk(dtype, positions=np.zeros(3, np.int64))
    qn, kn, _, _ = _heads_norm(inp, dtype, 1)
    assert np.array_equal(r.q_out, qn) and np.array_equal(r.k_out, kn)


@pytest.mark.parametrize("p", [64, 65, 10 ** 12, -1, -(2 ** 62)])
def test_out_of_cache_token_is_normalized_not_rotated(p):
    inp, r = _qk(torch.bfloat16, positions=np.array([3, p, 5]), cache_len=64)
    qn, kn, _, _ = _heads_norm(inp, torch.bfloat16, 1)
    assert np.array_equal(r.q_out[1], qn[1]) and np.array_equal(r.k_out[1], kn[1])
    # the in-cache tokens around it do rotate
    assert not np.array_equal(r.q_out[0], qn[0])


def test_pair_norm_preserved():
    inp, r = _qk(torch.float32, T=4, D=128, rho=128, positions=np.array([1, 100, 1000, 4095]),
                 cache_len=4096, theta=1e6)
    _, _, qpre, _ = _heads_norm(inp, torch.float32, 1)
    m = qpre.astype(np.float32).astype(np.float64)   # the rounded intermediate
    half = 64
    before = np.hypot(m[..., :half], m[..., half:])
    after = np.hypot(r.q_pre[..., :half], r.q_pre[..., half:])
    np.testing.assert_allclose(after, before, rtol=3e-7)


def test_interleaved_equals_rotate_half_under_permutation():
    # channel 2j <-> j and 2j+1 <-> j + rho/2 maps one layout onto the other
    T, Hq, Hk, D = 3, 2, 1, 16
    inp = synth.qk_inputs(5, torch.float32, T, Hq, Hk, D, D, theta=1e4, cache_len=32,
                          positions="arange")
    perm = np.empty(D, np.int64)
    perm[0::2] = np.arange(D // 2)
    perm[1::2] = np.arange(D // 2) + D // 2
    args = lambda q, k, wq, wk: (storage(q), storage(k), storage(wq), storage(wk))
    a = oracle.qk_norm_rope(*args(inp["q"], inp["k"], inp["wq"], inp["wk"]), oracle.F32, D,
                            oracle.ROTATE_HALF, inp["positions"].numpy(), storage(inp["cos"]),
                            storage(inp["sin"]), 1e-6, 1)
    b = oracle.qk_norm_rope(*args(inp["q"][..., perm], inp["k"][..., perm], inp["wq"][perm],
                                  inp["wk"][perm]), oracle.F32, D, oracle.INTERLEAVED,
                            inp["positions"].numpy(), storage(inp["cos"]), storage(inp["sin"]),
                            1e-6, 1)
    assert np.array_equal(a.q_out[..., perm], b.q_out)
    assert np.array_equal(a.k_out[..., perm], b.k_out)


def test_partial_rotary_passes_normalized_channels():
    # ninfer text profile: only the first 64 of 256 channels rotate
    inp, r = _qk(torch.bfloat16, T=3, Hq=2, Hk=1, D=256, rho=64, positions=np.array([1, 2, 3]),
                 cache_len=8, theta=1e7)
    qn, kn, _, _ = _heads_norm(inp, torch.bfloat16, 1)
    assert np.array_equal(r.q_out[..., 64:], qn[..., 64:])
    assert np.array_equal(r.k_out[..., 64:], kn[..., 64:])
    assert not np.array_equal(r.q_out[..., :64], qn[..., :64])


def test_relative_position_property():
    # <R_m q, R_n k> = <q, R_{n-m} k> (RoFormer), up to the fp32 cache error
    D = 64
    rng = np.random.default_rng(8)
    qv = rng.standard_normal(D).astype(np.float32)
    kv = rng.standard_normal(D).astype(np.float32)
    cos, sin = synth.rope_cache(1e4, D, 512)
    x = torch.from_numpy(np.stack([qv, kv, qv, kv])).view(4, 1, D)
    m, n = 37, 300
    out = oracle.rope(storage(x), oracle.F32, D, oracle.ROTATE_HALF, np.array([m, n, 0, n - m]),
                      storage(cos), storage(sin)).astype(np.float64)
    lhs = out[0, 0] @ out[1, 0]
    rhs = out[2, 0] @ out[3, 0]
    assert abs(lhs - rhs) <= 1e-4 * (np.linalg.norm(qv) * np.linalg.norm(kv))


def test_strength_control_sees_one_part_per_million():
    # a rotation scaled by 1.000001 (far below a bf16 ulp) must flip some exact
    # comparisons, as in the ninfer strength control; a tolerance would not
    inp, base = _qk(torch.bfloat16, T=64, Hq=16, Hk=2, D=256, rho=64, positions="offset",
                    cache_len=4096, theta=1e7, seed=33)
    with oracle.rotation_scale(1.000001):
        _, pert = _qk(torch.bfloat16, T=64, Hq=16, Hk=2, D=256, rho=64, positions="offset",
                      cache_len=4096, theta=1e7, seed=33)
    flips = np.count_nonzero(base.q_out != pert.q_out) + np.count_nonzero(base.k_out != pert.k_out)
    assert flips > 0
    # only rotated channels can move
    assert np.array_equal(base.q_out[..., 64:], pert.q_out[..., 64:])
    from helpers import ulp_distance
    assert ulp_distance(base.q_out, pert.q_out, oracle.BF16).max() <= 1


def test_fp32_intermediate_is_fp32_rounding():
    # for fp32 the "round to the input dtype" step is a binary32 rounding
    inp, r = _qk(torch.float32, positions=np.array([70, 70, 70]), cache_len=64)
    _, _, qpre, _ = _heads_norm(inp, torch.float32, 1)
    assert np.array_equal(r.q_out, qpre.astype(np.float32))


# ----------------------------------------------------------------- FP8 epilogue

def test_fp8_outputs_are_the_quantized_exact_values():
    inp = synth.rows_inputs(12, torch.bfloat16, 8, 512, outlier_frac=0.001)
    inv = np.float32(448.0 / 6.0)
    out, res, pre = oracle.add_rmsnorm(storage(inp["x"]), storage(inp["residual"]), None,
                                       oracle.BF16, 1e-6, 0, out_fmt=oracle.E4M3,
                                       inv_scale=float(inv))
    assert np.array_equal(out, oracle.quantize(pre, float(inv)))
    # saturation, never NaN, for finite inputs
    assert not np.any((out & 0x7F) == 0x7F)
    assert np.any((out & 0x7F) == 0x7E)


def test_fp8_calibrated_scale_hits_the_top_code():
    # static calibration: scale = amax / 448 on a calibration pass; quantizing
    # that same pass maps the amax element to the top code 448
    inp = synth.glu_inputs(1, torch.bfloat16, 16, 256)
    _, pre = oracle.glu_act(storage(inp["gate_up"]), oracle.BF16, oracle.GELU_TANH)
    amax = np.abs(pre).max()
    inv = float(np.float32(1.0 / np.float32(amax / 448.0)))
    out, _ = oracle.glu_act(storage(inp["gate_up"]), oracle.BF16, oracle.GELU_TANH,
                            out_fmt=oracle.E4M3, inv_scale=inv)
    i = np.unravel_index(np.argmax(np.abs(pre)), pre.shape)
    assert out[i] & 0x7F == 0x7E


def test_fp8_qk_quantizes_rotated_and_rounded_values():
    inp, r8 = None, None
    inp = synth.qk_inputs(2, torch.bfloat16, 4, 2, 1, 128, 64, theta=1e7, cache_len=16,
                          positions=np.array([1, 2, 40, 3]))
    a = [storage(inp[n]) for n in ("q", "k", "wq", "wk")]
    rb = oracle.qk_norm_rope(*a, oracle.BF16, 64, oracle.ROTATE_HALF, inp["positions"].numpy(),
                             storage(inp["cos"]), storage(inp["sin"]), 1e-6, 1)
    r8 = oracle.qk_norm_rope(*a, oracle.BF16, 64, oracle.ROTATE_HALF, inp["positions"].numpy(),
                             storage(inp["cos"]), storage(inp["sin"]), 1e-6, 1,
                             out_fmt=oracle.E4M3, inv_scale=32.0)
    # pass-through channels and the out-of-cache token quantize the bf16 value
    m = oracle.decode(rb.q_out, oracle.BF16)
    assert np.array_equal(r8.q_out[:, :, 64:], oracle.quantize(m[:, :, 64:], 32.0))
    assert np.array_equal(r8.q_out[2], oracle.quantize(m[2], 32.0))
    assert np.array_equal(r8.q_out, oracle.quantize(r8.q_pre, 32.0))


def test_tie_bounds_bracket_the_exact_value():
    # diagnostics for the GPU tie policy: lo <= pre <= hi everywhere, and the
    # interval is non-trivial only where an intermediate rounding was near a tie
    inp, r = _qk(torch.float16, T=64, Hq=8, Hk=2, D=64, rho=32, layout=oracle.INTERLEAVED,
                 positions="arange", cache_len=128)
    for lo, pre, hi in ((r.q_lo, r.q_pre, r.q_hi), (r.k_lo, r.k_pre, r.k_hi)):
        assert np.all(lo <= pre) and np.all(pre <= hi)
    wide = np.count_nonzero(r.q_hi > r.q_lo) + np.count_nonzero(r.k_hi > r.k_lo)
    assert 0 < wide < 0.2 * (r.q_lo.size + r.k_lo.size)
    # pass-through channels of a bf16/fp16 output round n itself: no interval
    assert np.array_equal(r.q_lo[..., 32:], r.q_hi[..., 32:])


# ----------------------------------------------------------------- review variant and standalone rope

@pytest.mark.parametrize("layout", [oracle.ROTATE_HALF, oracle.INTERLEAVED])
def test_unrounded_variant_rotates_the_exact_normalized_value(layout):
    # the ninfer review (item 1): rotate the fp32 RMSNorm result and round once.
    # Pin: torch fp64 rms_norm, then complex multiplication, then one rounding.
    T, H, D, rho = 6, 3, 64, 32
    inp = synth.qk_inputs(4, torch.bfloat16, T, H, 1, D, rho, theta=1e4, cache_len=64,
                          positions=np.array([0, 3, 9, 63, 64, -1]), w_std=0.1)
    r = oracle.qk_norm_rope(storage(inp["q"]), storage(inp["k"]), storage(inp["wq"]),
                            storage(inp["wk"]), oracle.BF16, rho, layout, inp["positions"].numpy(),
                            storage(inp["cos"]), storage(inp["sin"]), 1e-6, 1, unrounded=True)
    x64 = torch.from_numpy(dec(inp["q"]))
    w64 = torch.from_numpy(dec(inp["wq"])) + 1.0
    n = F.rms_norm(x64, (D,), weight=w64, eps=E32(1e-6)).numpy()
    half = rho // 2
    ia, ib = (np.arange(half), np.arange(half) + half) if layout == oracle.ROTATE_HALF else \
        (2 * np.arange(half), 2 * np.arange(half) + 1)
    ref = n.copy()
    pos = inp["positions"].numpy()
    for t in range(T):
        if 0 <= pos[t] < 64:
            e = (inp["cos"].double().numpy()[pos[t]] + 1j * inp["sin"].double().numpy()[pos[t]])
            z = (n[t][:, ia] + 1j * n[t][:, ib]) * e
            ref[t][:, ia], ref[t][:, ib] = z.real, z.imag
    np.testing.assert_allclose(r.q_pre, ref, rtol=1e-12, atol=1e-15)
    assert np.array_equal(r.q_out, oracle.encode(ref, oracle.BF16))
    # the rounded (default) form differs somewhere in the rotated channels only
    r0 = oracle.qk_norm_rope(storage(inp["q"]), storage(inp["k"]), storage(inp["wq"]),
                             storage(inp["wk"]), oracle.BF16, rho, layout, pos,
                             storage(inp["cos"]), storage(inp["sin"]), 1e-6, 1)
    assert np.array_equal(r0.q_out[..., rho:], r.q_out[..., rho:])


def test_unrounded_and_rounded_differ_somewhere():
    inp, r0 = _qk(torch.bfloat16, T=32, Hq=8, Hk=2, D=128, rho=128, positions="arange",
                  cache_len=64)
    a = [storage(inp[n]) for n in ("q", "k", "wq", "wk")]
    r1 = oracle.qk_norm_rope(*a, oracle.BF16, 128, oracle.ROTATE_HALF, inp["positions"].numpy(),
                             storage(inp["cos"]), storage(inp["sin"]), 1e-6, 1, unrounded=True)
    assert np.count_nonzero(r0.q_out != r1.q_out) > 0


def test_rope_diagnostics_and_fp8():
    T, H, D, rho = 4, 2, 32, 16
    rng = np.random.default_rng(9)
    x = torch.from_numpy(rng.standard_normal((T, H, D)).astype(np.float32)).to(torch.bfloat16)
    cos, sin = synth.rope_cache(1e4, rho, 8)
    pos = np.array([0, 5, 7, 8])
    out, pre, mag = oracle.rope(storage(x), oracle.BF16, rho, oracle.ROTATE_HALF, pos,
                                storage(cos), storage(sin), diagnostics=True)
    assert np.array_equal(out, oracle.encode(pre, oracle.BF16))
    assert np.all(mag >= np.abs(pre))
    # out-of-cache token (position 8 with 8 rows) is copied unchanged
    assert np.array_equal(out[3], storage(x)[3])
    q8 = oracle.rope(storage(x), oracle.BF16, rho, oracle.ROTATE_HALF, pos, storage(cos),
                     storage(sin), out_fmt=oracle.E4M3, inv_scale=16.0)
    assert np.array_equal(q8, oracle.quantize(pre, 16.0))


# ----------------------------------------------------------------- LayerNorm and static quantize

@pytest.mark.parametrize("dtype", DT)
@pytest.mark.parametrize("affine", [True, False])
def test_layernorm_vs_torch_fp64(dtype, affine):
    rng = np.random.default_rng(21)
    x = torch.from_numpy(rng.standard_normal((6, 77)) * 3 + 1.5).to(dtype)
    g = torch.from_numpy(1 + 0.1 * rng.standard_normal(77)).to(dtype) if affine else None
    b = torch.from_numpy(0.1 * rng.standard_normal(77)).to(dtype) if affine else None
    out, pre, mag = oracle.layernorm(storage(x), None if g is None else storage(g),
                                     None if b is None else storage(b), FMT[dtype], 1e-5)
    ref = F.layer_norm(torch.from_numpy(dec(x)), (77,),
                       weight=None if g is None else torch.from_numpy(dec(g)),
                       bias=None if b is None else torch.from_numpy(dec(b)),
                       eps=E32(1e-5)).numpy()
    np.testing.assert_allclose(pre, ref, rtol=1e-12, atol=1e-14)
    assert np.array_equal(out, oracle.encode(pre, FMT[dtype]))
    assert np.all(mag >= np.abs(pre) - 1e-12)


def test_layernorm_closed_forms():
    # no affine: each row has mean 0 and variance var/(var+eps); a constant row
    # normalizes to beta; adding a constant to a row changes nothing
    rng = np.random.default_rng(22)
    # values on a 2^-10 grid, so that x + 64 is exact in fp32
    x = torch.from_numpy(np.round(rng.standard_normal((4, 256)) * 1024) / 1024).float()
    _, pre, _ = oracle.layernorm(storage(x), None, None, oracle.F32, 1e-3)
    xv = x.double().numpy()
    var = xv.var(axis=1)
    np.testing.assert_allclose(pre.mean(axis=1), 0, atol=1e-13)
    np.testing.assert_allclose(pre.var(axis=1), var / (var + E32(1e-3)), rtol=1e-12)
    _, pre2, _ = oracle.layernorm(storage(x + 64.0), None, None, oracle.F32, 1e-3)
    np.testing.assert_allclose(pre2, pre, atol=1e-11)
    c = torch.full((1, 16), 2.5)
    beta = torch.linspace(-1, 1, 16)
    _, pc, _ = oracle.layernorm(storage(c), storage(torch.ones(16)), storage(beta), oracle.F32,
                                1e-5)
    np.testing.assert_allclose(pc[0], beta.double().numpy(), atol=1e-15)


@pytest.mark.parametrize("dtype", DT)
def test_quantize_static_vs_torch(dtype):
    rng = np.random.default_rng(23)
    x = torch.from_numpy(rng.standard_normal(5000) * 4).to(dtype)
    inv = np.float32(448.0 / 9.0)
    got = oracle.quantize_static(storage(x), FMT[dtype], float(inv))
    ref = (x.float() * torch.tensor(inv)).clamp(-448, 448).to(torch.float8_e4m3fn)
    assert np.array_equal(got, ref.view(torch.uint8).numpy())


# ----------------------------------------------------------------- fused QKV split + KV-cache write

@pytest.mark.parametrize("normalize", [True, False])
def test_qkv_rope_cache_is_split_prologue_and_scatter(normalize):
    T, Hq, Hk, D, rho, S = 6, 4, 2, 64, 32, 10
    dtype, fmt = torch.bfloat16, oracle.BF16
    rng = np.random.default_rng(61)
    qkv = torch.from_numpy(rng.standard_normal((T, (Hq + 2 * Hk) * D))).to(dtype)
    wq = torch.from_numpy(0.1 * rng.standard_normal(D)).to(dtype)
    wk = torch.from_numpy(0.1 * rng.standard_normal(D)).to(dtype)
    cos, sin = synth.rope_cache(1e4, rho, 16)
    pos = np.array([0, 3, 15, 16, -1, 7])
    slots = np.array([9, 0, -1, 4, 12, 5])
    kc0 = storage(torch.from_numpy(rng.standard_normal((S, Hk, D))).to(dtype))
    vc0 = storage(torch.from_numpy(rng.standard_normal((S, Hk, D))).to(dtype))
    r = oracle.qkv_rope_cache(storage(qkv), storage(wq), storage(wk), fmt, Hq, Hk, rho,
                              oracle.ROTATE_HALF, pos, storage(cos), storage(sin), slots, kc0, vc0,
                              1e-6, 1, normalize)
    x = storage(qkv).reshape(T, Hq + 2 * Hk, D)
    q, k, v = x[:, :Hq], x[:, Hq:Hq + Hk], x[:, Hq + Hk:]
    if normalize:
        ref = oracle.qk_norm_rope(q, k, storage(wq), storage(wk), fmt, rho, oracle.ROTATE_HALF,
                                  pos, storage(cos), storage(sin), 1e-6, 1)
        rq, rk = ref.q_out, ref.k_out
    else:
        rq = oracle.rope(q, fmt, rho, oracle.ROTATE_HALF, pos, storage(cos), storage(sin))
        rk = oracle.rope(k, fmt, rho, oracle.ROTATE_HALF, pos, storage(cos), storage(sin))
    assert np.array_equal(r.q_out, rq)
    for t in range(T):
        if 0 <= slots[t] < S:
            assert np.array_equal(r.k_cache[slots[t]], rk[t])
            assert np.array_equal(r.v_cache[slots[t]], v[t])
    untouched = [s for s in range(S) if s not in set(slots[(slots >= 0) & (slots < S)])]
    assert np.array_equal(r.k_cache[untouched], kc0[untouched])
    assert np.array_equal(r.v_cache[untouched], vc0[untouched])
