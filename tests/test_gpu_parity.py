"""GPU parity: every op through the C ABI against the CPU oracle.

The inputs are seeded and shaped like the five workloads.  The sizes span
several tiles and a ragged tail, and edge cases are included.  Bars:
  * the residual sum is bit-exact;
  * bf16/fp16 outputs are within 1 ulp, and pass the strict check (bit-exact
    except within a derived band eta around rounding midpoints);
  * FP8 codes are bit-exact outside that band;
  * fp32 outputs are within a relative error of 2e-6 of the exact value (at
    the pair norm for rotated channels).
Every output sits between guard regions that must come back untouched.

Bands: tests/tolerances.py, which gives the fp32 error analysis behind each
(ETA_NORM for every normalized output, a per-element band for the gates),
pinned on the CPU by tests/test_tolerances.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import (TORCH_FMT, f32_ok, position_delta_bf16, report, storage, strict_ok,
                     ulp_distance, within_one_ulp)
from memory_bound_decode_qk_gb300 import edge_ops, synth
from tolerances import ETA_NORM, REL_F32, gate_eta
import case_stats

pytestmark = pytest.mark.gpu

GUARD = 256  # bytes on each side of every output


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    edge_ops.lib(build_if_missing=True)


# ---------------------------------------------------------------- plumbing

class Guarded:
    """An output tensor between guard bytes filled with a known pattern."""

    def __init__(self, shape, dtype, misalign_elems=0):
        esz = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape))
        self.off = GUARD + misalign_elems * esz
        self.nbytes = n * esz
        self.raw = torch.empty(self.off + self.nbytes + GUARD, dtype=torch.uint8, device="cuda")
        self.raw.fill_(0xA5)
        self.t = self.raw[self.off:self.off + self.nbytes].view(dtype).view(shape)

    def check(self):
        r = self.raw.cpu().numpy()
        assert np.all(r[:self.off] == 0xA5), "write before the output"
        assert np.all(r[self.off + self.nbytes:] == 0xA5), "write past the output"


def dev(t, misalign_elems=0):
    """Copy a CPU tensor to the device, optionally at an element-misaligned address."""
    if t is None:
        return None
    if not misalign_elems:
        return t.contiguous().cuda()
    flat = torch.empty(t.numel() + misalign_elems, dtype=t.dtype, device="cuda")
    v = flat[misalign_elems:].view(t.shape)
    v.copy_(t)
    return v


def calib_inv(pre):
    """Static calibration: scale = amax / 448 of a calibration pass, inv = 1 / scale (fp32)."""
    amax = float(np.abs(pre).max())
    return float(np.float32(1.0) / np.float32(amax / 448.0))


def _rel(value, exact, mag):
    """|value - exact| over the magnitude scale (over |exact| where mag is 0)."""
    scale = np.where(mag > 0, mag, np.maximum(np.abs(exact), 1e-300))
    return np.abs(value - exact) / scale


def check_dtype_out(name, got, ref_bits, lo, hi, mag, fmt, eta):
    """bf16/fp16: <= 1 ulp everywhere (at the pair norm for rotated channels)
    and the strict check."""
    d = ulp_distance(got, ref_bits, fmt)
    if case_stats.enabled():
        case_stats.record(name, got, d, _rel(oracle.decode(got, fmt), lo, mag))
    one = within_one_ulp(got, ref_bits, mag, fmt)
    assert one.all(), report(name + " (1 ulp)", one)
    ok = strict_ok(got, lo, hi, mag, fmt, eta)
    assert ok.all(), report(name, ok)
    return float(np.mean(d == 0))


def check_fp8_out(name, got, lo, hi, mag, eta, inv):
    if case_stats.enabled():
        d = ulp_distance(got, oracle.quantize(lo, inv), oracle.E4M3)
        case_stats.record(name, got, d, _rel(oracle.decode(got, oracle.E4M3) / inv, lo, mag))
    ok = strict_ok(got, lo, hi, mag, oracle.E4M3, eta, inv_scale=inv)
    assert ok.all(), report(name, ok)


def check_out(name, got, ref_bits, pre, mag, fmt, out_fmt, eta, inv=1.0, lo=None, hi=None):
    lo = pre if lo is None else lo
    hi = pre if hi is None else hi
    if out_fmt == oracle.E4M3:
        check_fp8_out(name, got, lo, hi, mag, eta, inv)
    elif fmt == oracle.F32:
        if case_stats.enabled():
            d = ulp_distance(got, oracle.encode(pre, oracle.F32), oracle.F32)
            case_stats.record(name, got, d, _rel(got.view(np.float32).astype(np.float64), pre, mag))
        ok = f32_ok(got, pre, mag, REL_F32)
        assert ok.all(), report(name, ok)
    else:
        check_dtype_out(name, got, ref_bits, lo, hi, mag, fmt, eta)


# ---------------------------------------------------------------- QK prologue

QK_CASES = {
    # workload 1: fp32, D=128 full rotate-half, (8,2), T=4, one token out of cache, in place
    "cfg1_f32": dict(dtype=torch.float32, T=4, Hq=8, Hk=2, D=128, rot=128, layout=0,
                     w_mean=0.0, w_std=0.1, offset=1, theta=1e6, P=4096,
                     positions="cfg_out_of_cache", inplace=True),
    # workload 3: text profile, bf16 out of place, partial rotary 64 of 256
    "cfg3_16_2_T1": dict(dtype=torch.bfloat16, T=1, Hq=16, Hk=2, D=256, rot=64, layout=0,
                         w_mean=0.0, w_std=0.05, offset=1, theta=1e7, P=32768, positions="offset"),
    "cfg3_24_4_T8": dict(dtype=torch.bfloat16, T=8, Hq=24, Hk=4, D=256, rot=64, layout=0,
                         w_mean=0.0, w_std=0.05, offset=1, theta=1e7, P=32768, positions="offset"),
    "cfg3_16_2_T333": dict(dtype=torch.bfloat16, T=333, Hq=16, Hk=2, D=256, rot=64, layout=0,
                           w_mean=0.0, w_std=0.05, offset=1, theta=1e7, P=32768,
                           positions="offset"),
    # workload 4: interleaved full rotary, direct weights, in place, fp16 and bf16
    "cfg4_f16": dict(dtype=torch.float16, T=512, Hq=16, Hk=8, D=256, rot=256, layout=1,
                     w_mean=1.0, w_std=0.02, offset=0, theta=1e6, P=4096, positions="arange",
                     inplace=True),
    "cfg4_bf16": dict(dtype=torch.bfloat16, T=512, Hq=16, Hk=8, D=256, rot=256, layout=1,
                      w_mean=1.0, w_std=0.02, offset=0, theta=1e6, P=4096, positions="arange",
                      inplace=True),
    # head_dim 128 bf16: two heads per warp (half-warp lane groups)
    "d128_bf16": dict(dtype=torch.bfloat16, T=37, Hq=16, Hk=8, D=128, rot=128, layout=0,
                      w_mean=0.0, w_std=0.1, offset=1, theta=1e6, P=64,
                      positions=np.r_[np.arange(30), [63, 64, 65, -1, -5, 1 << 40, 7]]),
    "d64_f16_interleaved": dict(dtype=torch.float16, T=19, Hq=4, Hk=4, D=64, rot=32, layout=1,
                                w_mean=0.0, w_std=0.1, offset=1, theta=1e4, P=32,
                                positions="arange"),
    # generic paths: non-power-of-two vectors per head, ragged rotary, odd sizes
    "generic_d96": dict(dtype=torch.bfloat16, T=9, Hq=3, Hk=1, D=96, rot=96, layout=0,
                        w_mean=0.0, w_std=0.1, offset=1, theta=1e4, P=16, positions="arange"),
    "generic_rot24": dict(dtype=torch.bfloat16, T=5, Hq=4, Hk=2, D=256, rot=24, layout=0,
                          w_mean=0.0, w_std=0.1, offset=1, theta=1e4, P=16, positions="arange"),
    "generic_odd_d37": dict(dtype=torch.float16, T=6, Hq=2, Hk=3, D=37, rot=20, layout=1,
                            w_mean=1.0, w_std=0.1, offset=0, theta=1e4, P=6,
                            positions=np.array([0, 1, 2, 5, 6, -1])),
    "generic_f32_d256": dict(dtype=torch.float32, T=7, Hq=4, Hk=2, D=256, rot=128, layout=0,
                             w_mean=0.0, w_std=0.1, offset=1, theta=1e6, P=4096,
                             positions="arange"),
    "generic_misaligned": dict(dtype=torch.bfloat16, T=11, Hq=16, Hk=2, D=256, rot=64,
                               layout=0, w_mean=0.0, w_std=0.05, offset=1, theta=1e7, P=4096,
                               positions="offset", misalign=1),
    "no_k_heads": dict(dtype=torch.bfloat16, T=3, Hq=8, Hk=0, D=128, rot=64, layout=0,
                       w_mean=0.0, w_std=0.1, offset=1, theta=1e4, P=16, positions="arange"),
    "no_rotation": dict(dtype=torch.bfloat16, T=4, Hq=8, Hk=2, D=128, rot=0, layout=0,
                        w_mean=0.0, w_std=0.1, offset=1, theta=1e4, P=16, positions="arange"),
    "no_weight": dict(dtype=torch.bfloat16, T=4, Hq=8, Hk=2, D=256, rot=64, layout=0,
                      w_mean=None, w_std=0.0, offset=0, theta=1e7, P=64, positions="arange"),
    # DFlash2 pair [128, 32, W, B] (innermost first): q and k both 32 heads of
    # 128, in place, direct weights, full rotate-half rotary; B sequences of W
    # consecutive draft positions.  W*B = 64 runs the lane-group path, 512 the
    # four-threads-per-head path, 21 a ragged block count.
    "dflash2_W16_B4": dict(dtype=torch.bfloat16, T=64, Hq=32, Hk=32, D=128, rot=128, layout=0,
                           w_mean=1.0, w_std=0.02, offset=0, theta=1e6, P=32768,
                           positions="blocks:16", inplace=True),
    "dflash2_W16_B32": dict(dtype=torch.bfloat16, T=512, Hq=32, Hk=32, D=128, rot=128, layout=0,
                            w_mean=1.0, w_std=0.02, offset=0, theta=1e6, P=32768,
                            positions="blocks:16", inplace=True),
    "dflash2_W7_B3": dict(dtype=torch.bfloat16, T=21, Hq=32, Hk=32, D=128, rot=128, layout=0,
                          w_mean=1.0, w_std=0.02, offset=0, theta=1e6, P=32768,
                          positions="blocks:7", inplace=True),
    # many heads (the lane-group grid is over a wave of resident CTAs): the
    # four-threads-per-head path
    "quad_f32_d128": dict(dtype=torch.float32, T=2001, Hq=8, Hk=2, D=128, rot=128, layout=0,
                          w_mean=0.0, w_std=0.1, offset=1, theta=1e6, P=4096,
                          positions=np.r_[np.arange(1999), [4096, -3]]),
    "quad_f16_d64_interleaved": dict(dtype=torch.float16, T=6000, Hq=4, Hk=4, D=64, rot=32,
                                     layout=1, w_mean=0.0, w_std=0.1, offset=1, theta=1e4,
                                     P=4096, positions="arange"),
    "quad_bf16_d128_no_k": dict(dtype=torch.bfloat16, T=1700, Hq=32, Hk=0, D=128, rot=128,
                                layout=0, w_mean=1.0, w_std=0.02, offset=0, theta=1e6,
                                P=4096, positions="offset", inplace=True),
    "quad_no_weight": dict(dtype=torch.bfloat16, T=700, Hq=24, Hk=4, D=256, rot=64, layout=0,
                           w_mean=None, w_std=0.0, offset=0, theta=1e7, P=32768,
                           positions="offset"),
    # interleaved 512-byte heads with rotation stay on the lane-group path at
    # every width (the dispatch), here at many heads
    "quad_cfg4_interleaved": dict(dtype=torch.bfloat16, T=1000, Hq=16, Hk=8, D=256, rot=256,
                                  layout=1, w_mean=1.0, w_std=0.02, offset=0, theta=1e6,
                                  P=4096, positions="arange", inplace=True),
    "quad_no_rotation": dict(dtype=torch.float16, T=800, Hq=24, Hk=4, D=256, rot=0, layout=0,
                             w_mean=0.0, w_std=0.1, offset=1, theta=1e4, P=16,
                             positions="arange"),
    # mid widths of 16-bit 512-byte heads: two vectors per lane (the grid at
    # 0.44 and 1.38 of a one-vector wave), with tokens past the cache
    "two_vec_16_2_T150": dict(dtype=torch.bfloat16, T=150, Hq=16, Hk=2, D=256, rot=64, layout=0,
                              w_mean=0.0, w_std=0.05, offset=1, theta=1e7, P=100,
                              positions="arange"),
    "two_vec_f16_24_4_T300": dict(dtype=torch.float16, T=300, Hq=24, Hk=4, D=256, rot=128,
                                  layout=0, w_mean=1.0, w_std=0.02, offset=0, theta=1e6, P=4096,
                                  positions="arange"),
    # rotary width whose pairs are not thread-local for four threads per head:
    # the lane-group path serves it (two vectors per lane at this width)
    "quad_declined_rot32": dict(dtype=torch.bfloat16, T=800, Hq=24, Hk=4, D=256, rot=32,
                                layout=0, w_mean=0.0, w_std=0.05, offset=1, theta=1e7,
                                P=32768, positions="offset"),
}


def run_qk(c, fp8=False, seed=0, inv=None):
    dtype, fmt = c["dtype"], TORCH_FMT[c["dtype"]]
    inp = synth.qk_inputs(seed, dtype, c["T"], c["Hq"], c["Hk"], c["D"], c["rot"],
                          theta=c["theta"], cache_len=c["P"], positions=c["positions"],
                          w_mean=c["w_mean"] or 0.0, w_std=c["w_std"])
    if c["w_mean"] is None:
        inp["wq"] = inp["wk"] = None
    out_fmt = oracle.E4M3 if fp8 else fmt
    args = [storage(inp["q"]), storage(inp["k"]),
            None if inp["wq"] is None else storage(inp["wq"]),
            None if inp["wk"] is None else storage(inp["wk"]), fmt, c["rot"], c["layout"],
            inp["positions"].numpy(), storage(inp["cos"]) if c["rot"] else None,
            storage(inp["sin"]) if c["rot"] else None, 1e-6, c["offset"]]
    if fp8 and inv is None:
        cal = synth.qk_inputs(1, dtype, c["T"], c["Hq"], c["Hk"], c["D"], c["rot"],
                              theta=c["theta"], cache_len=c["P"], positions=c["positions"],
                              w_mean=c["w_mean"] or 0.0, w_std=c["w_std"])
        cw = (None, None) if c["w_mean"] is None else (storage(cal["wq"]), storage(cal["wk"]))
        rc = oracle.qk_norm_rope(storage(cal["q"]), storage(cal["k"]), *cw, *args[4:])
        inv = calib_inv(np.concatenate([rc.q_pre.ravel(), rc.k_pre.ravel()]))
    inv = 1.0 if inv is None else inv
    ref = oracle.qk_norm_rope(*args, out_fmt=out_fmt, inv_scale=inv, eta=ETA_NORM)

    mis = c.get("misalign", 0)
    q, k = dev(inp["q"], mis), dev(inp["k"], mis)
    wq, wk = dev(inp["wq"], mis), dev(inp["wk"], mis)
    pos, cs, sn = dev(inp["positions"]), dev(inp["cos"]), dev(inp["sin"])
    odt = torch.uint8 if fp8 else dtype
    if c.get("inplace") and not fp8:
        gq, gk = Guarded(q.shape, dtype), Guarded(k.shape, dtype)
        gq.t.copy_(q)
        gk.t.copy_(k)
        q, k = gq.t, gk.t
    else:
        gq, gk = Guarded(q.shape, odt, mis), Guarded(k.shape, odt, mis)
    edge_ops.qk_norm_rope(q, k, wq, wk, pos, cs, sn, rotary_dim=c["rot"], layout=c["layout"],
                          eps=1e-6, weight_offset=c["offset"], q_out=gq.t, k_out=gk.t, fp8=fp8,
                          inv_scale=inv, cache_len=c["P"])
    torch.cuda.synchronize()
    gq.check()
    gk.check()
    return ref, storage(gq.t.cpu()), storage(gk.t.cpu()), fmt, out_fmt, inv


@pytest.mark.parametrize("name", list(QK_CASES))
def test_qk_norm_rope(name):
    c = QK_CASES[name]
    ref, gq, gk, fmt, out_fmt, inv = run_qk(c)
    check_out(name + " q", gq, ref.q_out, ref.q_pre, ref.q_mag, fmt, out_fmt, ETA_NORM,
              lo=ref.q_lo, hi=ref.q_hi)
    if c["Hk"]:
        check_out(name + " k", gk, ref.k_out, ref.k_pre, ref.k_mag, fmt, out_fmt, ETA_NORM,
                  lo=ref.k_lo, hi=ref.k_hi)


@pytest.mark.parametrize("name", ["cfg3_16_2_T333", "cfg3_24_4_T8", "cfg4_bf16", "cfg1_f32",
                                  "two_vec_16_2_T150", "two_vec_f16_24_4_T300",
                                  "generic_odd_d37", "d128_bf16", "quad_f32_d128",
                                  "quad_f16_d64_interleaved", "quad_cfg4_interleaved",
                                  "dflash2_W16_B32"])
def test_qk_norm_rope_fp8(name):
    c = dict(QK_CASES[name])
    ref, gq, gk, fmt, out_fmt, inv = run_qk(c, fp8=True)
    check_fp8_out(name + " q", gq, ref.q_lo, ref.q_hi, ref.q_mag, ETA_NORM, inv)
    check_fp8_out(name + " k", gk, ref.k_lo, ref.k_hi, ref.k_mag, ETA_NORM, inv)


@pytest.mark.parametrize("T", [16, 1024])
def test_qk_dflash2_full_size(T):
    # the DFlash2 pair at the benchmark's block sizes (W = 16; B = 1 and 64)
    c = dict(QK_CASES["dflash2_W16_B4"], T=T)
    ref, gq, gk, fmt, out_fmt, _ = run_qk(c)
    check_out("q", gq, ref.q_out, ref.q_pre, ref.q_mag, fmt, out_fmt, ETA_NORM, lo=ref.q_lo,
              hi=ref.q_hi)
    check_out("k", gk, ref.k_out, ref.k_pre, ref.k_mag, fmt, out_fmt, ETA_NORM, lo=ref.k_lo,
              hi=ref.k_hi)


@pytest.mark.parametrize("geom", [(16, 2), (24, 4)])
@pytest.mark.parametrize("T", [256, 2048])
def test_qk_text_profile_full_size(geom, T):
    # workload 3 at its sweep sizes, in the launch configuration the benchmark times
    c = dict(QK_CASES["cfg3_16_2_T1"], T=T, Hq=geom[0], Hk=geom[1])
    ref, gq, gk, fmt, out_fmt, _ = run_qk(c)
    check_out("q", gq, ref.q_out, ref.q_pre, ref.q_mag, fmt, out_fmt, ETA_NORM, lo=ref.q_lo,
              hi=ref.q_hi)
    check_out("k", gk, ref.k_out, ref.k_pre, ref.k_mag, fmt, out_fmt, ETA_NORM, lo=ref.k_lo,
              hi=ref.k_hi)


def test_qk_out_of_cache_token_untouched_by_rotation():
    # the out-of-cache token of workload 1 equals the plain per-head RMSNorm
    c = QK_CASES["cfg1_f32"]
    ref, gq, gk, fmt, _, _ = run_qk(c)
    inp = synth.qk_inputs(0, c["dtype"], c["T"], c["Hq"], c["Hk"], c["D"], c["rot"],
                          theta=c["theta"], cache_len=c["P"], positions=c["positions"],
                          w_mean=0.0, w_std=0.1)
    x = dev(inp["q"][-1])
    norm = edge_ops.rmsnorm(x, dev(inp["wq"]), eps=1e-6, weight_offset=1)
    torch.cuda.synchronize()
    ok = f32_ok(storage(norm.cpu()), ref.q_pre[-1], ref.q_mag[-1], REL_F32)
    assert ok.all()
    okq = f32_ok(gq[-1], ref.q_pre[-1], ref.q_mag[-1], REL_F32)
    assert okq.all()


@pytest.mark.parametrize("T", [4, 1500])
def test_qk_without_cache_rows_rotates_nothing(T):
    # cache_len 0 with a rotary width: positions and cache are NULL and no
    # token rotates, so the outputs equal those of rotary width 0 bit for bit
    # (T = 4 takes the lane-group path, T = 1500 four threads per head)
    inp = synth.qk_inputs(0, torch.bfloat16, T, 16, 2, 256, 0, theta=1e7, cache_len=0,
                          positions="arange", w_std=0.05)
    q, k, wq, wk = dev(inp["q"]), dev(inp["k"]), dev(inp["wq"]), dev(inp["wk"])
    a = edge_ops.qk_norm_rope(q, k, wq, wk, None, None, None, rotary_dim=64, cache_len=0,
                              weight_offset=1)
    b = edge_ops.qk_norm_rope(q, k, wq, wk, None, None, None, rotary_dim=0, weight_offset=1)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


# Geometries of the lane-group prologue under a position rewrite: one head per
# warp (bf16, 256), two heads per warp (bf16, 128), fp32 heads (one per warp,
# four channels per lane), the interleaved cache load, and enough heads for
# the two-vectors-per-lane form (12 tokens of 136 heads: 0.27 of a wave).
REWRITE_GEOMS = {
    "bf16_d256_rot64": (torch.bfloat16, 16, 2, 256, 64, 0),
    "bf16_d256_rot64_two_vectors": (torch.bfloat16, 128, 8, 256, 64, 0),
    "bf16_d128_rot128": (torch.bfloat16, 8, 2, 128, 128, 0),
    "f32_d128_rot64": (torch.float32, 4, 2, 128, 64, 0),
    "bf16_d256_interleaved": (torch.bfloat16, 8, 2, 256, 256, 1),
}


@pytest.mark.parametrize("op,geom", [("qk", g) for g in REWRITE_GEOMS] + [("qkv", "bf16_d256_rot64")])
def test_positions_rewritten_by_the_preceding_kernel(op, geom):
    # The kernel just before the prologue on the stream (a residual add whose
    # residual is the positions array) rewrites the positions while the
    # prologue's CTAs may already be resident, computing addresses and
    # prefetching before their dependent-launch wait: every position and
    # cache row must still be read after the wait.
    dtype, Hq, Hk, D, rot, layout = REWRITE_GEOMS[geom]
    T, P = 12, 200
    old = np.array([5, 6, 7, 250, 9, 10, 11, 12, 13, 14, 15, 16], np.int64)
    new = np.array([7, 6, 201, 3, 100, 10, 0, 199, 13, 255, 1, 2], np.int64)
    inp = synth.qk_inputs(0, dtype, T, Hq, Hk, D, rot, theta=1e7, cache_len=P,
                          positions=new, w_std=0.05)
    fmt = TORCH_FMT[dtype]
    pos = dev(torch.from_numpy(old))
    cs, sn = dev(inp["cos"]), dev(inp["sin"])
    wq, wk = dev(inp["wq"]), dev(inp["wk"])
    delta = dev(position_delta_bf16(old, new))
    scratch = torch.empty_like(delta)
    if op == "qk":
        ref = oracle.qk_norm_rope(storage(inp["q"]), storage(inp["k"]), storage(inp["wq"]),
                                  storage(inp["wk"]), fmt, rot, layout, new,
                                  storage(inp["cos"]), storage(inp["sin"]), 1e-6, 1, eta=ETA_NORM)
        q, k = dev(inp["q"]), dev(inp["k"])
        qo, ko = torch.empty_like(q), torch.empty_like(k)
        edge_ops.add_rmsnorm(delta, pos.view(torch.bfloat16).view(1, -1), None, out=scratch)
        edge_ops.qk_norm_rope(q, k, wq, wk, pos, cs, sn, rotary_dim=rot, layout=layout,
                              weight_offset=1, q_out=qo, k_out=ko)
        torch.cuda.synchronize()
        assert np.array_equal(pos.cpu().numpy(), new)
        check_out("q", storage(qo.cpu()), ref.q_out, ref.q_pre, ref.q_mag, fmt, fmt, ETA_NORM,
                  lo=ref.q_lo, hi=ref.q_hi)
        check_out("k", storage(ko.cpu()), ref.k_out, ref.k_pre, ref.k_mag, fmt, fmt, ETA_NORM,
                  lo=ref.k_lo, hi=ref.k_hi)
        return
    qkv = torch.cat([inp["q"].reshape(T, -1), inp["k"].reshape(T, -1),
                     inp["k"].reshape(T, -1)], dim=1).contiguous()
    slots = np.arange(T, dtype=np.int64)
    z = np.zeros((T, Hk, D), np.uint16)
    ref = oracle.qkv_rope_cache(storage(qkv), storage(inp["wq"]), storage(inp["wk"]), fmt, Hq,
                                Hk, rot, oracle.ROTATE_HALF, new, storage(inp["cos"]),
                                storage(inp["sin"]), slots, z, z, 1e-6, 1, 1, eta=ETA_NORM)
    kc = torch.zeros(T, Hk, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    qo = torch.empty(T, Hq, D, dtype=torch.bfloat16, device="cuda")
    edge_ops.add_rmsnorm(delta, pos.view(torch.bfloat16).view(1, -1), None, out=scratch)
    edge_ops.qkv_rope_cache(dev(qkv), Hq, Hk, wq, wk, pos, cs, sn, dev(torch.from_numpy(slots)),
                            kc, vc, rotary_dim=rot, weight_offset=1, q_out=qo)
    torch.cuda.synchronize()
    assert np.array_equal(pos.cpu().numpy(), new)
    check_out("q", storage(qo.cpu()), ref.q_out, ref.q_pre, ref.q_mag, fmt, fmt, ETA_NORM,
              lo=ref.q_lo, hi=ref.q_hi)
    check_out("k_cache", storage(kc.cpu()), ref.k_cache, ref.k_pre, ref.k_mag, fmt, fmt,
              ETA_NORM, lo=ref.k_lo, hi=ref.k_hi)
    assert np.array_equal(storage(vc.cpu()), ref.v_cache)


# ---------------------------------------------------------------- rows

ROW_CASES = {
    # workload 2: decode residual-add RMSNorm, bf16, Llama and Gemma weights
    "cfg2_h2560_T1_direct": dict(dtype=torch.bfloat16, T=1, H=2560, w_mean=1.0, w_std=0.02, off=0),
    "cfg2_h2560_T4_offset": dict(dtype=torch.bfloat16, T=4, H=2560, w_mean=0.0, w_std=0.02, off=1),
    "cfg2_h1024_T16_direct": dict(dtype=torch.bfloat16, T=16, H=1024, w_mean=1.0, w_std=0.02, off=0),
    "cfg2_h1024_T64_offset": dict(dtype=torch.bfloat16, T=64, H=1024, w_mean=0.0, w_std=0.02, off=1),
    "cfg2_h2560_T64_direct": dict(dtype=torch.bfloat16, T=64, H=2560, w_mean=1.0, w_std=0.02, off=0),
    # workload 5 shapes in the activation dtype (the FP8 forms are below)
    "h2048_T512": dict(dtype=torch.bfloat16, T=512, H=2048, w_mean=1.0, w_std=0.02, off=0,
                       outliers=0.001),
    "h2560_T700_ragged": dict(dtype=torch.bfloat16, T=700, H=2560, w_mean=0.0, w_std=0.02, off=1),
    "f16_h1024_T33": dict(dtype=torch.float16, T=33, H=1024, w_mean=1.0, w_std=0.02, off=0),
    "f32_h2048_T9": dict(dtype=torch.float32, T=9, H=2048, w_mean=0.0, w_std=0.1, off=1),
    "f32_h4096_T300": dict(dtype=torch.float32, T=300, H=4096, w_mean=1.0, w_std=0.1, off=0),
    "h16384_T3": dict(dtype=torch.bfloat16, T=3, H=16384, w_mean=1.0, w_std=0.1, off=0),
    "generic_h37": dict(dtype=torch.bfloat16, T=64, H=37, w_mean=1.0, w_std=0.1, off=0),
    "generic_f16_h1000_misaligned": dict(dtype=torch.float16, T=5, H=1000, w_mean=0.0,
                                         w_std=0.1, off=1, misalign=1),
    "generic_h40000": dict(dtype=torch.bfloat16, T=2, H=40000, w_mean=1.0, w_std=0.1, off=0),
    "no_weight_h2048": dict(dtype=torch.bfloat16, T=128, H=2048, w_mean=None, w_std=0.0, off=0),
    # a row of 512 vectors at few rows: two vectors per thread, 8 warps per row
    "h4096_T64_offset": dict(dtype=torch.bfloat16, T=64, H=4096, w_mean=0.0, w_std=0.02, off=1),
}


def run_rows(c, fused, fp8=False, inplace=False, seed=0):
    dtype, fmt = c["dtype"], TORCH_FMT[c["dtype"]]
    mk = lambda s: synth.rows_inputs(s, dtype, c["T"], c["H"], w_mean=c["w_mean"] or 0.0,
                                     w_std=c["w_std"], outlier_frac=c.get("outliers", 0.0))
    inp = mk(seed)
    w = None if c["w_mean"] is None else inp["w"]
    ws = None if w is None else storage(w)
    out_fmt = oracle.E4M3 if fp8 else fmt
    inv = 1.0
    if fp8:
        cal = mk(1)
        if fused:
            _, _, pre = oracle.add_rmsnorm(storage(cal["x"]), storage(cal["residual"]), ws, fmt,
                                           1e-6, c["off"])
        else:
            _, pre = oracle.rmsnorm(storage(cal["x"]), ws, fmt, 1e-6, c["off"])
        inv = calib_inv(pre)
    if fused:
        ref_out, ref_res, pre = oracle.add_rmsnorm(storage(inp["x"]), storage(inp["residual"]),
                                                   ws, fmt, 1e-6, c["off"], out_fmt, inv)
    else:
        ref_out, pre = oracle.rmsnorm(storage(inp["x"]), ws, fmt, 1e-6, c["off"], out_fmt, inv)
        ref_res = None
    mis = c.get("misalign", 0)
    x, wd = dev(inp["x"], mis), dev(w, mis)
    odt = torch.uint8 if fp8 else dtype
    if inplace:
        g = Guarded(x.shape, dtype)
        g.t.copy_(x)
        x = g.t
    else:
        g = Guarded(x.shape, odt, mis)
    gr = None
    if fused:
        gr = Guarded(x.shape, dtype, mis)
        gr.t.copy_(dev(inp["residual"]))
        edge_ops.add_rmsnorm(x, gr.t, wd, eps=1e-6, weight_offset=c["off"], out=g.t, fp8=fp8,
                             inv_scale=inv)
    else:
        edge_ops.rmsnorm(x, wd, eps=1e-6, weight_offset=c["off"], out=g.t, fp8=fp8,
                         inv_scale=inv)
    torch.cuda.synchronize()
    g.check()
    if gr is not None:
        gr.check()
        res = storage(gr.t.cpu())
        if case_stats.enabled():
            case_stats.record("residual", res, ulp_distance(res, ref_res, fmt))
        assert np.array_equal(res, ref_res), "residual sum not bit-exact"
    got = storage(g.t.cpu())
    check_out("out", got, ref_out, pre, np.abs(pre), fmt, out_fmt, ETA_NORM, inv)


@pytest.mark.parametrize("name", list(ROW_CASES))
@pytest.mark.parametrize("fused", [True, False])
def test_rows(name, fused):
    run_rows(ROW_CASES[name], fused)


@pytest.mark.parametrize("name", ["cfg2_h2560_T4_offset", "cfg2_h2560_T64_direct", "h2048_T512",
                                  "generic_h37"])
@pytest.mark.parametrize("fused", [True, False])
def test_rows_in_place(name, fused):
    c = ROW_CASES[name]
    if c.get("misalign"):
        pytest.skip("in-place case uses aligned buffers")
    run_rows(c, fused, inplace=True)


FP8_ROWS = {
    # workload 5: bf16 in, FP8 out, D in {2048, 1024}, T=512, 0.1% outliers x20
    "cfg5_d2048_w": dict(dtype=torch.bfloat16, T=512, H=2048, w_mean=1.0, w_std=0.02, off=0,
                         outliers=0.001),
    "cfg5_d1024_w": dict(dtype=torch.bfloat16, T=512, H=1024, w_mean=0.0, w_std=0.02, off=1,
                         outliers=0.001),
    "cfg5_d2048_noweight": dict(dtype=torch.bfloat16, T=512, H=2048, w_mean=None, w_std=0.0,
                                off=0, outliers=0.001),
    "cfg5_d1024_noweight_T4096": dict(dtype=torch.bfloat16, T=4096, H=1024, w_mean=None,
                                      w_std=0.0, off=0, outliers=0.001),
    "cfg5_d2048_T1": dict(dtype=torch.bfloat16, T=1, H=2048, w_mean=None, w_std=0.0, off=0,
                          outliers=0.001),
    "f32_h1024": dict(dtype=torch.float32, T=77, H=1024, w_mean=1.0, w_std=0.1, off=0),
    "generic_h37": dict(dtype=torch.bfloat16, T=64, H=37, w_mean=1.0, w_std=0.1, off=0),
    # the decode width with the FP8 epilogue: two vectors per thread, 5 warps per row
    "h2560_T64": dict(dtype=torch.bfloat16, T=64, H=2560, w_mean=1.0, w_std=0.02, off=0,
                      outliers=0.001),
}


@pytest.mark.parametrize("name", list(FP8_ROWS))
@pytest.mark.parametrize("fused", [True, False])
def test_rows_fp8(name, fused):
    run_rows(FP8_ROWS[name], fused, fp8=True)


# ---------------------------------------------------------------- gates

GLU_CASES = {
    # workload 2: decode gates [T, 2*9728], bf16, N(0,1)
    "cfg2_T1": dict(dtype=torch.bfloat16, T=1, d=9728, std=1.0),
    "cfg2_T4": dict(dtype=torch.bfloat16, T=4, d=9728, std=1.0),
    "cfg2_T64": dict(dtype=torch.bfloat16, T=64, d=9728, std=1.0),
    # workload 4: prefill gates, N(0,2), fp16 and bf16
    "cfg4_f16_I6912_T128": dict(dtype=torch.float16, T=128, d=6912, std=2.0),
    "cfg4_bf16_I10240_T512": dict(dtype=torch.bfloat16, T=512, d=10240, std=2.0),
    "cfg4_f16_I10240_T512": dict(dtype=torch.float16, T=512, d=10240, std=2.0),
    "f32_accurate": dict(dtype=torch.float32, T=33, d=1024, std=3.0),
    "generic_d37": dict(dtype=torch.bfloat16, T=21, d=37, std=2.0),
    "generic_misaligned": dict(dtype=torch.float16, T=7, d=1000, std=2.0, misalign=1),
    "wide_tail": dict(dtype=torch.bfloat16, T=3, d=8 * 1000 + 8, std=1.0),
}


def run_glu(c, act, fp8=False, seed=0):
    dtype, fmt = c["dtype"], TORCH_FMT[c["dtype"]]
    mk = lambda s: synth.glu_inputs(s, dtype, c["T"], c["d"], std=c["std"],
                                    outlier_frac=c.get("outliers", 0.0))
    inp = mk(seed)
    out_fmt = oracle.E4M3 if fp8 else fmt
    inv = 1.0
    if fp8:
        _, pre = oracle.glu_act(storage(mk(1)["gate_up"]), fmt, act)
        inv = calib_inv(pre)
    ref, pre = oracle.glu_act(storage(inp["gate_up"]), fmt, act, out_fmt, inv)
    mis = c.get("misalign", 0)
    gu = dev(inp["gate_up"], mis)
    g = Guarded((c["T"], c["d"]), torch.uint8 if fp8 else dtype, mis)
    edge_ops.glu_act(gu, act, out=g.t, fp8=fp8, inv_scale=inv)
    torch.cuda.synchronize()
    g.check()
    gate = oracle.decode(storage(inp["gate_up"]), fmt)[:, :c["d"]]
    eta = gate_eta(gate, act)
    check_out("glu", storage(g.t.cpu()), ref, pre, np.abs(pre), fmt, out_fmt, eta, inv)


@pytest.mark.parametrize("name", list(GLU_CASES))
@pytest.mark.parametrize("act", [oracle.SILU, oracle.GELU_TANH])
def test_glu(name, act):
    run_glu(GLU_CASES[name], act)


# (g, u) pairs at the edges of each dtype's range.  Where the logistic argument
# v is past 200 (sigma exactly 0 or 1 in fp32) or the exact result underflows
# to zero, the output must match the oracle bit for bit (signed zeros
# included); the others take the gate band.  (-3e38, 3e38) and (-1e20, 1e20)
# would give inf * 0 = NaN if g * u were formed before sigma.  e^-|v| stays an
# fp32 normal wherever a result is representable and nonzero.
GLU_EXTREMES = {
    torch.bfloat16: [(-1e20, 1e20), (1e20, 1e18), (-1e20, -1e20), (1e20, -1e18), (-3e38, 1.0),
                     (-3e38, 3e38), (3e38, 1.0), (0.0, 3e38), (-0.0, 5.0), (-60.0, 1e30),
                     (-80.0, 1e35), (100.0, 1e30), (-1e5, 1e33), (1e-30, 1e-30), (-200.0, 3.0),
                     (-3.0, 1e30)],
    torch.float16: [(-6e4, 6e4), (6e4, 1.0), (-6e4, -6e4), (-20.0, 6e4), (-9.0, 6e4), (0.0, 6e4),
                    (-0.0, 5.0), (100.0, 600.0), (-1e4, 6e4), (1e-7, 1e-7), (15.0, 4000.0),
                    (-15.0, 4000.0), (-60.0, 6e4), (-3.0, 6e4), (30.0, -2000.0), (-30.0, 2000.0)],
}
GLU_EXTREMES[torch.float32] = GLU_EXTREMES[torch.bfloat16]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("act", [oracle.SILU, oracle.GELU_TANH])
@pytest.mark.parametrize("extra", [0, 1])
def test_glu_extremes(dtype, act, extra):
    # extra = 1 adds a seventeenth pair, which takes the scalar kernel
    pairs = GLU_EXTREMES[dtype] + [(1.0, 1.0)] * extra
    d = len(pairs)
    g = torch.tensor([p[0] for p in pairs], dtype=torch.float64)
    u = torch.tensor([p[1] for p in pairs], dtype=torch.float64)
    gu = torch.cat([g, u]).to(dtype).view(1, 2 * d)
    fmt = TORCH_FMT[dtype]
    ref, pre = oracle.glu_act(storage(gu), fmt, act)
    out = Guarded((1, d), dtype)
    edge_ops.glu_act(gu.cuda(), act, out=out.t)
    torch.cuda.synchronize()
    out.check()
    got = storage(out.t.cpu())
    gv = oracle.decode(storage(gu), fmt)[:, :d]
    v = gv if act == oracle.SILU else \
        2.0 * math.sqrt(2.0 / math.pi) * (gv + 0.044715 * gv ** 3)
    exact = (np.abs(v) >= 200.0) | (oracle.decode(ref, fmt) == 0.0)
    assert np.array_equal(got[exact], ref[exact]), report("glu extremes (exact)", got == ref)
    check_out("glu extremes", got[~exact], ref[~exact], pre[~exact], np.abs(pre[~exact]), fmt,
              fmt, gate_eta(gv[~exact], act))


FP8_GLU = {
    # workload 5: GELU-tanh gate [T, 2D] with FP8 output, D in {2048, 1024}, T=512
    "cfg5_d2048": dict(dtype=torch.bfloat16, T=512, d=2048, std=1.0, outliers=0.001),
    "cfg5_d1024": dict(dtype=torch.bfloat16, T=512, d=1024, std=1.0, outliers=0.001),
    "cfg5_d2048_T4096": dict(dtype=torch.bfloat16, T=4096, d=2048, std=1.0, outliers=0.001),
    "generic_d37": dict(dtype=torch.bfloat16, T=21, d=37, std=2.0),
    "f32_d256": dict(dtype=torch.float32, T=9, d=256, std=2.0),
}


@pytest.mark.parametrize("name", list(FP8_GLU))
@pytest.mark.parametrize("act", [oracle.SILU, oracle.GELU_TANH])
def test_glu_fp8(name, act):
    run_glu(FP8_GLU[name], act, fp8=True)


# ---------------------------------------------------------------- misc

def test_invalid_call_raises_and_launches_nothing():
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    # an FP8 output cannot be written in place over its input
    with pytest.raises(edge_ops.EdgeError, match="ALIAS"):
        edge_ops.rmsnorm(x, None, out=x, fp8=True, inv_scale=1.0)
    assert torch.count_nonzero(x) == 0


def test_runs_on_a_side_stream_and_in_a_cuda_graph():
    c = QK_CASES["cfg3_24_4_T8"]
    inp = synth.qk_inputs(0, torch.bfloat16, 8, 24, 4, 256, 64, theta=1e7, cache_len=32768,
                          positions="offset", w_std=0.05)
    q, k, wq, wk = (dev(inp[n]) for n in ("q", "k", "wq", "wk"))
    pos, cs, sn = dev(inp["positions"]), dev(inp["cos"]), dev(inp["sin"])
    qo, ko = torch.empty_like(q), torch.empty_like(k)
    ref_q, ref_k = edge_ops.qk_norm_rope(q, k, wq, wk, pos, cs, sn, rotary_dim=64,
                                         weight_offset=1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        edge_ops.qk_norm_rope(q, k, wq, wk, pos, cs, sn, rotary_dim=64, weight_offset=1,
                              q_out=qo, k_out=ko)
    torch.cuda.synchronize()
    assert torch.equal(qo, ref_q) and torch.equal(ko, ref_k)
    qo.zero_()
    ko.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        edge_ops.qk_norm_rope(q, k, wq, wk, pos, cs, sn, rotary_dim=64, weight_offset=1,
                              q_out=qo, k_out=ko)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(qo, ref_q) and torch.equal(ko, ref_k)
    assert c["T"] == 8


# ---------------------------------------------------------------- standalone rotary

ROPE_CASES = {
    "bf16_partial_rotate_half": dict(dtype=torch.bfloat16, T=37, Hq=16, Hk=2, D=256, rot=64,
                                     layout=0, P=64, positions=np.r_[np.arange(34), [64, -1, 63]]),
    "f16_full_interleaved_in_place": dict(dtype=torch.float16, T=19, Hq=16, Hk=8, D=256, rot=256,
                                          layout=1, P=4096, positions="arange", inplace=True),
    "f32_full_rotate_half": dict(dtype=torch.float32, T=5, Hq=8, Hk=2, D=128, rot=128, layout=0,
                                 P=4096, positions="cfg_out_of_cache"),
    "many_heads_bf16": dict(dtype=torch.bfloat16, T=900, Hq=24, Hk=4, D=256, rot=64, layout=0,
                            P=32768, positions="offset"),
    "mid_heads_two_vectors": dict(dtype=torch.bfloat16, T=128, Hq=24, Hk=4, D=256, rot=64,
                                  layout=0, P=32768, positions="offset"),
    "many_heads_interleaved": dict(dtype=torch.bfloat16, T=1000, Hq=16, Hk=8, D=256, rot=256,
                                   layout=1, P=4096, positions="arange"),
    "generic_d96": dict(dtype=torch.bfloat16, T=9, Hq=3, Hk=1, D=96, rot=40, layout=0, P=16,
                        positions="arange"),
    "no_k": dict(dtype=torch.bfloat16, T=7, Hq=4, Hk=0, D=128, rot=64, layout=0, P=16,
                 positions="arange"),
}


def run_rope(c, fp8=False):
    dtype, fmt = c["dtype"], TORCH_FMT[c["dtype"]]
    inp = synth.qk_inputs(0, dtype, c["T"], c["Hq"], c["Hk"], c["D"], c["rot"], theta=1e6,
                          cache_len=c["P"], positions=c["positions"])
    out_fmt = oracle.E4M3 if fp8 else fmt
    inv = 448.0 / 6.0
    pos, cs, sn = inp["positions"].numpy(), storage(inp["cos"]), storage(inp["sin"])
    refs = [oracle.rope(storage(inp[n]), fmt, c["rot"], c["layout"], pos, cs, sn,
                        out_fmt=out_fmt, inv_scale=inv, diagnostics=True) for n in ("q", "k")]
    q, k = dev(inp["q"]), dev(inp["k"])
    odt = torch.uint8 if fp8 else dtype
    if c.get("inplace") and not fp8:
        gq, gk = Guarded(q.shape, dtype), Guarded(k.shape, dtype)
        gq.t.copy_(q)
        gk.t.copy_(k)
        q, k = gq.t, gk.t
    else:
        gq, gk = Guarded(q.shape, odt), Guarded(k.shape, odt)
    edge_ops.rope(q, k, dev(inp["positions"]), dev(inp["cos"]), dev(inp["sin"]),
                  rotary_dim=c["rot"], layout=c["layout"], q_out=gq.t, k_out=gk.t, fp8=fp8,
                  inv_scale=inv, cache_len=c["P"])
    torch.cuda.synchronize()
    gq.check()
    gk.check()
    for name, g, (ref, pre, mag) in (("q", gq, refs[0]), ("k", gk, refs[1])):
        if ref.size:
            check_out(name, storage(g.t.cpu()), ref, pre, mag, fmt, out_fmt, ETA_NORM, inv)


@pytest.mark.parametrize("name", list(ROPE_CASES))
def test_rope(name):
    run_rope(ROPE_CASES[name])


@pytest.mark.parametrize("name", ["bf16_partial_rotate_half", "many_heads_interleaved",
                                  "f32_full_rotate_half", "mid_heads_two_vectors"])
def test_rope_fp8(name):
    run_rope(ROPE_CASES[name], fp8=True)


# ---------------------------------------------------------------- review variant

@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("name", ["cfg3_16_2_T333", "cfg4_bf16", "cfg1_f32", "generic_rot24",
                                  "quad_cfg4_interleaved", "d128_bf16", "generic_odd_d37",
                                  "quad_no_weight", "dflash2_W16_B32"])
def test_qk_norm_rope_unrounded(name, fp8):
    # rotation of the fp32 normalized value, one rounding (ninfer review,
    # item 1); quad_no_weight and dflash2_W16_B32 take four threads per head
    c = QK_CASES[name]
    dtype, fmt = c["dtype"], TORCH_FMT[c["dtype"]]
    inp = synth.qk_inputs(0, dtype, c["T"], c["Hq"], c["Hk"], c["D"], c["rot"],
                          theta=c["theta"], cache_len=c["P"], positions=c["positions"],
                          w_mean=c["w_mean"] or 0.0, w_std=c["w_std"])
    wq = None if inp["wq"] is None or c["w_mean"] is None else storage(inp["wq"])
    wk = None if inp["wk"] is None or c["w_mean"] is None else storage(inp["wk"])
    inv = 40.0 if fp8 else 1.0
    ref = oracle.qk_norm_rope(storage(inp["q"]), storage(inp["k"]), wq, wk, fmt, c["rot"],
                              c["layout"], inp["positions"].numpy(), storage(inp["cos"]),
                              storage(inp["sin"]), 1e-6, c["offset"],
                              out_fmt=oracle.E4M3 if fp8 else fmt, inv_scale=inv, eta=ETA_NORM,
                              unrounded=True)
    d = {n: dev(inp[n]) for n in ("q", "k", "positions", "cos", "sin")}
    dwq = None if wq is None else dev(inp["wq"])
    dwk = None if wk is None else dev(inp["wk"])
    qo, ko = edge_ops.qk_norm_rope(d["q"], d["k"], dwq, dwk, d["positions"], d["cos"],
                                   d["sin"], rotary_dim=c["rot"], layout=c["layout"], eps=1e-6,
                                   weight_offset=c["offset"], cache_len=c["P"], unrounded=True,
                                   fp8=fp8, inv_scale=inv)
    torch.cuda.synchronize()
    if fp8:
        check_fp8_out(name + " q", qo.cpu().numpy(), ref.q_lo, ref.q_hi, ref.q_mag, ETA_NORM, inv)
        check_fp8_out(name + " k", ko.cpu().numpy(), ref.k_lo, ref.k_hi, ref.k_mag, ETA_NORM, inv)
        return
    check_out(name + " q", storage(qo.cpu()), ref.q_out, ref.q_pre, ref.q_mag, fmt, fmt,
              ETA_NORM, lo=ref.q_lo, hi=ref.q_hi)
    check_out(name + " k", storage(ko.cpu()), ref.k_out, ref.k_pre, ref.k_mag, fmt, fmt,
              ETA_NORM, lo=ref.k_lo, hi=ref.k_hi)


# ---------------------------------------------------------------- LayerNorm and static quantize

LN_CASES = {
    "siglip_bf16_h1152_T512": dict(dtype=torch.bfloat16, T=512, H=1152, affine=True),
    "bf16_h2048_T3_noaffine": dict(dtype=torch.bfloat16, T=3, H=2048, affine=False),
    "f32_h1024_T77": dict(dtype=torch.float32, T=77, H=1024, affine=True),
    "f16_h37_generic": dict(dtype=torch.float16, T=40, H=37, affine=True),
    "bf16_h1000_misaligned": dict(dtype=torch.bfloat16, T=9, H=1000, affine=True, misalign=1),
    "bf16_h16384_T2": dict(dtype=torch.bfloat16, T=2, H=16384, affine=True),
    # one warp per row (<= 256 vectors, many rows): 1, 4, 5 and 8 vectors per
    # lane; several warps per row for few rows or longer rows
    "bf16_h256_T1000": dict(dtype=torch.bfloat16, T=1000, H=256, affine=True),
    "f16_h1024_T1000": dict(dtype=torch.float16, T=1000, H=1024, affine=True),
    "siglip_bf16_h1152_T1000": dict(dtype=torch.bfloat16, T=1000, H=1152, affine=True),
    "bf16_h2048_T1600_noaffine": dict(dtype=torch.bfloat16, T=1600, H=2048, affine=False),
    "f16_h640_T33": dict(dtype=torch.float16, T=33, H=640, affine=True),
    "bf16_h4096_T300": dict(dtype=torch.bfloat16, T=300, H=4096, affine=True),
}


def run_ln(c, fp8=False, inplace=False):
    dtype, fmt = c["dtype"], TORCH_FMT[c["dtype"]]
    rng = np.random.default_rng(31)
    x = synth.to_dtype(synth.normal(0, 41, c["T"] * c["H"], 0.7, 2.0), dtype).view(c["T"], c["H"])
    g = synth.to_dtype(synth.normal(0, 42, c["H"], 1.0, 0.1), dtype) if c["affine"] else None
    b = synth.to_dtype(synth.normal(0, 43, c["H"], 0.0, 0.1), dtype) if c["affine"] else None
    out_fmt = oracle.E4M3 if fp8 else fmt
    inv = 448.0 / 5.0
    ref, pre, mag = oracle.layernorm(storage(x), None if g is None else storage(g),
                                     None if b is None else storage(b), fmt, 1e-5, out_fmt, inv)
    mis = c.get("misalign", 0)
    xd, gd, bd = dev(x, mis), dev(g, mis), dev(b, mis)
    if inplace:
        gout = Guarded(xd.shape, dtype)
        gout.t.copy_(xd)
        xd = gout.t
    else:
        gout = Guarded(xd.shape, torch.uint8 if fp8 else dtype, mis)
    edge_ops.layernorm(xd, gd, bd, eps=1e-5, out=gout.t, fp8=fp8, inv_scale=inv)
    torch.cuda.synchronize()
    gout.check()
    check_out("layernorm", storage(gout.t.cpu()), ref, pre, mag, fmt, out_fmt, ETA_NORM, inv)
    del rng


@pytest.mark.parametrize("name", list(LN_CASES))
def test_layernorm(name):
    run_ln(LN_CASES[name])


@pytest.mark.parametrize("name", ["siglip_bf16_h1152_T512", "f16_h37_generic", "f16_h1024_T1000",
                                  "siglip_bf16_h1152_T1000", "bf16_h4096_T300"])
def test_layernorm_fp8_and_in_place(name):
    run_ln(LN_CASES[name], fp8=True)
    run_ln(LN_CASES[name], inplace=True)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("n,mis", [(1, 0), (8 * 1000 + 5, 0), (3 * 2 ** 20, 0),
                                   (8 * 131109 + 3, 0), (77, 1)])
def test_quantize_fp8(dtype, n, mis):
    fmt = TORCH_FMT[dtype]
    x = synth.to_dtype(synth.with_outliers(synth.normal(0, 51, n, 0.0, 1.0), 0, 52, 0.001, 20.0),
                       dtype)
    inv = float(np.float32(448.0 / 7.0))
    ref = oracle.quantize_static(storage(x), fmt, inv)
    xd = dev(x, mis)
    g = Guarded((n,), torch.uint8, mis)
    edge_ops.quantize_fp8(xd, inv, out=g.t)
    torch.cuda.synchronize()
    g.check()
    # exact: the input is exact in fp32, so both sides take the same fp32 decision
    assert np.array_equal(storage(g.t.cpu()), ref)


# ---------------------------------------------------------------- fused QKV split + KV-cache write

QKV_CASES = {
    "text_bf16_d256_16x2": dict(dtype=torch.bfloat16, T=37, Hq=16, Hk=2, D=256, rot=64, layout=0,
                                norm=True, offset=1, S=64),
    "qwen_bf16_d128_32x8": dict(dtype=torch.bfloat16, T=64, Hq=32, Hk=8, D=128, rot=128, layout=0,
                                norm=True, offset=0, S=100),
    "f16_interleaved": dict(dtype=torch.float16, T=9, Hq=8, Hk=4, D=256, rot=256, layout=1,
                            norm=True, offset=0, S=16),
    "f32_d128": dict(dtype=torch.float32, T=5, Hq=8, Hk=2, D=128, rot=128, layout=0, norm=True,
                     offset=1, S=8),
    "no_norm_d256_8x1": dict(dtype=torch.bfloat16, T=10, Hq=8, Hk=1, D=256, rot=256, layout=0,
                             norm=False, offset=0, S=12),
    "decode_T1": dict(dtype=torch.bfloat16, T=1, Hq=24, Hk=4, D=256, rot=64, layout=0, norm=True,
                      offset=1, S=4),
    "prefill_T2000": dict(dtype=torch.bfloat16, T=2000, Hq=16, Hk=2, D=256, rot=64, layout=0,
                          norm=True, offset=1, S=2048),
    # mid widths of the text-profile heads: two vectors per lane (0.49 and 1.32
    # of a one-vector wave)
    "two_vec_text_T150": dict(dtype=torch.bfloat16, T=150, Hq=16, Hk=2, D=256, rot=64, layout=0,
                              norm=True, offset=1, S=256),
    "two_vec_f16_no_norm_T400": dict(dtype=torch.float16, T=400, Hq=16, Hk=2, D=256, rot=128,
                                     layout=0, norm=False, offset=0, S=512),
    # many heads (the lane-group grid is over a wave): four threads per head
    "quad_qwen_d128_T1000": dict(dtype=torch.bfloat16, T=1000, Hq=32, Hk=8, D=128, rot=128,
                                 layout=0, norm=True, offset=0, S=1024),
    "quad_f16_interleaved_d128": dict(dtype=torch.float16, T=700, Hq=16, Hk=4, D=128, rot=64,
                                      layout=1, norm=True, offset=1, S=700),
    "quad_f32_d64_no_norm": dict(dtype=torch.float32, T=2000, Hq=8, Hk=2, D=64, rot=64, layout=0,
                                 norm=False, offset=0, S=2000),
    "quad_no_cache_T1500": dict(dtype=torch.bfloat16, T=1500, Hq=16, Hk=2, D=256, rot=64,
                                layout=0, norm=True, offset=1, S=0),
    # no cache given (kv_heads > 0, num_slots 0, slots and caches NULL): q only
    "no_cache": dict(dtype=torch.bfloat16, T=12, Hq=8, Hk=2, D=128, rot=128, layout=0,
                     norm=True, offset=1, S=0),
    # the scalar path: head sizes that are no power-of-two number of vectors,
    # odd sizes, ragged rotary, misaligned tensors
    "generic_d96": dict(dtype=torch.bfloat16, T=7, Hq=4, Hk=1, D=96, rot=96, layout=0, norm=True,
                        offset=1, S=8),
    "generic_odd_d37_f16": dict(dtype=torch.float16, T=6, Hq=3, Hk=2, D=37, rot=20, layout=1,
                                norm=True, offset=0, S=7),
    "generic_f32_rot24": dict(dtype=torch.float32, T=5, Hq=4, Hk=2, D=256, rot=24, layout=0,
                              norm=False, offset=0, S=6),
    "generic_misaligned": dict(dtype=torch.bfloat16, T=9, Hq=16, Hk=2, D=256, rot=64, layout=0,
                               norm=True, offset=1, S=16, misalign=1),
}


def run_qkv(c):
    dtype, fmt = c["dtype"], TORCH_FMT[c["dtype"]]
    T, Hq, Hk, D, S = c["T"], c["Hq"], c["Hk"], c["D"], c["S"]
    qkv = synth.to_dtype(synth.normal(0, 71, T * (Hq + 2 * Hk) * D), dtype).view(T, -1)
    wq = synth.to_dtype(synth.normal(0, 72, D, 0.0 if c["offset"] else 1.0, 0.05), dtype)
    wk = synth.to_dtype(synth.normal(0, 73, D, 0.0 if c["offset"] else 1.0, 0.05), dtype)
    P = 4096
    cos, sin = synth.rope_cache(1e6, c["rot"], P)
    pos = np.floor(synth.uniform(0, 74, T) * P).astype(np.int64)
    pos[T // 3] = P            # out of cache: normalized, not rotated
    # distinct slots (two tokens on one slot leave either row: unspecified)
    assert S == 0 or T <= S, "the case needs a slot per token"
    slots = np.arange(T, dtype=np.int64) % max(S, 1) if S else np.full(T, -1, np.int64)
    if T > 2:
        slots[1] = -1          # padding token: no cache write
        slots[2] = S + 5       # out of range: no cache write
    kc0 = synth.to_dtype(synth.normal(0, 75, S * Hk * D), dtype).view(S, Hk, D)
    vc0 = synth.to_dtype(synth.normal(0, 76, S * Hk * D), dtype).view(S, Hk, D)
    ref = oracle.qkv_rope_cache(storage(qkv), storage(wq), storage(wk), fmt, Hq, Hk, c["rot"],
                                c["layout"], pos, storage(cos), storage(sin), slots, storage(kc0),
                                storage(vc0), 1e-6, c["offset"], c["norm"], eta=ETA_NORM)
    mis = c.get("misalign", 0)
    qo = Guarded((T, Hq, D), dtype, mis)
    if S == 0:
        edge_ops.qkv_rope_cache(dev(qkv, mis), Hq, Hk, dev(wq, mis), dev(wk, mis),
                                dev(torch.from_numpy(pos)), dev(cos), dev(sin), None, None, None,
                                rotary_dim=c["rot"], layout=c["layout"], eps=1e-6,
                                weight_offset=c["offset"], normalize=c["norm"], q_out=qo.t)
        torch.cuda.synchronize()
        qo.check()
        check_out("q", storage(qo.t.cpu()), ref.q_out, ref.q_pre, ref.q_mag, fmt, fmt, ETA_NORM,
                  lo=ref.q_lo, hi=ref.q_hi)
        return
    kc = Guarded((S, Hk, D), dtype, mis)
    vc = Guarded((S, Hk, D), dtype, mis)
    kc.t.copy_(kc0)
    vc.t.copy_(vc0)
    edge_ops.qkv_rope_cache(dev(qkv, mis), Hq, Hk, dev(wq, mis), dev(wk, mis),
                            dev(torch.from_numpy(pos)), dev(cos), dev(sin),
                            dev(torch.from_numpy(slots)), kc.t, vc.t, rotary_dim=c["rot"],
                            layout=c["layout"], eps=1e-6, weight_offset=c["offset"],
                            normalize=c["norm"], q_out=qo.t)
    torch.cuda.synchronize()
    for g in (kc, vc, qo):
        g.check()
    check_out("q", storage(qo.t.cpu()), ref.q_out, ref.q_pre, ref.q_mag, fmt, fmt, ETA_NORM,
              lo=ref.q_lo, hi=ref.q_hi)
    gk, gv = storage(kc.t.cpu()), storage(vc.t.cpu())
    written = np.zeros(S, bool)
    written[slots[(slots >= 0) & (slots < S)]] = True
    # untouched rows keep their contents; value rows are exact copies
    assert np.array_equal(gk[~written], storage(kc0)[~written])
    assert np.array_equal(gv, ref.v_cache)
    if written.any():
        check_out("k_cache", gk[written], ref.k_cache[written], ref.k_pre[written],
                  ref.k_mag[written], fmt, fmt, ETA_NORM, lo=ref.k_lo[written],
                  hi=ref.k_hi[written])


@pytest.mark.parametrize("name", list(QKV_CASES))
def test_qkv_rope_cache(name):
    run_qkv(QKV_CASES[name])


# ---------------------------------------------------------------- the benchmark's step

def test_benchmark_decode_step_matches_oracle():
    # The benchmark's own step: 36 layers of seam ops on its per-layer buffers,
    # replayed once from its captured CUDA graph (the launch configuration the
    # benchmark times).  Capturing runs the step once eagerly, so layers 0 and
    # 35 are checked against the oracle applied to their state just before
    # the replay.
    import bench

    layers, sh = bench.build_layers(torch, synth, torch.device("cuda"), seed=0)
    stream = torch.cuda.Stream()

    def step():
        for L in layers:
            for _, fn in bench.layer_ops(edge_ops, L, sh):
                fn()
    graph = bench.capture(torch, step, stream)
    names = ("res", "q", "k", "mlp_out", "attn_out", "gate_up")
    checked = (0, len(layers) - 1)
    before = {i: {n: storage(getattr(layers[i], n).cpu()) for n in names} for i in checked}
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    fmt = oracle.BF16
    pos, cos, sin = (sh[n].cpu().numpy() for n in ("pos", "cos", "sin"))
    for i in checked:
        L, b = layers[i], before[i]
        h1, res1, pre1 = oracle.add_rmsnorm(b["mlp_out"], b["res"], storage(L.w_in.cpu()), fmt,
                                            bench.EPS)
        qk = oracle.qk_norm_rope(b["q"], b["k"], storage(L.wq.cpu()), storage(L.wk.cpu()), fmt,
                                 bench.HD, oracle.ROTATE_HALF, pos, cos, sin, bench.EPS, 0,
                                 eta=ETA_NORM)
        h2, res2, pre2 = oracle.add_rmsnorm(b["attn_out"], res1, storage(L.w_post.cpu()), fmt,
                                            bench.EPS)
        act, prea = oracle.glu_act(b["gate_up"], fmt, oracle.SILU)
        assert np.array_equal(storage(L.res.cpu()), res2), f"layer {i}: residual not bit-exact"
        check_out(f"layer {i} h1", storage(L.h1.cpu()), h1, pre1, np.abs(pre1), fmt, fmt,
                  ETA_NORM)
        check_out(f"layer {i} h2", storage(L.h2.cpu()), h2, pre2, np.abs(pre2), fmt, fmt,
                  ETA_NORM)
        check_out(f"layer {i} q", storage(L.q.cpu()), qk.q_out, qk.q_pre, qk.q_mag, fmt, fmt,
                  ETA_NORM, lo=qk.q_lo, hi=qk.q_hi)
        check_out(f"layer {i} k", storage(L.k.cpu()), qk.k_out, qk.k_pre, qk.k_mag, fmt, fmt,
                  ETA_NORM, lo=qk.k_lo, hi=qk.k_hi)
        gate = oracle.decode(b["gate_up"], fmt)[:, :bench.INTER]
        check_out(f"layer {i} act", storage(L.act.cpu()), act, prea, np.abs(prea), fmt, fmt,
                  gate_eta(gate, oracle.SILU))


# ---------------------------------------------------------------- the declared size limits

def test_rows_at_the_largest_row():
    # hidden = 2**24, the largest row the library takes (the scalar path, one
    # CTA per row, fp64 reductions)
    c = dict(dtype=torch.bfloat16, T=1, H=1 << 24, w_mean=1.0, w_std=0.02, off=0)
    run_rows(c, fused=True)
    run_rows(dict(c, w_mean=0.0, off=1), fused=False)


def test_layernorm_at_the_largest_row():
    run_ln(dict(dtype=torch.bfloat16, T=1, H=1 << 24, affine=True))


@pytest.mark.parametrize("c", [
    dict(dtype=torch.bfloat16, T=3, Hq=2, Hk=1, D=2048, rot=2048, layout=0, w_mean=0.0,
         w_std=0.1, offset=1, theta=1e4, P=16, positions="arange"),
    dict(dtype=torch.float16, T=2, Hq=1, Hk=2, D=2048, rot=1024, layout=1, w_mean=1.0,
         w_std=0.02, offset=0, theta=1e4, P=8, positions=np.array([3, 9])),
])
def test_qk_at_the_largest_head(c):
    # head_dim = 2048, the largest head the prologue takes
    ref, gq, gk, fmt, out_fmt, _ = run_qk(c)
    check_out("q", gq, ref.q_out, ref.q_pre, ref.q_mag, fmt, out_fmt, ETA_NORM, lo=ref.q_lo,
              hi=ref.q_hi)
    check_out("k", gk, ref.k_out, ref.k_pre, ref.k_mag, fmt, out_fmt, ETA_NORM, lo=ref.k_lo,
              hi=ref.k_hi)


def test_qkv_at_the_largest_head():
    run_qkv(dict(dtype=torch.bfloat16, T=3, Hq=2, Hk=1, D=2048, rot=1024, layout=0, norm=True,
                 offset=1, S=4))


# ---------------------------------------------------------------- yardstick copy

@pytest.mark.parametrize("nbytes,dst_off,src_off", [
    (16, 0, 0), (4096, 0, 0), (4096 + 7, 0, 0), ((1 << 20) + 48, 0, 0), ((1 << 22) + 5, 0, 0),
    (3001, 1, 3), (65536 + 9, 8, 8), (1, 0, 0)])
def test_copy_is_exact(nbytes, dst_off, src_off):
    # the measurements' yardstick: every byte copied, nothing written outside
    g = torch.Generator().manual_seed(nbytes)
    src_raw = torch.randint(0, 256, (nbytes + 32,), generator=g, dtype=torch.uint8).cuda()
    src = src_raw[src_off:src_off + nbytes]
    out = Guarded((nbytes,), torch.uint8, dst_off)
    edge_ops.copy(src, out=out.t)
    torch.cuda.synchronize()
    out.check()
    assert torch.equal(out.t.cpu(), src.cpu())
