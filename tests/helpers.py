"""Shared test helpers: dtype plumbing and the parity acceptance rules.

Acceptance rules (the GPU computes in fp32, the oracle in fp64):

* integer-like results (residual sums) are compared bit for bit;
* bf16/fp16 outputs must lie within 1 ulp of the oracle's rounded value;
* the strict check additionally requires every output to be a correct
  rounding of some value within ``eta * mag`` of the oracle's exact value
  (or of the interval of values an intermediate rounding at a near tie can
  lead to).  That is bit-exactness except near rounding boundaries, with a
  band ``eta`` derived from the fp32 error of the kernel;
* FP8 codes are held to the strict check (bit-exact outside the band);
* fp32 outputs must satisfy |y - pre| <= rel * mag (+ a tiny absolute floor).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TORCH_FMT = {torch.float32: oracle.F32, torch.float16: oracle.F16, torch.bfloat16: oracle.BF16}


def storage(t: torch.Tensor) -> np.ndarray:
    """Raw element storage of a CPU tensor, as the oracle takes it."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return t.view(torch.uint8).numpy()
    raise TypeError(t.dtype)


def ordered(bits: np.ndarray, fmt: int) -> np.ndarray:
    """Map bit patterns to integers whose order is the value order (for ulp distances)."""
    if fmt == oracle.F32:
        b = bits.view(np.uint32).astype(np.int64)
        sign = b >> 31
        mag = b & 0x7FFFFFFF
    elif fmt == oracle.E4M3:
        b = bits.astype(np.int64)
        sign = b >> 7
        mag = b & 0x7F
    else:
        b = bits.astype(np.int64)
        sign = b >> 15
        mag = b & 0x7FFF
    return np.where(sign == 1, -mag, mag)


def ulp_distance(a: np.ndarray, b: np.ndarray, fmt: int) -> np.ndarray:
    return np.abs(ordered(a, fmt) - ordered(b, fmt))


_MANT = {oracle.F16: 10, oracle.BF16: 7, oracle.E4M3: 3, oracle.F32: 23}
_EMIN = {oracle.F16: -14, oracle.BF16: -126, oracle.E4M3: -6, oracle.F32: -126}


def ulp_at(x: np.ndarray, fmt: int) -> np.ndarray:
    """Spacing of format ``fmt`` at magnitude x (the subnormal spacing below the normals)."""
    x = np.abs(np.asarray(x, np.float64))
    e = np.where(x > 0, np.floor(np.log2(np.where(x > 0, x, 1.0))), _EMIN[fmt])
    e = np.maximum(e, _EMIN[fmt])
    return np.ldexp(1.0, (e - _MANT[fmt]).astype(np.int64))


def within_one_ulp(got: np.ndarray, ref: np.ndarray, mag: np.ndarray, fmt: int) -> np.ndarray:
    """|got - ref| <= one ulp of the format at max(|ref|, mag).  For a rotated
    channel mag is the pair norm, which absorbs the cancellation of a c - b s."""
    g = oracle.decode(got, fmt)
    r = oracle.decode(ref, fmt)
    return np.abs(g - r) <= ulp_at(np.maximum(np.abs(r), mag), fmt)


def _round_codes(v: np.ndarray, out_fmt: int, inv_scale: float) -> np.ndarray:
    if out_fmt == oracle.E4M3:
        return oracle.quantize(v, inv_scale)
    return oracle.encode(v, out_fmt)


def strict_ok(got: np.ndarray, lo: np.ndarray, hi: np.ndarray, mag: np.ndarray, out_fmt: int,
              eta, inv_scale: float = 1.0) -> np.ndarray:
    """Per element: got is the rounding of some value in
    [lo - eta*mag, hi + eta*mag].  lo = hi = the exact value, except where an
    intermediate rounding sat at a near tie (then [lo, hi] spans the
    candidates).  Rounding is monotone, so it suffices to bracket the ends."""
    got_o = ordered(got, out_fmt)
    a = ordered(_round_codes(lo - eta * mag, out_fmt, inv_scale), out_fmt)
    b = ordered(_round_codes(hi + eta * mag, out_fmt, inv_scale), out_fmt)
    return (got_o >= np.minimum(a, b)) & (got_o <= np.maximum(a, b))


def f32_ok(got: np.ndarray, pre: np.ndarray, mag: np.ndarray, rel: float,
           floor: float = 1e-30) -> np.ndarray:
    g = got.view(np.float32).astype(np.float64)
    return np.abs(g - pre) <= rel * mag + floor


def report(name: str, ok: np.ndarray) -> str:
    bad = np.flatnonzero(~ok.ravel())
    return f"{name}: {bad.size} of {ok.size} outside tolerance; first at {bad[:8].tolist()}"


def position_delta_bf16(old, new):
    """bf16 words that a residual add turns `old` positions into `new` ones.

    An int64 position k < 256 is the little-endian words [k, 0, 0, 0], and the
    bf16 word k is the value k * 2^-133 (subnormal below 128, exponent 1 from
    128 to 255).  So adding the words [new - old, 0, 0, 0] in fp32 gives the
    new position exactly."""
    d = (new - old).astype(np.int64)
    w = np.zeros((len(old), 4), np.uint16)
    w[:, 0] = np.where(d >= 0, d, 0x8000 | -d).astype(np.uint16)
    return torch.from_numpy(w.reshape(-1).view(np.int16).copy()).view(torch.bfloat16).view(1, -1)
