"""Seeded synthetic inputs shaped like the decode-seam workloads.

Shared by the GPU path's tests and benchmark and by the CPU oracle's tests.
It draws inputs only and holds none of the operators' arithmetic.

Generator: counter-based SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", 2014).  Element i of stream s under seed S is
mix(key(S, s) + (i + 1) * golden).  Its top 53 bits give a uniform in (0, 1),
and Box-Muller turns pairs of uniforms into fp64 normals.  A value reaches its
dtype through numpy's fp64->fp32 cast and then torch's cast to the dtype.

The rotary cache is an input of the prologue too, because the caller owns
theta.  Row p, entry j holds cos and sin of p * theta^(-2j/rotary_dim) for
j < rotary_dim/2.  The angle is taken in fp64 and the result stored as fp32
(RoFormer frequencies over the rotary width, as partial rotary uses them).
"""
from __future__ import annotations

import math

import numpy as np
import torch

_MASK = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15


def _mix_int(z: int) -> int:
    z &= _MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
    return z ^ (z >> 31)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def raw_bits(seed: int, stream: int, n: int) -> np.ndarray:
    """n uint64 draws of stream ``stream`` under ``seed``."""
    key = _mix_int(_mix_int(seed * _GOLDEN + 0x632BE59BD9B4E019) ^ (stream * 0xD1B54A32D192ED03))
    i = np.arange(1, n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(key) + i * np.uint64(_GOLDEN))


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """n fp64 uniforms in the open interval (0, 1)."""
    b = raw_bits(seed, stream, n) >> np.uint64(11)
    return (b.astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """n fp64 draws of N(mean, std^2) by Box-Muller."""
    m = (n + 1) // 2
    u = uniform(seed, stream, 2 * m)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    t = 2.0 * math.pi * u[1::2]
    z = np.empty(2 * m)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    return mean + std * z[:n]


def to_dtype(x64: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    """fp64 draws -> CPU tensor of ``dtype`` (numpy to fp32, torch to dtype)."""
    t = torch.from_numpy(np.ascontiguousarray(x64, dtype=np.float32))
    return t.to(dtype).contiguous()


def with_outliers(x64: np.ndarray, seed: int, stream: int, frac: float, mult: float) -> np.ndarray:
    """Multiply a seeded fraction ``frac`` of the elements by ``mult``."""
    if frac <= 0.0:
        return x64
    pick = uniform(seed, stream, x64.size).reshape(x64.shape) < frac
    return np.where(pick, x64 * mult, x64)


def rope_cache(theta: float, rotary_dim: int, cache_len: int):
    """(cos, sin) fp32 tensors of shape [cache_len, rotary_dim // 2]."""
    half = rotary_dim // 2
    j = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * j / rotary_dim)
    ang = np.arange(cache_len, dtype=np.float64)[:, None] * inv_freq[None, :]
    cos = torch.from_numpy(np.cos(ang).astype(np.float32))
    sin = torch.from_numpy(np.sin(ang).astype(np.float32))
    return cos.contiguous(), sin.contiguous()


# Stream identifiers: one per drawn tensor, so that changing one shape leaves
# the others' values unchanged.
S_Q, S_K, S_WQ, S_WK, S_POS = 1, 2, 3, 4, 5
S_X, S_RES, S_W = 11, 12, 13
S_GU = 21
S_OUT_X, S_OUT_RES, S_OUT_GU = 31, 32, 33


def block_positions(seed: int, W: int, B: int, cache_len: int) -> np.ndarray:
    """Positions of B sequences of W consecutive tokens each, tokens ordered
    [B][W]: sequence b starts at a seeded offset in [0, cache_len - W]."""
    u = uniform(seed, S_POS, max(B, 1))
    off = np.floor(u[:B] * (cache_len - W + 1)).astype(np.int64)
    return (off[:, None] + np.arange(W, dtype=np.int64)[None, :]).reshape(-1)


def qk_inputs(seed, dtype, T, Hq, Hk, D, rotary_dim, *, theta, cache_len, positions,
              w_mean=0.0, w_std=0.1, x_std=1.0):
    """Inputs of the fused QK prologue.

    positions: an int64 array of length T, or one of "cfg_out_of_cache"
    (uniform in [0, cache_len) with the last token at cache_len), "offset"
    (a seeded offset in [0, cache_len - T] plus 0..T-1), "arange" (0..T-1) or
    "blocks:W" (T // W sequences of W consecutive tokens, block_positions).
    """
    q = to_dtype(normal(seed, S_Q, T * Hq * D, 0.0, x_std), dtype).view(T, Hq, D)
    k = to_dtype(normal(seed, S_K, T * Hk * D, 0.0, x_std), dtype).view(T, Hk, D)
    wq = to_dtype(normal(seed, S_WQ, D, w_mean, w_std), dtype)
    wk = to_dtype(normal(seed, S_WK, D, w_mean, w_std), dtype)
    if isinstance(positions, str):
        u = uniform(seed, S_POS, max(T, 1))
        if positions == "cfg_out_of_cache":
            pos = np.floor(u[:T] * cache_len).astype(np.int64)
            if T:
                pos[-1] = cache_len
        elif positions == "offset":
            off = int(np.floor(u[0] * (cache_len - T + 1)))
            pos = off + np.arange(T, dtype=np.int64)
        elif positions == "arange":
            pos = np.arange(T, dtype=np.int64)
        elif positions.startswith("blocks:"):
            W = int(positions.split(":", 1)[1])
            if W <= 0 or T % W:
                raise ValueError(positions)
            pos = block_positions(seed, W, T // W, cache_len)
        else:
            raise ValueError(positions)
    else:
        pos = np.asarray(positions, dtype=np.int64)
    cos, sin = rope_cache(theta, rotary_dim, cache_len) if rotary_dim else (None, None)
    return dict(q=q, k=k, wq=wq, wk=wk, positions=torch.from_numpy(pos.copy()), cos=cos, sin=sin)


def rows_inputs(seed, dtype, T, H, *, w_mean=1.0, w_std=0.02, residual=True, x_std=1.0,
                outlier_frac=0.0, outlier_mult=20.0):
    """Inputs of RMSNorm / residual-add RMSNorm: x [T, H], residual [T, H], w [H]."""
    x64 = with_outliers(normal(seed, S_X, T * H, 0.0, x_std), seed, S_OUT_X, outlier_frac,
                        outlier_mult)
    out = dict(x=to_dtype(x64, dtype).view(T, H),
               w=to_dtype(normal(seed, S_W, H, w_mean, w_std), dtype))
    if residual:
        r64 = with_outliers(normal(seed, S_RES, T * H, 0.0, x_std), seed, S_OUT_RES,
                            outlier_frac, outlier_mult)
        out["residual"] = to_dtype(r64, dtype).view(T, H)
    return out


def glu_inputs(seed, dtype, T, d, *, std=1.0, outlier_frac=0.0, outlier_mult=20.0):
    """Merged gate+up projection output [T, 2d], gate in the first half."""
    g64 = with_outliers(normal(seed, S_GU, T * 2 * d, 0.0, std), seed, S_OUT_GU, outlier_frac,
                        outlier_mult)
    return dict(gate_up=to_dtype(g64, dtype).view(T, 2 * d))
