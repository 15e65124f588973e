"""CPU oracle for the fused decode-seam operators -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``edge_oracle.c`` (plain C, fp64 scalar loops, no
fast-math).  This module compiles it with the host C compiler and wraps it with
ctypes over numpy arrays.  It shares no code with the CUDA library and never
imports it.  Only the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may use it; the product path never does.

Arrays hold raw element storage: ``float32`` for binary32, ``uint16`` for
binary16 and bfloat16, ``uint8`` for E4M3 codes.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess

import numpy as np

F32, F16, BF16, E4M3 = 0, 1, 2, 3
ROTATE_HALF, INTERLEAVED = 0, 1
SILU, GELU_TANH = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "edge_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = None

STORAGE = {F32: np.float32, F16: np.uint16, BF16: np.uint16, E4M3: np.uint8}


def lib_path() -> str:
    return os.path.join(_OUT_DIR, f"liboracle_{platform.machine()}.so")


def build(force: bool = False) -> str:
    """Compile the oracle for this host (x86_64 here, aarch64 on the GPU host)."""
    out = lib_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = [os.environ.get("CC", "cc"), "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib():
    global _LIB
    if _LIB is None:
        L = ctypes.CDLL(build())
        P, I64, I, F, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_double
        L.oracle_round.argtypes = [D, I]
        L.oracle_round.restype = D
        L.oracle_bits.argtypes = [D, I]
        L.oracle_bits.restype = ctypes.c_uint32
        L.oracle_value.argtypes = [ctypes.c_uint32, I]
        L.oracle_value.restype = D
        L.oracle_decode_array.argtypes = [P, I, I64, P]
        L.oracle_encode_array.argtypes = [P, I64, I, P]
        L.oracle_quantize_array.argtypes = [P, I64, F, P]
        L.oracle_rmsnorm.argtypes = [P, I, P, P, P, I, I64, I64, F, I, F]
        L.oracle_add_rmsnorm.argtypes = [P, I, P, P, P, P, P, I, I64, I64, F, I, F]
        L.oracle_glu_act.argtypes = [P, I, P, P, I, I64, I64, I, F]
        L.oracle_rope.argtypes = [P, I, P, P, P, I, I64, I, I, I, I, P, P, P, I64, F]
        L.oracle_qk_norm_rope.argtypes = [P, P, I, P, P, P, P, P, P, P, P, P, P, P, P, I, I64, I,
                                          I, I, I, I, P, P, P, I64, F, I, F, D, I]
        L.oracle_layernorm.argtypes = [P, I, P, P, P, P, P, I, I64, I64, F, F]
        L.oracle_quantize_static.argtypes = [P, P, I, I64, F]
        L.oracle_qkv_rope_cache.argtypes = [P] * 14 + [I, I64, I, I, I, I, I, P, P, P, I64, P, I64,
                                                         F, I, I, D]
        L.oracle_set_rotation_scale.argtypes = [D]
        L.oracle_near_tie.argtypes = [D, I, D, ctypes.POINTER(D)]
        L.oracle_near_tie.restype = ctypes.c_int
        for name in ("oracle_rmsnorm", "oracle_add_rmsnorm", "oracle_glu_act", "oracle_rope",
                     "oracle_qk_norm_rope", "oracle_layernorm", "oracle_quantize_static",
                     "oracle_qkv_rope_cache",
                     "oracle_version"):
            getattr(L, name).restype = ctypes.c_int
        _LIB = L
    return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if dtype is not None and a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (rc={rc})")


# ---------------------------------------------------------------- formats

def round_to(v, fmt: int) -> float:
    """Round one fp64 value to ``fmt`` (nearest, ties to even)."""
    return _lib().oracle_round(float(v), fmt)


def bits_of(v, fmt: int) -> int:
    return int(_lib().oracle_bits(float(v), fmt))


def value_of(bits: int, fmt: int) -> float:
    return _lib().oracle_value(int(bits), fmt)


def near_tie(v, fmt: int, eta: float):
    """The tie policy's decision for one exact value: (flagged, other), where
    flagged says the rounding of v to fmt lies within the relative band eta of
    a rounding boundary and other is the neighbour across it (v's own rounding
    when not flagged)."""
    o = ctypes.c_double(0.0)
    t = _lib().oracle_near_tie(float(v), fmt, float(eta), ctypes.byref(o))
    return bool(t), o.value


def decode(a: np.ndarray, fmt: int) -> np.ndarray:
    """Raw element storage -> fp64 values."""
    a = _c(a, STORAGE[fmt])
    out = np.empty(a.shape, np.float64)
    _lib().oracle_decode_array(_ptr(a), fmt, a.size, _ptr(out))
    return out


def encode(v: np.ndarray, fmt: int) -> np.ndarray:
    """fp64 values -> raw storage of their rounding to ``fmt``."""
    v = _c(np.asarray(v, np.float64))
    out = np.empty(v.shape, STORAGE[fmt])
    _lib().oracle_encode_array(_ptr(v), v.size, fmt, _ptr(out))
    return out


def quantize(v: np.ndarray, inv_scale: float) -> np.ndarray:
    """Exact values -> the E4M3 codes the FP8 epilogue emits for them."""
    v = _c(np.asarray(v, np.float64))
    out = np.empty(v.shape, np.uint8)
    _lib().oracle_quantize_array(_ptr(v), v.size, ctypes.c_float(inv_scale), _ptr(out))
    return out


# ---------------------------------------------------------------- ops

def rmsnorm(x, w, fmt, eps, weight_offset=0, out_fmt=None, inv_scale=1.0):
    """x: [rows, hidden] storage.  Returns (out storage, exact pre-rounding values)."""
    out_fmt = fmt if out_fmt is None else out_fmt
    x = _c(x, STORAGE[fmt])
    w = _c(w, STORAGE[fmt])
    rows, hidden = x.shape
    out = np.empty(x.shape, STORAGE[out_fmt])
    pre = np.empty(x.shape, np.float64)
    rc = _lib().oracle_rmsnorm(_ptr(out), out_fmt, _ptr(pre), _ptr(x), _ptr(w), fmt, rows, hidden,
                               eps, weight_offset, inv_scale)
    _check(rc, "rmsnorm")
    return out, pre


def add_rmsnorm(x, residual, w, fmt, eps, weight_offset=0, out_fmt=None, inv_scale=1.0):
    """Returns (out storage, new residual storage, exact pre-rounding values)."""
    out_fmt = fmt if out_fmt is None else out_fmt
    x = _c(x, STORAGE[fmt])
    residual = _c(residual, STORAGE[fmt])
    w = _c(w, STORAGE[fmt])
    rows, hidden = x.shape
    out = np.empty(x.shape, STORAGE[out_fmt])
    res = np.empty(x.shape, STORAGE[fmt])
    pre = np.empty(x.shape, np.float64)
    rc = _lib().oracle_add_rmsnorm(_ptr(out), out_fmt, _ptr(pre), _ptr(res), _ptr(x),
                                   _ptr(residual), _ptr(w), fmt, rows, hidden, eps, weight_offset,
                                   inv_scale)
    _check(rc, "add_rmsnorm")
    return out, res, pre


def layernorm(x, gamma, beta, fmt, eps, out_fmt=None, inv_scale=1.0):
    """x: [rows, hidden] storage.  Returns (out storage, exact values, error scale)."""
    out_fmt = fmt if out_fmt is None else out_fmt
    x = _c(x, STORAGE[fmt])
    gamma = _c(gamma, STORAGE[fmt])
    beta = _c(beta, STORAGE[fmt])
    rows, hidden = x.shape
    out = np.empty(x.shape, STORAGE[out_fmt])
    pre = np.empty(x.shape)
    mag = np.empty(x.shape)
    rc = _lib().oracle_layernorm(_ptr(out), out_fmt, _ptr(pre), _ptr(mag), _ptr(x), _ptr(gamma),
                                 _ptr(beta), fmt, rows, hidden, eps, inv_scale)
    _check(rc, "layernorm")
    return out, pre, mag


def quantize_static(x, fmt, inv_scale):
    """E4M3 codes of a stored tensor under the static-scale epilogue."""
    x = _c(x, STORAGE[fmt])
    out = np.empty(x.shape, np.uint8)
    rc = _lib().oracle_quantize_static(_ptr(out), _ptr(x), fmt, x.size, ctypes.c_float(inv_scale))
    _check(rc, "quantize_static")
    return out


def glu_act(gate_up, fmt, act, out_fmt=None, inv_scale=1.0):
    """gate_up: [rows, 2d] storage (gate first).  Returns (out storage, exact values)."""
    out_fmt = fmt if out_fmt is None else out_fmt
    gate_up = _c(gate_up, STORAGE[fmt])
    rows, two_d = gate_up.shape
    d = two_d // 2
    out = np.empty((rows, d), STORAGE[out_fmt])
    pre = np.empty((rows, d), np.float64)
    rc = _lib().oracle_glu_act(_ptr(out), out_fmt, _ptr(pre), _ptr(gate_up), fmt, rows, d, act,
                               inv_scale)
    _check(rc, "glu_act")
    return out, pre


def rope(x, fmt, rotary_dim, layout, positions, cos, sin, out_fmt=None, inv_scale=1.0,
         cache_len=None, diagnostics=False):
    """Standalone rotary embedding of x: [tokens, heads, head_dim] storage.
    With diagnostics=True returns (out, pre, mag): the exact values before the
    output rounding and their error scale (the pair norm of rotated channels)."""
    out_fmt = fmt if out_fmt is None else out_fmt
    x = _c(x, STORAGE[fmt])
    tokens, heads, head_dim = x.shape
    positions = _c(np.asarray(positions, np.int64))
    cos = _c(cos, np.float32)
    sin = _c(sin, np.float32)
    if cache_len is None:
        cache_len = 0 if cos is None else cos.shape[0]
    out = np.empty(x.shape, STORAGE[out_fmt])
    pre = np.empty(x.shape) if diagnostics else None
    mag = np.empty(x.shape) if diagnostics else None
    rc = _lib().oracle_rope(_ptr(out), out_fmt, _ptr(pre), _ptr(mag), _ptr(x), fmt, tokens, heads,
                            head_dim, rotary_dim, layout, _ptr(positions), _ptr(cos), _ptr(sin),
                            cache_len, ctypes.c_float(inv_scale))
    _check(rc, "rope")
    return (out, pre, mag) if diagnostics else out


class QKResult:
    """Outputs of the fused prologue plus the tie-policy diagnostics."""

    def __init__(self, **kw):
        self.__dict__.update(kw)


def qk_norm_rope(q, k, wq, wk, fmt, rotary_dim, layout, positions, cos, sin, eps,
                 weight_offset=0, out_fmt=None, inv_scale=1.0, eta=2.0 ** -20, cache_len=None,
                 unrounded=False):
    """q: [T, Hq, D], k: [T, Hk, D] storage; cos/sin: [P, rotary_dim/2] fp32.

    Besides the outputs, returns per element the exact pre-rounding value
    (q_pre, k_pre), its bounds over the near-tie neighbours of the
    intermediate roundings (q_lo/q_hi, k_lo/k_hi; band eta, relative) and the
    error scale (q_mag, k_mag: the pair norm for rotated channels)."""
    out_fmt = fmt if out_fmt is None else out_fmt
    q = _c(q, STORAGE[fmt])
    k = _c(k, STORAGE[fmt])
    wq = _c(wq, STORAGE[fmt])
    wk = _c(wk, STORAGE[fmt])
    T, Hq, D = q.shape
    Hk = k.shape[1]
    positions = _c(np.asarray(positions, np.int64))
    cos = _c(cos, np.float32)
    sin = _c(sin, np.float32)
    if cache_len is None:
        cache_len = 0 if cos is None else cos.shape[0]
    res = QKResult(
        q_out=np.empty(q.shape, STORAGE[out_fmt]), k_out=np.empty(k.shape, STORAGE[out_fmt]),
        q_pre=np.empty(q.shape), k_pre=np.empty(k.shape),
        q_lo=np.empty(q.shape), k_lo=np.empty(k.shape),
        q_hi=np.empty(q.shape), k_hi=np.empty(k.shape),
        q_mag=np.empty(q.shape), k_mag=np.empty(k.shape))
    rc = _lib().oracle_qk_norm_rope(
        _ptr(res.q_out), _ptr(res.k_out), out_fmt, _ptr(res.q_pre), _ptr(res.k_pre),
        _ptr(res.q_lo), _ptr(res.k_lo), _ptr(res.q_hi), _ptr(res.k_hi), _ptr(res.q_mag),
        _ptr(res.k_mag), _ptr(q), _ptr(k),
        _ptr(wq), _ptr(wk), fmt, T, Hq, Hk, D, rotary_dim, layout, _ptr(positions), _ptr(cos),
        _ptr(sin), cache_len, eps, weight_offset, inv_scale, eta, 1 if unrounded else 0)
    _check(rc, "qk_norm_rope")
    return res


def qkv_rope_cache(qkv, wq, wk, fmt, q_heads, kv_heads, rotary_dim, layout, positions, cos, sin,
                   slots, k_cache, v_cache, eps, weight_offset=0, normalize=True,
                   eta=2.0 ** -20, cache_len=None):
    """Fused QKV split + prologue + KV-cache write.  qkv: [T, (Hq + 2 Hk) D]
    storage; k_cache, v_cache: [S, Hk, D] storage, updated in copies (rows
    whose slot is invalid keep their contents).  Returns a QKResult with
    q_out, k_cache, v_cache and the diagnostics of q (q_*) and of the cache
    rows (k_*)."""
    qkv = _c(qkv, STORAGE[fmt])
    T = qkv.shape[0]
    D = qkv.shape[1] // (q_heads + 2 * kv_heads)
    positions = _c(np.asarray(positions, np.int64))
    slots = _c(np.asarray(slots, np.int64))
    cos = _c(cos, np.float32)
    sin = _c(sin, np.float32)
    if cache_len is None:
        cache_len = 0 if cos is None else cos.shape[0]
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    S = kc.shape[0]
    res = QKResult(q_out=np.empty((T, q_heads, D), STORAGE[fmt]), k_cache=kc, v_cache=vc,
                   q_pre=np.empty((T, q_heads, D)), q_lo=np.empty((T, q_heads, D)),
                   q_hi=np.empty((T, q_heads, D)), q_mag=np.empty((T, q_heads, D)),
                   k_pre=np.full(kc.shape, np.nan), k_lo=np.full(kc.shape, np.nan),
                   k_hi=np.full(kc.shape, np.nan), k_mag=np.full(kc.shape, np.nan))
    rc = _lib().oracle_qkv_rope_cache(
        _ptr(res.q_out), _ptr(kc), _ptr(vc), _ptr(res.q_pre), _ptr(res.q_lo), _ptr(res.q_hi),
        _ptr(res.q_mag), _ptr(res.k_pre), _ptr(res.k_lo), _ptr(res.k_hi), _ptr(res.k_mag),
        _ptr(qkv), _ptr(_c(wq, STORAGE[fmt])), _ptr(_c(wk, STORAGE[fmt])), fmt, T, q_heads,
        kv_heads, D, rotary_dim, layout, _ptr(positions), _ptr(cos), _ptr(sin), cache_len,
        _ptr(slots), S, eps, weight_offset, 1 if normalize else 0, eta)
    _check(rc, "qkv_rope_cache")
    return res


class rotation_scale:
    """Context manager that plants a factor into the oracle's rotation (the
    strength control of the ninfer text-profile pull request, "Output")."""

    def __init__(self, s: float):
        self.s = s

    def __enter__(self):
        _lib().oracle_set_rotation_scale(self.s)
        return self

    def __exit__(self, *exc):
        _lib().oracle_set_rotation_scale(1.0)
        return False
