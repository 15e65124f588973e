"""Thin ctypes binding over the C ABI of libedge_ops.so (include/edge_ops.h).

Argument marshalling only.  Every step of every op runs in the library's
CUDA kernels, and there is no CPU or eager fallback: if the library is
missing, the first call raises.  Torch is used for device memory, dtypes and
the current stream.  The binding allocates outputs through torch only when
the caller passes none.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

F32, F16, BF16, FP8_E4M3 = 0, 1, 2, 3
ROTATE_HALF, INTERLEAVED = 0, 1
SILU, GELU_TANH = 0, 1

STATUS = {
    0: "EDGE_OK", 1: "EDGE_ERR_NULL", 2: "EDGE_ERR_DTYPE", 3: "EDGE_ERR_SHAPE",
    4: "EDGE_ERR_ALIGN", 5: "EDGE_ERR_ALIAS", 6: "EDGE_ERR_UNSUPPORTED", 7: "EDGE_ERR_CUDA",
    8: "EDGE_ERR_VALUE",
}
EXPORTS = ("edge_rmsnorm", "edge_add_rmsnorm", "edge_glu_act", "edge_qk_norm_rope",
           "edge_qk_norm_rope_ex", "edge_rope", "edge_layernorm", "edge_quantize_fp8",
           "edge_qkv_rope_cache", "edge_copy",
           "edge_status_str", "edge_last_cuda_error", "edge_version")
QK_ROTATE_UNROUNDED = 1

_DT = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}
_LIB = None


class EdgeError(RuntimeError):
    def __init__(self, status: int, op: str):
        self.status = status
        msg = lib().edge_status_str(status).decode()
        extra = ""
        if status == 7:
            extra = f" (cudaError {lib().edge_last_cuda_error()})"
        super().__init__(f"{op}: {STATUS.get(status, status)}: {msg}{extra}")


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = False) -> ctypes.CDLL:
    """The loaded C ABI.  Raises if libedge_ops.so is absent (no fallback)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(
                f"libedge_ops.so is not built ({path}); run __graft_entry__.build() or "
                "python -m memory_bound_decode_qk_gb300._build")
        _build.build()
    L = ctypes.CDLL(path)
    P, I64, I32, I, F = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int,
                         ctypes.c_float)
    L.edge_rmsnorm.argtypes = [P, I, P, P, I, I64, I64, F, I, F, P]
    L.edge_add_rmsnorm.argtypes = [P, I, P, P, P, I, I64, I64, F, I, F, P]
    L.edge_glu_act.argtypes = [P, I, P, I, I64, I64, I, F, P]
    L.edge_qk_norm_rope.argtypes = [P, P, I, P, P, P, P, I, I64, I32, I32, I32, I32, I, P, P, P,
                                    I64, F, I, F, P]
    L.edge_qk_norm_rope_ex.argtypes = [P, P, I, P, P, P, P, I, I64, I32, I32, I32, I32, I, P, P,
                                       P, I64, F, I, F, ctypes.c_uint32, P]
    L.edge_rope.argtypes = [P, P, I, P, P, I, I64, I32, I32, I32, I32, I, P, P, P, I64, F, P]
    L.edge_layernorm.argtypes = [P, I, P, P, P, I, I64, I64, F, F, P]
    L.edge_quantize_fp8.argtypes = [P, P, I, I64, F, P]
    L.edge_qkv_rope_cache.argtypes = [P, P, P, P, P, P, I, I64, I32, I32, I32, I32, I, P, P, P,
                                      I64, P, I64, F, I, I, P]
    L.edge_copy.argtypes = [P, P, I64, P]
    for name in ("edge_rmsnorm", "edge_add_rmsnorm", "edge_glu_act", "edge_qk_norm_rope",
                 "edge_qk_norm_rope_ex", "edge_rope", "edge_layernorm", "edge_quantize_fp8",
                 "edge_qkv_rope_cache", "edge_copy"):
        getattr(L, name).restype = I
    L.edge_status_str.argtypes = [I]
    L.edge_status_str.restype = ctypes.c_char_p
    L.edge_last_cuda_error.restype = I
    L.edge_version.restype = I
    _LIB = L
    return L


def _ptr(t):
    return None if t is None else t.data_ptr()


# The current stream's raw handle without building a Stream object (about 2
# us cheaper per call); the public route where torch lacks it.
_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is None:
        if _RAW_STREAM is not None:
            return _RAW_STREAM(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _dt(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _out_dt(fp8: bool, dt: int) -> int:
    return FP8_E4M3 if fp8 else dt


def _check(st: int, op: str):
    if st != 0:
        raise EdgeError(st, op)


def _need_contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous (row-major)")


def _alloc(like: torch.Tensor, shape, fp8: bool):
    return torch.empty(shape, dtype=torch.uint8 if fp8 else like.dtype, device=like.device)


def rmsnorm(x, w=None, *, eps=1e-6, weight_offset=0, out=None, fp8=False, inv_scale=1.0,
            stream=None):
    """RMSNorm over the last dim of x ([rows, hidden])."""
    _need_contig(x, w, out)
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    if out is None:
        out = _alloc(x, x.shape, fp8)
    dt = _dt(x)
    _check(lib().edge_rmsnorm(_ptr(out), _out_dt(fp8, dt), _ptr(x), _ptr(w), dt, rows, hidden,
                              eps, weight_offset, inv_scale, _stream(stream)), "edge_rmsnorm")
    return out


def add_rmsnorm(x, residual, w=None, *, eps=1e-6, weight_offset=0, out=None, fp8=False,
                inv_scale=1.0, stream=None):
    """residual <- x + residual (rounded to the dtype); returns RMSNorm(residual)."""
    _need_contig(x, residual, w, out)
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    if out is None:
        out = _alloc(x, x.shape, fp8)
    dt = _dt(x)
    _check(lib().edge_add_rmsnorm(_ptr(out), _out_dt(fp8, dt), _ptr(x), _ptr(residual), _ptr(w),
                                  dt, rows, hidden, eps, weight_offset, inv_scale,
                                  _stream(stream)), "edge_add_rmsnorm")
    return out


def layernorm(x, gamma=None, beta=None, *, eps=1e-6, out=None, fp8=False, inv_scale=1.0,
              stream=None):
    """One-read LayerNorm over the last dim of x ([rows, hidden])."""
    _need_contig(x, gamma, beta, out)
    hidden = x.shape[-1]
    rows = x.numel() // hidden if hidden else 0
    if out is None:
        out = _alloc(x, x.shape, fp8)
    dt = _dt(x)
    _check(lib().edge_layernorm(_ptr(out), _out_dt(fp8, dt), _ptr(x), _ptr(gamma), _ptr(beta), dt,
                                rows, hidden, eps, inv_scale, _stream(stream)), "edge_layernorm")
    return out


def copy(src, *, out=None, stream=None):
    """The yardstick copy: src's bytes into out (a new tensor like src when
    None), in the operators' launch form.  Returns out."""
    _need_contig(src, out)
    if out is None:
        out = torch.empty_like(src)
    nbytes = src.numel() * src.element_size()
    if out.numel() * out.element_size() != nbytes:
        raise ValueError("copy: out must hold as many bytes as src")
    _check(lib().edge_copy(_ptr(out), _ptr(src), nbytes, _stream(stream)), "edge_copy")
    return out


def quantize_fp8(x, inv_scale, *, out=None, stream=None):
    """Static-scale E4M3 codes of x (any shape, contiguous); uint8 output."""
    _need_contig(x, out)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(lib().edge_quantize_fp8(_ptr(out), _ptr(x), _dt(x), x.numel(), inv_scale,
                                   _stream(stream)), "edge_quantize_fp8")
    return out


def qkv_rope_cache(qkv, q_heads, kv_heads, wq, wk, positions, cos, sin, slots, k_cache, v_cache,
                   *, rotary_dim=None, layout=ROTATE_HALF, eps=1e-6, weight_offset=0,
                   normalize=True, q_out=None, cache_len=None, stream=None):
    """Fused QKV split + prologue + KV-cache write.  qkv: [T, (Hq + 2 Hk) D];
    k_cache, v_cache: [S, Hk, D] (written at rows slots[t]).  Returns q_out."""
    _need_contig(qkv, wq, wk, positions, cos, sin, slots, k_cache, v_cache, q_out)
    T = qkv.shape[0]
    D = qkv.shape[-1] // (q_heads + 2 * kv_heads)
    if rotary_dim is None:
        rotary_dim = D if cos is None else 2 * cos.shape[-1]
    if cache_len is None:
        cache_len = 0 if cos is None else cos.shape[0]
    if isinstance(layout, str):
        layout = {"rotate_half": ROTATE_HALF, "interleaved": INTERLEAVED}[layout]
    if q_out is None:
        q_out = torch.empty((T, q_heads, D), dtype=qkv.dtype, device=qkv.device)
    S = k_cache.shape[0] if k_cache is not None else 0
    _check(lib().edge_qkv_rope_cache(_ptr(q_out), _ptr(k_cache), _ptr(v_cache), _ptr(qkv),
                                     _ptr(wq), _ptr(wk), _dt(qkv), T, q_heads, kv_heads, D,
                                     rotary_dim, layout, _ptr(positions), _ptr(cos), _ptr(sin),
                                     cache_len, _ptr(slots), S, eps, weight_offset,
                                     1 if normalize else 0, _stream(stream)), "edge_qkv_rope_cache")
    return q_out


def glu_act(gate_up, act=SILU, *, out=None, fp8=False, inv_scale=1.0, stream=None):
    """act(gate) * up for gate_up = [rows, 2d] (gate first); returns [rows, d]."""
    _need_contig(gate_up, out)
    two_d = gate_up.shape[-1]
    d = two_d // 2
    rows = gate_up.numel() // two_d if two_d else 0
    if isinstance(act, str):
        act = {"silu": SILU, "gelu_tanh": GELU_TANH}[act]
    if out is None:
        out = _alloc(gate_up, tuple(gate_up.shape[:-1]) + (d,), fp8)
    dt = _dt(gate_up)
    _check(lib().edge_glu_act(_ptr(out), _out_dt(fp8, dt), _ptr(gate_up), dt, rows, d, act,
                              inv_scale, _stream(stream)), "edge_glu_act")
    return out


def _qk_shapes(q, k, cos, rotary_dim, cache_len, layout, fp8, q_out, k_out):
    T, Hq, D = q.shape
    Hk = k.shape[1] if k is not None else 0
    if rotary_dim is None:
        rotary_dim = D if cos is None else 2 * cos.shape[-1]
    if cache_len is None:
        cache_len = 0 if cos is None else cos.shape[0]
    if isinstance(layout, str):
        layout = {"rotate_half": ROTATE_HALF, "interleaved": INTERLEAVED}[layout]
    if q_out is None:
        q_out = _alloc(q, q.shape, fp8)
    if k_out is None and k is not None:
        k_out = _alloc(k, k.shape, fp8)
    return T, Hq, Hk, D, rotary_dim, cache_len, layout, q_out, k_out


def qk_norm_rope(q, k, wq, wk, positions, cos, sin, *, rotary_dim=None, layout=ROTATE_HALF,
                 eps=1e-6, weight_offset=0, q_out=None, k_out=None, fp8=False, inv_scale=1.0,
                 cache_len=None, unrounded=False, stream=None):
    """Per-head QK-RMSNorm + RoPE.  q: [T, Hq, D], k: [T, Hk, D];
    cos/sin: [P, rotary_dim/2] fp32; positions: [T] int64.  Pass q_out=q and
    k_out=k for the in-place form.  unrounded=True rotates the fp32 normalized
    value (edge_qk_norm_rope_ex with EDGE_QK_ROTATE_UNROUNDED).  Returns
    (q_out, k_out)."""
    _need_contig(q, k, wq, wk, positions, cos, sin, q_out, k_out)
    T, Hq, Hk, D, rotary_dim, cache_len, layout, q_out, k_out = _qk_shapes(
        q, k, cos, rotary_dim, cache_len, layout, fp8, q_out, k_out)
    dt = _dt(q)
    args = (_ptr(q_out), _ptr(k_out), _out_dt(fp8, dt), _ptr(q), _ptr(k), _ptr(wq), _ptr(wk), dt,
            T, Hq, Hk, D, rotary_dim, layout, _ptr(positions), _ptr(cos), _ptr(sin), cache_len,
            eps, weight_offset, inv_scale)
    if unrounded:
        _check(lib().edge_qk_norm_rope_ex(*args, QK_ROTATE_UNROUNDED, _stream(stream)),
               "edge_qk_norm_rope_ex")
    else:
        _check(lib().edge_qk_norm_rope(*args, _stream(stream)), "edge_qk_norm_rope")
    return q_out, k_out


def rope(q, k, positions, cos, sin, *, rotary_dim=None, layout=ROTATE_HALF, q_out=None,
         k_out=None, fp8=False, inv_scale=1.0, cache_len=None, stream=None):
    """Standalone rotary embedding of q: [T, Hq, D] and k: [T, Hk, D] (k may
    be None).  Pass q_out=q (k_out=k) for the in-place form.  Returns (q_out, k_out)."""
    _need_contig(q, k, positions, cos, sin, q_out, k_out)
    T, Hq, Hk, D, rotary_dim, cache_len, layout, q_out, k_out = _qk_shapes(
        q, k, cos, rotary_dim, cache_len, layout, fp8, q_out, k_out)
    dt = _dt(q)
    _check(lib().edge_rope(_ptr(q_out), _ptr(k_out), _out_dt(fp8, dt), _ptr(q), _ptr(k), dt, T, Hq,
                           Hk, D, rotary_dim, layout, _ptr(positions), _ptr(cos), _ptr(sin),
                           cache_len, inv_scale, _stream(stream)), "edge_rope")
    return q_out, k_out
