"""Run one op at one shape a few times, for a profiler to capture.

    python -m memory_bound_decode_qk_gb300.probe --op qk --T 2048 --hq 24 --hk 4
    python -m memory_bound_decode_qk_gb300.probe --sweep --reps 3

--sweep runs the benchmark's T sweep (every op and width), each case `reps`
times in order, so that a profiler's launch list gives per-kernel device
times versus T.  Inputs are seeded synthetic tensors (synth), and every call
goes through the C ABI.
"""
from __future__ import annotations

import argparse

import torch

from . import edge_ops as ops
from . import synth

DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def make_case(op, dtype, T, hq=16, hk=2, d=256, rot=64, hidden=2048, inter=9728, fp8=False,
              layout=0, weight=True, device="cuda"):  # noqa: C901 (one branch per op)
    """A zero-argument callable that launches the op once on fresh buffers."""
    if op == "qk":
        i = synth.qk_inputs(0, dtype, T, hq, hk, d, rot, theta=1e7, cache_len=32768,
                            positions="offset", w_std=0.05)
        t = {k: (v.to(device) if v is not None else None) for k, v in i.items()}
        qo = torch.empty(t["q"].shape, dtype=torch.uint8 if fp8 else dtype, device=device)
        ko = torch.empty(t["k"].shape, dtype=torch.uint8 if fp8 else dtype, device=device)
        return lambda: ops.qk_norm_rope(t["q"], t["k"], t["wq"], t["wk"], t["positions"],
                                        t["cos"], t["sin"], rotary_dim=rot, layout=layout,
                                        weight_offset=1, q_out=qo, k_out=ko, fp8=fp8,
                                        inv_scale=40.0)
    if op == "qk_dflash2":
        # DFlash2 pair: 32 + 32 heads of 128, full rotary, direct weights, in place
        i = synth.qk_inputs(0, dtype, T, 32, 32, 128, 128, theta=1e6, cache_len=32768,
                            positions="blocks:16", w_mean=1.0, w_std=0.02)
        t = {k: v.to(device) for k, v in i.items()}
        return lambda: ops.qk_norm_rope(t["q"], t["k"], t["wq"], t["wk"], t["positions"],
                                        t["cos"], t["sin"], rotary_dim=128, q_out=t["q"],
                                        k_out=t["k"])
    if op in ("add_rmsnorm", "rmsnorm"):
        i = synth.rows_inputs(0, dtype, T, hidden, residual=op == "add_rmsnorm")
        x = i["x"].to(device)
        w = i["w"].to(device) if weight else None
        o = torch.empty(T, hidden, dtype=torch.uint8 if fp8 else dtype, device=device)
        if op == "rmsnorm":
            return lambda: ops.rmsnorm(x, w, out=o, fp8=fp8, inv_scale=40.0)
        r = i["residual"].to(device)
        return lambda: ops.add_rmsnorm(x, r, w, out=o, fp8=fp8, inv_scale=40.0)
    if op == "rope":
        i = synth.qk_inputs(0, dtype, T, hq, hk, d, rot, theta=1e7, cache_len=32768,
                            positions="offset")
        t = {k: (v.to(device) if v is not None else None) for k, v in i.items()}
        qo, ko = torch.empty_like(t["q"]), torch.empty_like(t["k"])
        return lambda: ops.rope(t["q"], t["k"], t["positions"], t["cos"], t["sin"],
                                rotary_dim=rot, layout=layout, q_out=qo, k_out=ko)
    if op == "layernorm":
        i = synth.rows_inputs(0, dtype, T, hidden, residual=False)
        x, g = i["x"].to(device), i["w"].to(device)
        o = torch.empty(T, hidden, dtype=torch.uint8 if fp8 else dtype, device=device)
        return lambda: ops.layernorm(x, g, g, out=o, fp8=fp8, inv_scale=40.0)
    if op == "quantize":
        x = synth.rows_inputs(0, dtype, T, hidden, residual=False)["x"].to(device)
        o = torch.empty(x.shape, dtype=torch.uint8, device=device)
        return lambda: ops.quantize_fp8(x, 40.0, out=o)
    if op == "qkv_cache":
        qkv = synth.to_dtype(synth.normal(0, 71, T * (hq + 2 * hk) * d), dtype).view(T, -1)
        qkv = qkv.to(device)
        w = synth.to_dtype(synth.normal(0, 72, d, 0.0, 0.05), dtype).to(device)
        cos, sin = synth.rope_cache(1e7, rot, 32768)
        cos, sin = cos.to(device), sin.to(device)
        pos = torch.arange(T, dtype=torch.int64, device=device)
        kc = torch.empty(T, hk, d, dtype=dtype, device=device)
        vc = torch.empty_like(kc)
        qo = torch.empty(T, hq, d, dtype=dtype, device=device)
        return lambda: ops.qkv_rope_cache(qkv, hq, hk, w, w, pos, cos, sin, pos, kc, vc,
                                          rotary_dim=rot, weight_offset=1, q_out=qo)
    if op in ("glu_silu", "glu_gelu"):
        gu = synth.glu_inputs(0, dtype, T, inter)["gate_up"].to(device)
        o = torch.empty(T, inter, dtype=torch.uint8 if fp8 else dtype, device=device)
        act = ops.SILU if op == "glu_silu" else ops.GELU_TANH
        return lambda: ops.glu_act(gu, act, out=o, fp8=fp8, inv_scale=40.0)
    raise ValueError(op)


SWEEP = (
    [("qk", dict(T=T, hq=16, hk=2)) for T in (1, 8, 32, 128, 256, 512, 1024, 2048)]
    + [("qk", dict(T=T, hq=24, hk=4)) for T in (1, 8, 32, 128, 256, 512, 1024, 2048)]
    + [("add_rmsnorm", dict(T=T, hidden=H)) for H in (2048, 1024, 2560)
       for T in (1, 16, 64, 256, 512, 1024, 4096)]
    + [("add_rmsnorm", dict(T=T, hidden=H, fp8=True)) for H in (2048, 1024)
       for T in (256, 512, 4096)]
    + [("rmsnorm", dict(T=T, hidden=2048, fp8=True, weight=False)) for T in (64, 512, 4096)]
    + [("glu_silu", dict(T=T, inter=9728)) for T in (1, 64, 512, 4096)]
    + [("glu_gelu", dict(T=T, inter=2048, fp8=True)) for T in (64, 512, 4096)]
    + [("qk_dflash2", dict(T=16 * B)) for B in (1, 16, 64)]
    + [("rope", dict(T=T, hq=24, hk=4)) for T in (1, 512, 2048)]
    + [("layernorm", dict(T=T, hidden=1152)) for T in (1, 512, 4096)]
    + [("quantize", dict(T=T, hidden=2048)) for T in (512, 4096)]
    + [("qkv_cache", dict(T=T, hq=16, hk=2)) for T in (1, 512, 2048)]
)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--op", default="qk", choices=["qk", "add_rmsnorm", "rmsnorm", "glu_silu",
                                                   "glu_gelu", "rope", "layernorm", "quantize",
                                                   "qkv_cache", "qk_dflash2"])
    ap.add_argument("--dtype", default="bf16", choices=list(DT))
    ap.add_argument("--T", type=int, default=2048)
    ap.add_argument("--hq", type=int, default=16)
    ap.add_argument("--hk", type=int, default=2)
    ap.add_argument("--d", type=int, default=256)
    ap.add_argument("--rot", type=int, default=64)
    ap.add_argument("--hidden", type=int, default=2048)
    ap.add_argument("--inter", type=int, default=9728)
    ap.add_argument("--fp8", action="store_true")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--sweep", action="store_true")
    a = ap.parse_args()
    ops.lib()
    cases = SWEEP if a.sweep else [(a.op, dict(T=a.T, hq=a.hq, hk=a.hk, d=a.d, rot=a.rot,
                                               hidden=a.hidden, inter=a.inter, fp8=a.fp8))]
    for op, kw in cases:
        fn = make_case(op, DT[a.dtype], **kw)
        for _ in range(a.reps):
            fn()
        torch.cuda.synchronize()
        print(op, kw, "ok", flush=True)


if __name__ == "__main__":
    main()
