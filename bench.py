#!/usr/bin/env python3
"""Decode-seam benchmark: HBM GB/s of the fused ops on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl edge|reference]

Prints one JSON line on rank 0.

Workload (one step).  The seam ops of one decode pass through a 36-layer
decoder shaped like the decode configuration:
  - hidden 2560, gate 2 x 9728, 32 query and 8 key heads of head_dim 128;
  - T = 64 tokens (the largest decode width of that configuration), bf16.
Per layer, in order:
    add_rmsnorm(x=mlp_out, residual) -> h1                input norm, direct weight
    qk_norm_rope(q, k) in place, rotate-half 128 of 128   theta 1e6, cache 4096
    add_rmsnorm(x=attn_out, residual) -> h2               post-attention norm
    glu_act(gate_up [T, 2*9728], SiLU) -> act
Every layer owns its buffers, so one step touches about 277 MB, more than
the 129 MB L2.  Successive steps therefore read their inputs from HBM, and
no L2 flush is needed.  The step (144 launches) is captured in one CUDA graph
and replayed.  `value` is the algorithmic bytes of all ranks' steps divided
by the slowest rank's device time, in GB/s.

Extra keys:
  - roofline: the dominant kernel's achieved GB/s over the measured HBM
    copy peak;
  - cpu_baseline: the CPU oracle timed on the host;
  - e2e: host-pinned inputs -> device -> host results, through the same
    C-ABI calls; consecutive steps overlap their copies and compute on
    three streams over two device buffer sets;
  - sweep: per-op GB/s vs T, cold L2;
  - t1_us_per_call: graph-replayed microseconds per call at T=1 with a
    warm L2, 32 launches per sample.

--impl reference times the CPU oracle instead, on a bounded sample of the
same workload (8 tokens of one layer per step), on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "QK-norm+RoPE & add-RMSNorm: HBM GB/s (% peak) vs T; µs/call at T=1"
UNIT = "GB/s"
L2_BYTES = 129 * 1024 * 1024

# decode workload geometry
T_DEC, HID, INTER, HQ, HK, HD, LAYERS = 64, 2560, 9728, 32, 8, 128, 36
THETA, CACHE, EPS = 1e6, 4096, 1e-6


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["edge", "reference"], default="edge")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-t1", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=6.0)
    # --probe: launch one op (or the whole sweep) a few times for a profiler to
    # capture; no timing, no JSON line
    ap.add_argument("--probe", metavar="OP", choices=PROBE_OPS + ("sweep",))
    ap.add_argument("--T", type=int, default=2048)
    ap.add_argument("--hq", type=int, default=16)
    ap.add_argument("--hk", type=int, default=2)
    ap.add_argument("--d", type=int, default=256)
    ap.add_argument("--rot", type=int, default=64)
    ap.add_argument("--hidden", type=int, default=2048)
    ap.add_argument("--inter", type=int, default=9728)
    ap.add_argument("--fp8", action="store_true")
    ap.add_argument("--no-weight", action="store_true")
    ap.add_argument("--reps", type=int, default=3)
    return ap.parse_args()


PROBE_OPS = ("qk", "qk_dflash2", "add_rmsnorm", "rmsnorm", "rope", "layernorm", "quantize",
             "qkv_cache", "glu_silu", "glu_gelu", "copy")


def run_probe(args):
    """Launch one op (or every case of the sweep) `reps` times on cuda:0,
    through the C ABI, for ncu to capture."""
    import torch

    from memory_bound_decode_qk_gb300 import edge_ops as ops, synth

    ops.lib()
    if args.probe == "sweep":
        cases = [(op, dict(kw, T=T)) for _, op, kw, Ts in SWEEP for T in Ts]
    else:
        cases = [(args.probe, dict(T=args.T, hq=args.hq, hk=args.hk, d=args.d, rot=args.rot,
                                   hidden=args.hidden, inter=args.inter, fp8=args.fp8,
                                   weight=not args.no_weight))]
    for op, kw in cases:
        fn = probe_case(torch, ops, synth, op, torch.bfloat16, **kw)
        for _ in range(args.reps):
            fn()
        torch.cuda.synchronize()
        print(op, kw, "ok", flush=True)
    return 0


# ---------------------------------------------------------------- bytes

def bytes_add_rmsnorm(T, H, s=2, out_s=2, weight=True):
    return T * H * s * 3 + T * H * out_s + (H * s if weight else 0)


def bytes_rmsnorm(T, H, s=2, out_s=2, weight=True):
    return T * H * s + T * H * out_s + (H * s if weight else 0)


def bytes_qk(T, Hq, Hk, D, rot, s=2, out_s=2):
    # q, k read and written; two norm weights; one position and two cache
    # rows of rot/2 fp32 per token
    return T * (Hq + Hk) * D * (s + out_s) + 2 * D * s + T * 8 + T * 2 * (rot // 2) * 4


def bytes_glu(T, d, s=2, out_s=2):
    return T * d * 2 * s + T * d * out_s


def bytes_rope(T, Hq, Hk, D, rot, s=2, out_s=2):
    return T * (Hq + Hk) * D * (s + out_s) + T * 8 + T * 2 * (rot // 2) * 4


def bytes_layernorm(T, H, s=2, out_s=2, affine=True):
    return T * H * (s + out_s) + (2 * H * s if affine else 0)


def bytes_quant(n, s=2):
    return n * (s + 1)


def bytes_qkv_cache(T, Hq, Hk, D, rot, s=2):
    # qkv read; q_out and the k/v cache rows written; weights, positions,
    # slots and two cache rows of rot/2 fp32 per token
    return 2 * T * (Hq + 2 * Hk) * D * s + 2 * D * s + 16 * T + T * 2 * (rot // 2) * 4


def layer_bytes(T=T_DEC):
    return (2 * bytes_add_rmsnorm(T, HID) + bytes_qk(T, HQ, HK, HD, HD) + bytes_glu(T, INTER))


# ---------------------------------------------------------------- environment

def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples (50 ms) of SM clock and throttle reasons."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = [r for (t, r) in self.rows if t0 <= t <= t1 + 0.06]
        window = "timed"
        if not rows:
            rows = [r for (_, r) in self.rows]
            window = "run"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows), "window": window,
                "power_w_max": max((float(r[4]) for r in rows
                                    if r[4].replace(".", "").isdigit()), default=None)}


def visible_index(local_rank):
    v = os.environ.get("CUDA_VISIBLE_DEVICES")
    if v:
        ids = [x.strip() for x in v.split(",")]
        if local_rank < len(ids) and ids[local_rank].isdigit():
            return int(ids[local_rank])
    return local_rank


def reduce_max(v, world, device):
    """The slowest rank's value (all ranks get it); the identity on one rank."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(step_bytes, steps, world, ms):
    """Whole-job GB/s: every rank's algorithmic bytes over the slowest rank's time."""
    return step_bytes * steps * world / (ms * 1e-3) / 1e9


# ---------------------------------------------------------------- CPU oracle timing

def oracle_layer_args(T, seed=0):
    """Storage arrays for one layer of the workload (the oracle's inputs)."""
    import torch

    import oracle
    from memory_bound_decode_qk_gb300 import synth

    def st(t):
        t = t.contiguous()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 \
            else t.numpy()

    r1 = synth.rows_inputs(seed, torch.bfloat16, T, HID)
    r2 = synth.rows_inputs(seed + 100, torch.bfloat16, T, HID)
    q = synth.qk_inputs(seed, torch.bfloat16, T, HQ, HK, HD, HD, theta=THETA, cache_len=CACHE,
                        positions="arange", w_mean=1.0, w_std=0.02)
    g = synth.glu_inputs(seed, torch.bfloat16, T, INTER)
    return dict(
        r1=[st(r1["x"]), st(r1["residual"]), st(r1["w"])],
        r2=[st(r2["x"]), st(r2["residual"]), st(r2["w"])],
        qk=[st(q["q"]), st(q["k"]), st(q["wq"]), st(q["wk"])],
        pos=q["positions"].numpy(), cos=q["cos"].numpy(), sin=q["sin"].numpy(),
        gu=st(g["gate_up"]), oracle=oracle)


def oracle_layer(a):
    o = a["oracle"]
    o.add_rmsnorm(*a["r1"], o.BF16, EPS)
    o.qk_norm_rope(*a["qk"], o.BF16, HD, o.ROTATE_HALF, a["pos"], a["cos"], a["sin"], EPS, 0)
    o.add_rmsnorm(*a["r2"], o.BF16, EPS)
    o.glu_act(a["gu"], o.BF16, o.SILU)


def cpu_info():
    """(logical cores, CPU model) of the host."""
    model = platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return os.cpu_count() or 1, model


def oracle_layers_for(a, seconds, threads):
    """Run whole layers of the oracle for about `seconds` on `threads` host
    threads (each runs its own layers; the C oracle releases the GIL), and
    return (layers, elapsed seconds)."""
    from concurrent.futures import ThreadPoolExecutor

    t0 = time.perf_counter()
    deadline = t0 + seconds

    def worker(_):
        n = 0
        while True:
            oracle_layer(a)
            n += 1
            if time.perf_counter() >= deadline:
                return n
    if threads == 1:
        n = worker(0)
    else:
        with ThreadPoolExecutor(threads) as ex:
            n = sum(ex.map(worker, range(threads)))
    return n, time.perf_counter() - t0


def cpu_baseline(seconds):
    """The oracle as it stands on the host: single-threaded, and split over all
    cores (one layer per thread at a time), `seconds` each."""
    a = oracle_layer_args(T_DEC)
    oracle_layer(a)
    cores, model = cpu_info()
    n1, el1 = oracle_layers_for(a, seconds, 1)
    n, el = oracle_layers_for(a, seconds, cores)
    gbs1 = layer_bytes() * n1 / el1 / 1e9
    gbs = layer_bytes() * n / el / 1e9
    return {"value": round(gbs, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "cpu": model, "ms_per_layer": round(el / n * 1e3, 3),
            "single_thread": {"value": round(gbs1, 4), "unit": UNIT, "cores": 1,
                              "ms_per_layer": round(el1 / n1 * 1e3, 3)},
            "sample": f"{n} of the workload's layers (T={T_DEC}, 4 ops each) in {el:.1f} s on "
                      f"{cores} threads (one layer each at a time), and {n1} layers in "
                      f"{el1:.1f} s on one thread; the C fp64 oracle on the host"}


def step_config(world):
    """The workload description both arms report."""
    step_bytes = LAYERS * layer_bytes()
    return {"workload": "decode seams of a 36-layer decoder: per layer add_rmsnorm, "
                        "qk_norm_rope, add_rmsnorm, silu_and_mul",
            "T": T_DEC, "hidden": HID, "gate": INTER, "heads": [HQ, HK], "head_dim": HD,
            "rotary": [HD, "rotate_half"], "layers": LAYERS, "global_batch": T_DEC * world,
            "l2": f"inputs larger than L2: {step_bytes / 1e6:.0f} MB per step, "
                  "distinct buffers per layer",
            "parallelism": f"replicas x{world}"}


def run_reference(args):
    """The oracle as it stands, on the host cores, on the benchmark's own step:
    the layers of a step (T = 64) split over the host threads, one layer per
    thread at a time.  A step takes all 36 layers when K + W steps of them fit
    in about two minutes; otherwise each step takes the largest whole number
    of layers that does (at least one per thread)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from concurrent.futures import ThreadPoolExecutor

    a = oracle_layer_args(T_DEC)
    cores, model = cpu_info()
    t0 = time.perf_counter()
    oracle_layer(a)
    t_layer = time.perf_counter() - t0
    total = args.steps + args.warmup
    per_step = LAYERS
    if total * per_step * t_layer / cores > 120.0:
        per_step = max(cores, int(120.0 * cores / (total * t_layer)) // cores * cores)
        per_step = min(per_step, LAYERS)
    with ThreadPoolExecutor(cores) as ex:
        def step():
            list(ex.map(lambda _: oracle_layer(a), range(per_step)))
        for _ in range(args.warmup):
            step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        el = time.perf_counter() - t0
    gbs = layer_bytes() * per_step * args.steps / el / 1e9
    sample = (f"{per_step} of the step's {LAYERS} layers (T={T_DEC}, 4 ops each) per step, on "
              f"{cores} host threads (one layer each at a time); the C fp64 oracle ({model})")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(1),
        "cpu_baseline": {"value": round(gbs, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "cpu": model, "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU workload

class Layer:
    pass


def build_layers(torch, synth, device, seed):
    """Per-layer device buffers, carved from three arenas so that the
    end-to-end leg moves each direction in two large copies:
      A (in and out): residual, q, k of every layer;
      B (in only):    mlp_out, attn_out, gate_up;
      C (out only):   h1, h2, act.
    Values come from one seeded layer, copied into every layer."""
    bf = torch.bfloat16
    r1 = synth.rows_inputs(seed, bf, T_DEC, HID)
    r2 = synth.rows_inputs(seed + 100, bf, T_DEC, HID)
    q = synth.qk_inputs(seed, bf, T_DEC, HQ, HK, HD, HD, theta=THETA, cache_len=CACHE,
                        positions="arange", w_mean=1.0, w_std=0.02)
    g = synth.glu_inputs(seed, bf, T_DEC, INTER)
    shared = dict(pos=q["positions"].to(device), cos=q["cos"].to(device),
                  sin=q["sin"].to(device))
    n_res, n_q, n_k = T_DEC * HID, T_DEC * HQ * HD, T_DEC * HK * HD
    n_gu, n_act = T_DEC * 2 * INTER, T_DEC * INTER
    per_a = n_res + n_q + n_k
    per_b = 2 * n_res + n_gu
    per_c = 2 * n_res + n_act
    A = torch.empty(LAYERS * per_a, dtype=bf, device=device)
    B = torch.empty(LAYERS * per_b, dtype=bf, device=device)
    C = torch.empty(LAYERS * per_c, dtype=bf, device=device)
    layers = []
    for i in range(LAYERS):
        L = Layer()
        a, b, c = A[i * per_a:(i + 1) * per_a], B[i * per_b:(i + 1) * per_b], C[i * per_c:(i + 1) * per_c]
        L.res = a[:n_res].view(T_DEC, HID)
        L.q = a[n_res:n_res + n_q].view(T_DEC, HQ, HD)
        L.k = a[n_res + n_q:].view(T_DEC, HK, HD)
        L.mlp_out = b[:n_res].view(T_DEC, HID)
        L.attn_out = b[n_res:2 * n_res].view(T_DEC, HID)
        L.gate_up = b[2 * n_res:].view(T_DEC, 2 * INTER)
        L.h1 = c[:n_res].view(T_DEC, HID)
        L.h2 = c[n_res:2 * n_res].view(T_DEC, HID)
        L.act = c[2 * n_res:].view(T_DEC, INTER)
        L.res.copy_(r1["residual"])
        L.q.copy_(q["q"])
        L.k.copy_(q["k"])
        L.mlp_out.copy_(r1["x"])
        L.attn_out.copy_(r2["x"])
        L.gate_up.copy_(g["gate_up"])
        L.w_in = r1["w"].to(device)
        L.w_post = r2["w"].to(device)
        L.wq = q["wq"].to(device)
        L.wk = q["wk"].to(device)
        layers.append(L)
    shared["arenas"] = (A, B, C)
    return layers, shared


OPS = ("add_rmsnorm_in", "qk_norm_rope", "add_rmsnorm_post", "glu_silu")
KERNEL_OPS = {"rows_vec_kernel": ("add_rmsnorm_in", "add_rmsnorm_post"),
              "qk_vec_kernel": ("qk_norm_rope",), "glu_vec_kernel": ("glu_silu",)}
# algorithmic bytes of one launch of each kernel in the step (both row-norm
# launches of a layer move the same bytes)
KERNEL_BYTES = {"rows_vec_kernel": bytes_add_rmsnorm(T_DEC, HID),
                "qk_vec_kernel": bytes_qk(T_DEC, HQ, HK, HD, HD),
                "glu_vec_kernel": bytes_glu(T_DEC, INTER)}
OP_SOURCE = {"rows_vec_kernel": "rows.cu", "qk_vec_kernel": "qk_norm_rope.cu",
             "glu_vec_kernel": "glu.cu"}


def layer_ops(ops, L, sh):
    """The four seam ops of one layer, as (name, thunk) pairs."""
    return [
        ("add_rmsnorm_in", lambda: ops.add_rmsnorm(L.mlp_out, L.res, L.w_in, eps=EPS, out=L.h1)),
        ("qk_norm_rope", lambda: ops.qk_norm_rope(L.q, L.k, L.wq, L.wk, sh["pos"], sh["cos"],
                                                  sh["sin"], rotary_dim=HD, eps=EPS,
                                                  weight_offset=0, q_out=L.q, k_out=L.k)),
        ("add_rmsnorm_post", lambda: ops.add_rmsnorm(L.attn_out, L.res, L.w_post, eps=EPS,
                                                     out=L.h2)),
        ("glu_silu", lambda: ops.glu_act(L.gate_up, ops.SILU, out=L.act)),
    ]


def graph_event(torch):
    """A timing event that records a timestamp node when captured in a graph."""
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return torch.cuda.Event(enable_timing=True)


class RawGraph:
    """A CUDA graph captured and launched through the CUDA runtime itself.

    torch.cuda.graph records the same kernel nodes and the same programmatic
    (dependent-launch) edges, but its replay ran the large prologue kernels
    25-30% slower on GB300 (13.6 against 10.6 us per launch at T = 2048, 24 +
    4 heads), and about 1% slower at decode widths.  Torch's own captured
    graph, instantiated through the runtime (with or without auto-free or
    node priorities) and launched with cudaGraphLaunch, ran at the fast time.
    So the benchmark captures and launches its graphs here.  replay()
    launches on the stream the graph was captured on."""

    _rt = None

    @classmethod
    def runtime(cls, torch):
        if cls._rt is None:
            import ctypes
            import glob
            cands = glob.glob(os.path.join(os.path.dirname(torch.__file__), "lib", "libcudart.so*"))
            cands += glob.glob("/usr/local/cuda/lib64/libcudart.so*")
            cands += glob.glob("/usr/local/cuda/targets/*/lib/libcudart.so*")
            if not cands:
                raise RuntimeError("libcudart not found: cannot capture CUDA graphs")
            rt = ctypes.CDLL(sorted(cands)[-1])
            rt.cudaStreamBeginCapture.argtypes = [ctypes.c_void_p, ctypes.c_int]
            rt.cudaStreamEndCapture.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
            rt.cudaGraphInstantiateWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p,
                                                        ctypes.c_ulonglong]
            rt.cudaGraphLaunch.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
            rt.cudaGraphExecDestroy.argtypes = [ctypes.c_void_p]
            rt.cudaGraphDestroy.argtypes = [ctypes.c_void_p]
            cls._rt = rt
        return cls._rt

    def __init__(self, torch, fn, stream):
        import ctypes
        rt = self.runtime(torch)
        self.rt, self.stream = rt, stream
        self.graph, self.exe = ctypes.c_void_p(), ctypes.c_void_p()
        raw = ctypes.c_void_p(stream.cuda_stream)
        with torch.cuda.stream(stream):
            if rt.cudaStreamBeginCapture(raw, 2) != 0:  # relaxed: no other stream is touched
                raise RuntimeError("cudaStreamBeginCapture failed")
            try:
                fn()
            finally:
                rc = rt.cudaStreamEndCapture(raw, ctypes.byref(self.graph))
        if rc != 0 or rt.cudaGraphInstantiateWithFlags(ctypes.byref(self.exe), self.graph, 0) != 0:
            raise RuntimeError("CUDA graph capture or instantiation failed")
        self._raw = raw

    def replay(self):
        if self.rt.cudaGraphLaunch(self.exe, self._raw) != 0:
            raise RuntimeError("cudaGraphLaunch failed")

    def __del__(self):
        try:
            self.rt.cudaGraphExecDestroy(self.exe)
            self.rt.cudaGraphDestroy(self.graph)
        except Exception:
            pass


def capture(torch, fn, stream):
    """One eager run (library load, launch checks), then a graph of fn on
    `stream`; replay() launches it there."""
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = RawGraph(torch, fn, stream)
    torch.cuda.synchronize()
    return g


def source_sha(kernel):
    """Hash of the code of the source file that holds the kernel and of the
    shared device helpers it includes, so that a stored capture goes stale
    whenever the kernel's code may have changed.  Comments and whitespace are
    left out: editing them changes no kernel."""
    csrc = os.path.join(ROOT, "memory_bound_decode_qk_gb300", "csrc")
    h = hashlib.sha256()
    for name in (OP_SOURCE[kernel], "edge_common.cuh"):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def traffic_for(kernel):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source is unchanged since it was captured."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get("decode_step", {}).get(kernel)
    if not e or e.get("source_sha") != source_sha(kernel):
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- sweep

def probe_case(torch, ops, synth, op, dtype, T, hq=16, hk=2, d=256, rot=64, hidden=2048,
               inter=9728, fp8=False, weight=True, device="cuda"):  # noqa: C901 (one branch per op)
    """A zero-argument callable that launches one op once, on buffers of its own
    (seeded synthetic inputs shaped like the workloads), through the C ABI."""
    u8 = torch.uint8
    if op == "qk":
        i = synth.qk_inputs(0, dtype, T, hq, hk, d, rot, theta=1e7, cache_len=32768,
                            positions="offset", w_std=0.05)
        t = {k: (v.to(device) if v is not None else None) for k, v in i.items()}
        qo = torch.empty(t["q"].shape, dtype=u8 if fp8 else dtype, device=device)
        ko = torch.empty(t["k"].shape, dtype=u8 if fp8 else dtype, device=device)
        return lambda: ops.qk_norm_rope(t["q"], t["k"], t["wq"], t["wk"], t["positions"],
                                        t["cos"], t["sin"], rotary_dim=rot, weight_offset=1,
                                        q_out=qo, k_out=ko, fp8=fp8, inv_scale=40.0)
    if op == "qk_dflash2":
        # DFlash2 pair: 32 + 32 heads of 128, full rotary, direct weights, in
        # place; W = 16 draft positions per sequence
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
        o = torch.empty(T, hidden, dtype=u8 if fp8 else dtype, device=device)
        if op == "rmsnorm":
            return lambda: ops.rmsnorm(x, w, eps=EPS, out=o, fp8=fp8, inv_scale=40.0)
        r = i["residual"].to(device)
        return lambda: ops.add_rmsnorm(x, r, w, eps=EPS, out=o, fp8=fp8, inv_scale=40.0)
    if op == "rope":
        i = synth.qk_inputs(0, dtype, T, hq, hk, d, rot, theta=1e7, cache_len=32768,
                            positions="offset")
        t = {k: (v.to(device) if v is not None else None) for k, v in i.items()}
        qo, ko = torch.empty_like(t["q"]), torch.empty_like(t["k"])
        return lambda: ops.rope(t["q"], t["k"], t["positions"], t["cos"], t["sin"],
                                rotary_dim=rot, q_out=qo, k_out=ko)
    if op == "layernorm":
        i = synth.rows_inputs(0, dtype, T, hidden, residual=False)
        x, g = i["x"].to(device), i["w"].to(device)
        o = torch.empty(T, hidden, dtype=u8 if fp8 else dtype, device=device)
        return lambda: ops.layernorm(x, g, g, eps=1e-6, out=o, fp8=fp8, inv_scale=40.0)
    if op == "quantize":
        x = synth.rows_inputs(0, dtype, T, hidden, residual=False)["x"].to(device)
        o = torch.empty(x.shape, dtype=u8, device=device)
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
        o = torch.empty(T, inter, dtype=u8 if fp8 else dtype, device=device)
        act = ops.SILU if op == "glu_silu" else ops.GELU_TANH
        return lambda: ops.glu_act(gu, act, out=o, fp8=fp8, inv_scale=40.0)
    if op == "copy":
        # the yardstick: `hidden` bytes moved, half read and half written
        src = torch.zeros(hidden // 2, dtype=u8, device=device)
        dst = torch.empty_like(src)
        return lambda: ops.copy(src, out=dst)
    raise ValueError(op)


def case_bytes(op, T, hq=16, hk=2, d=256, rot=64, hidden=2048, inter=9728, fp8=False,
               weight=True):
    """Algorithmic bytes of one call of a probe case."""
    o = 1 if fp8 else 2
    if op == "qk":
        return bytes_qk(T, hq, hk, d, rot, out_s=o)
    if op == "qk_dflash2":
        return bytes_qk(T, 32, 32, 128, 128)
    if op == "add_rmsnorm":
        return bytes_add_rmsnorm(T, hidden, out_s=o, weight=weight)
    if op == "rmsnorm":
        return bytes_rmsnorm(T, hidden, out_s=o, weight=weight)
    if op == "rope":
        return bytes_rope(T, hq, hk, d, rot)
    if op == "layernorm":
        return bytes_layernorm(T, hidden, out_s=o)
    if op == "quantize":
        return bytes_quant(T * hidden)
    if op == "qkv_cache":
        return bytes_qkv_cache(T, hq, hk, d, rot)
    if op in ("glu_silu", "glu_gelu"):
        return bytes_glu(T, inter, out_s=o)
    if op == "copy":
        return hidden
    raise ValueError(op)


# The sweep: (key, op, fixed arguments, values of T).  Every op has a T = 256
# point, the width at which the ops should reach 70% of HBM peak.
SWEEP = [
    ("qk_norm_rope_bf16_16x2_d256_r64", "qk", dict(hq=16, hk=2),
     (1, 8, 32, 128, 256, 512, 1024, 2048)),
    ("qk_norm_rope_bf16_24x4_d256_r64", "qk", dict(hq=24, hk=4),
     (1, 8, 32, 128, 256, 512, 1024, 2048)),
    ("qk_norm_rope_dflash2_bf16_32x32_d128_inplace_W16", "qk_dflash2", {},
     (16, 64, 256, 1024, 2048)),
    ("add_rmsnorm_bf16_h2048", "add_rmsnorm", dict(hidden=2048), (1, 16, 64, 256, 512, 1024, 4096)),
    ("add_rmsnorm_bf16_h2048_fp8", "add_rmsnorm", dict(hidden=2048, fp8=True),
     (1, 16, 64, 256, 512, 1024, 4096)),
    ("add_rmsnorm_bf16_h1024", "add_rmsnorm", dict(hidden=1024), (1, 16, 64, 256, 512, 1024, 4096)),
    ("add_rmsnorm_bf16_h1024_fp8", "add_rmsnorm", dict(hidden=1024, fp8=True),
     (1, 16, 64, 256, 512, 1024, 4096)),
    ("add_rmsnorm_bf16_h2560", "add_rmsnorm", dict(hidden=2560), (1, 16, 64, 256, 512, 1024, 4096)),
    ("add_rmsnorm_bf16_h2560_fp8", "add_rmsnorm", dict(hidden=2560, fp8=True),
     (1, 16, 64, 256, 512, 1024, 4096)),
    ("rmsnorm_noweight_bf16_h2048_fp8", "rmsnorm", dict(hidden=2048, fp8=True, weight=False),
     (1, 64, 256, 512, 4096)),
    ("rope_bf16_24x4_d256_r64", "rope", dict(hq=24, hk=4), (1, 64, 256, 512, 2048)),
    ("layernorm_bf16_h1152", "layernorm", dict(hidden=1152), (1, 64, 256, 512, 4096)),
    ("quantize_fp8_bf16_rows_x2048", "quantize", dict(hidden=2048), (1, 256, 512, 4096)),
    ("qkv_rope_cache_bf16_16x2_d256_r64", "qkv_cache", dict(hq=16, hk=2), (1, 64, 256, 512, 2048)),
    ("glu_silu_bf16_d9728", "glu_silu", dict(inter=9728), (1, 64, 256, 512, 4096)),
    ("glu_gelu_bf16_d2048_fp8", "glu_gelu", dict(inter=2048, fp8=True), (1, 64, 256, 512, 4096)),
    ("glu_gelu_bf16_d10240", "glu_gelu", dict(inter=10240), (1, 64, 256, 512, 4096)),
]


def sweep(torch, ops, synth, device, peak):
    """Per-op time vs T, each beside the yardstick copy of the same bytes.

    S copies of a call's buffers, with S * bytes over 2.5x L2 where that fits
    in 64 copies, are cycled by a graph of at least 32 back-to-back launches,
    so every launch reads cold inputs from HBM.  The graph is replayed 10
    times after 3 warm-ups and timed with events.  Below that size the data
    stays L2-resident, and the entry is marked warm.  The copy moves the op's
    algorithmic bytes (half read, half written) with the ops' launch form
    (edge_copy), timed the same way: its time is what a kernel that only moves
    those bytes needs."""
    bf = torch.bfloat16
    stream = torch.cuda.Stream(device)

    def timed(make, nbytes):
        sets = int(min(64, max(2, -(-int(2.5 * L2_BYTES) // nbytes))))
        fns = [make() for _ in range(sets)]
        reps = sets * max(1, -(-32 // sets))

        def body():
            for i in range(reps):
                fns[i % sets]()
        g = capture(torch, body, stream)
        for _ in range(3):
            g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(10):
                g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / (10 * reps)
        cold = sets * nbytes >= 2 * L2_BYTES
        del g, fns
        return us, cold

    out = {}
    for key, op, kw, Ts in SWEEP:
        out[key] = {}
        for T in Ts:
            nb = case_bytes(op, T, **kw)
            us, cold = timed(lambda: probe_case(torch, ops, synth, op, bf, T, **kw), nb)
            cus, _ = timed(lambda: probe_case(torch, ops, synth, "copy", bf, 1,
                                              hidden=(nb + 31) // 32 * 32), nb)
            gbs = nb / (us * 1e-6) / 1e9
            tag = f"B{T // 16}" if op == "qk_dflash2" else str(T)
            out[key][tag] = [round(us, 3), round(gbs, 1), round(gbs / peak, 4),
                             "cold" if cold else "warm", round(cus, 3), round(cus / us, 3)]
    return out


ALIAS = {
    "qk_norm_rope_bf16_16x2_d256_r64": "qk16x2", "qk_norm_rope_bf16_24x4_d256_r64": "qk24x4",
    "qk_norm_rope_dflash2_bf16_32x32_d128_inplace_W16": "dflash2",
    "add_rmsnorm_bf16_h2048": "arn2048", "add_rmsnorm_bf16_h2048_fp8": "arn2048f8",
    "add_rmsnorm_bf16_h1024": "arn1024", "add_rmsnorm_bf16_h1024_fp8": "arn1024f8",
    "add_rmsnorm_bf16_h2560": "arn2560", "add_rmsnorm_bf16_h2560_fp8": "arn2560f8",
    "rmsnorm_noweight_bf16_h2048_fp8": "rmsnw2048f8", "rope_bf16_24x4_d256_r64": "rope24x4",
    "layernorm_bf16_h1152": "ln1152", "quantize_fp8_bf16_rows_x2048": "quant2048",
    "qkv_rope_cache_bf16_16x2_d256_r64": "qkv16x2", "glu_silu_bf16_d9728": "silu9728",
    "glu_gelu_bf16_d2048_fp8": "gelu2048f8", "glu_gelu_bf16_d10240": "gelu10240"}
T1_ALIAS = {"qk_norm_rope_16x2": "qk16x2", "qk_norm_rope_24x4": "qk24x4",
            "add_rmsnorm_h2560": "arn2560", "glu_silu_d9728": "silu9728",
            "launch_floor_quantize_16": "floor"}


def sweep_summary(sw, t1):
    """The key figures of the sweep in under 1.5 KB (the end of the JSON line):
    per op, the fraction of measured HBM peak and of the same-bytes copy at
    T = 256, 512 and the largest T, as "T:peak/copy"; and the T = 1
    microseconds per call."""
    rows = {}
    for key, by_t in sw.items():
        ts = list(by_t)
        pick = [t for t in ts if t in ("256", "512", "B16", "B64")] + [ts[-1]]
        rows[ALIAS.get(key, key)] = " ".join(
            f"{t}:{by_t[t][2]:.2f}/{by_t[t][5]:.2f}" for t in dict.fromkeys(pick))
    return {"format": "T:fraction of HBM peak/fraction of copy speed",
            "t1_us": {T1_ALIAS.get(k, k): v["median"] for k, v in (t1 or {}).items()
                      if "median" in v},
            "ops": rows}


def t1_latency(torch, ops, synth, device):
    """Graph replay of 32 back-to-back T=1 calls on the same buffers (warm L2):
    200 samples after 20 warm-up replays, median and IQR in us per call."""
    bf = torch.bfloat16
    stream = torch.cuda.Stream(device)
    res = {}

    def measure(fn):
        def many():
            for _ in range(32):
                fn()
        g = capture(torch, many, stream)
        for _ in range(20):
            g.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(200)]
        with torch.cuda.stream(stream):
            for a, b in evs:
                a.record(stream)
                g.replay()
                b.record(stream)
        torch.cuda.synchronize()
        per = np.array([a.elapsed_time(b) for a, b in evs]) * 1e3 / 32
        q1, med, q3 = np.percentile(per, [25, 50, 75])
        return {"median": round(float(med), 3), "iqr": [round(float(q1), 3), round(float(q3), 3)]}

    for (hq, hk) in ((16, 2), (24, 4)):
        i = synth.qk_inputs(0, bf, 1, hq, hk, 256, 64, theta=1e7, cache_len=32768,
                            positions="offset", w_std=0.05)
        d = {k: v.to(device) for k, v in i.items()}
        qo, ko = torch.empty_like(d["q"]), torch.empty_like(d["k"])
        res[f"qk_norm_rope_{hq}x{hk}"] = measure(
            lambda: ops.qk_norm_rope(d["q"], d["k"], d["wq"], d["wk"], d["positions"], d["cos"],
                                     d["sin"], rotary_dim=64, weight_offset=1, q_out=qo,
                                     k_out=ko))
    i = synth.rows_inputs(0, bf, 1, HID)
    x, r, w = (i[k].to(device) for k in ("x", "residual", "w"))
    o = torch.empty_like(x)
    res["add_rmsnorm_h2560"] = measure(lambda: ops.add_rmsnorm(x, r, w, eps=EPS, out=o))
    gu = synth.glu_inputs(0, bf, 1, INTER)["gate_up"].to(device)
    og = torch.empty(1, INTER, dtype=bf, device=device)
    res["glu_silu_d9728"] = measure(lambda: ops.glu_act(gu, ops.SILU, out=og))
    # the floor of a dependent launch: a 16-element quantize (one CTA, one
    # load, one store) chained the same way
    xq = torch.ones(16, dtype=bf, device=device)
    oq = torch.empty(16, dtype=torch.uint8, device=device)
    res["launch_floor_quantize_16"] = measure(lambda: ops.quantize_fp8(xq, 1.0, out=oq))

    # host cost of one eager call at T = 1 (no graph): validation, dispatch
    # and cudaLaunchKernelEx in the C library, called once through ctypes
    # directly and once through the Python binding, on a stream drained every
    # 64 calls so that the launch queue never fills
    lib = ops.lib()
    i = synth.qk_inputs(0, bf, 1, 16, 2, 256, 64, theta=1e7, cache_len=32768,
                        positions="offset", w_std=0.05)
    d = {k: v.to(device) for k, v in i.items()}
    qo, ko = torch.empty_like(d["q"]), torch.empty_like(d["k"])
    sptr = stream.cuda_stream
    cargs = (qo.data_ptr(), ko.data_ptr(), ops.BF16, d["q"].data_ptr(), d["k"].data_ptr(),
             d["wq"].data_ptr(), d["wk"].data_ptr(), ops.BF16, 1, 16, 2, 256, 64,
             ops.ROTATE_HALF, d["positions"].data_ptr(), d["cos"].data_ptr(),
             d["sin"].data_ptr(), 32768, EPS, 1, 1.0, sptr)

    def host_us(call, n=2048):
        for _ in range(64):
            call()
        torch.cuda.synchronize()
        t = 0.0
        for _ in range(n // 64):
            t0 = time.perf_counter()
            for _ in range(64):
                call()
            t += time.perf_counter() - t0
            torch.cuda.synchronize()
        return round(t / n * 1e6, 3)
    with torch.cuda.stream(stream):
        st = lib.edge_qk_norm_rope(*cargs)
        if st != 0:
            raise RuntimeError(f"edge_qk_norm_rope returned {ops.STATUS.get(st, st)}")
        res["host_us_per_eager_call"] = {
            "qk_norm_rope_16x2_ctypes": host_us(lambda: lib.edge_qk_norm_rope(*cargs)),
            "qk_norm_rope_16x2_python": host_us(
                lambda: ops.qk_norm_rope(d["q"], d["k"], d["wq"], d["wk"], d["positions"],
                                         d["cos"], d["sin"], rotary_dim=64, weight_offset=1,
                                         q_out=qo, k_out=ko)),
        }
    return res


# ---------------------------------------------------------------- main

def main():
    args = parse()
    if args.probe:
        return run_probe(args)
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    from memory_bound_decode_qk_gb300 import _build, edge_ops as ops, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if not os.path.exists(_build.LIB):
        if rank == 0:
            _build.build()
        if world > 1:
            dist.barrier()
    ops.lib()  # loud failure if the CUDA library is missing: no fallback
    peak, peak_kind = measured_peak()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(v):
        return reduce_max(v, world, device)

    layers, sh = build_layers(torch, synth, device, seed=rank)
    stream = torch.cuda.Stream(device)

    def step():
        for L in layers:
            for _, fn in layer_ops(ops, L, sh):
                fn()

    graph = capture(torch, step, stream)
    launches_per_step = LAYERS * len(OPS)
    step_bytes = LAYERS * layer_bytes()

    # per-kernel graphs: every launch of one kernel in a step, in step order,
    # on the same per-layer buffers; timed over K replays like the step
    kernel_graphs = {}
    for kern, names in KERNEL_OPS.items():
        def only(names=names):
            for L in layers:
                for name, fn in layer_ops(ops, L, sh):
                    if name in names:
                        fn()
        kernel_graphs[kern] = capture(torch, only, stream)

    sampler = ClockSampler(visible_index(local)) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)

    # ---- timed region: K graph replays of the step
    for _ in range(args.warmup):
        graph.replay()
    barrier()
    t_wall0 = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    barrier()
    t_wall1 = time.time()
    ms = max_over_ranks(e0.elapsed_time(e1))

    # ---- per-kernel average launch duration: K replays of each kernel's graph
    kernel_us = {}
    for kern, g in kernel_graphs.items():
        for _ in range(max(1, args.warmup)):
            g.replay()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(args.steps):
                g.replay()
            b.record(stream)
        barrier()
        n = args.steps * LAYERS * len(KERNEL_OPS[kern])
        kernel_us[kern] = max_over_ranks(a.elapsed_time(b)) * 1e3 / n
    if sampler:
        sampler.stop()

    # ---- e2e: pinned host inputs -> device, the step, results -> host
    # (the activations live in arenas: two copies in, two copies out).  Two
    # device buffer sets let consecutive steps overlap on three streams: step
    # i + 1's inputs go in while step i computes and step i - 1's results come
    # out (the host link is full duplex).  Every step still moves its own
    # inputs in and its results out inside the timed region.
    layers2, sh2 = build_layers(torch, synth, device, seed=rank)

    def step2():
        for L in layers2:
            for _, fn in layer_ops(ops, L, sh2):
                fn()
    graph2 = capture(torch, step2, stream)
    slots = [(sh["arenas"], graph), (sh2["arenas"], graph2)]
    A, B, C = sh["arenas"]
    hA = torch.empty(A.shape, dtype=A.dtype, pin_memory=True).copy_(A)
    hB = torch.empty(B.shape, dtype=B.dtype, pin_memory=True).copy_(B)
    oA = torch.empty(A.shape, dtype=A.dtype, pin_memory=True)
    oC = torch.empty(C.shape, dtype=C.dtype, pin_memory=True)
    h2d_bytes = (A.numel() + B.numel()) * A.element_size()
    d2h_bytes = (A.numel() + C.numel()) * A.element_size()
    e2e_steps = max(2, min(args.steps, 50))
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    evs = [{k: torch.cuda.Event() for k in ("in", "comp", "out")} for _ in slots]

    def e2e_run(n, first=None):
        for i in range(n):
            (a, b, c), g = slots[i % 2]
            ev = evs[i % 2]
            with torch.cuda.stream(s_in):
                if i == 0 and first is not None:
                    first.record(s_in)
                if i >= 2:
                    s_in.wait_event(ev["out"])  # this set's last results are out
                a.copy_(hA, non_blocking=True)
                b.copy_(hB, non_blocking=True)
                ev["in"].record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(ev["in"])
                g.replay()
                ev["comp"].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["comp"])
                oA.copy_(a, non_blocking=True)
                oC.copy_(c, non_blocking=True)
                ev["out"].record(s_out)

    e2e_run(2)
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(e2e_steps, first=f0)
    with torch.cuda.stream(s_out):
        f1.record(s_out)
    barrier()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1))

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return 0

    value = weak_scaling_value(step_bytes, args.steps, world, ms)
    e2e_value = weak_scaling_value(step_bytes, e2e_steps, world, e2e_ms)

    # dominant kernel: the largest share of the step's device time
    kern_ms = {k: kernel_us[k] * LAYERS * len(KERNEL_OPS[k]) for k in KERNEL_OPS}
    dom = max(kern_ms, key=kern_ms.get)
    avg_us = kernel_us[dom]
    dom_bytes = KERNEL_BYTES[dom]
    achieved = dom_bytes / (avg_us * 1e-6) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy)",
                "traffic": traffic_for(dom), "bytes_per_launch": dom_bytes,
                "avg_launch_us": round(avg_us, 3),
                "launch_us": {k: round(v, 3) for k, v in kernel_us.items()},
                "share": {k: round(v / sum(kern_ms.values()), 4) for k, v in kern_ms.items()}}

    clocks = sampler.summary(t_wall0, t_wall1) if sampler else {}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": step_config(world),
        "launch": {"graph": "one CUDA graph per step (144 launches)",
                   "pdl": os.environ.get("EDGE_OPS_PDL", "1") != "0"},
        "step_bytes": step_bytes,
        "roofline": roofline,
        "gpu_launches": launches_per_step * args.steps,
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d_bytes,
                "d2h_bytes_per_step": d2h_bytes, "steps": e2e_steps,
                "pipeline": "two device buffer sets; copies in, the step and copies out of "
                            "consecutive steps overlap on three streams"},
        "clocks": clocks,
    }
    if world == 1:
        t1 = None
        if not args.no_t1:
            t1 = line["t1_us_per_call"] = t1_latency(torch, ops, synth, device)
        if not args.no_sweep:
            line["sweep"] = sweep(torch, ops, synth, device, peak)
            line["sweep_format"] = ("T -> [us per call in back-to-back graph replay, GB/s, "
                                    "fraction of measured HBM peak, L2 state, us of the copy "
                                    "of the same bytes, copy us / op us]")
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        if not args.no_sweep:
            # last, so that the end of the line carries the key figures
            line["summary"] = sweep_summary(line["sweep"], t1)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
