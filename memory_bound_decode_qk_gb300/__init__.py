"""GB300-native fused decode-seam operators.

The per-head QK-RMSNorm + RoPE attention prologue, residual-add RMSNorm,
RMSNorm and SiLU / tanh-GELU gated activations.  Each op has an optional
static-scale FP8 E4M3 output.  Every op is a hand-written sm_103a CUDA kernel
behind the C ABI declared in ``include/edge_ops.h``; ``edge_ops`` is the thin
ctypes binding over it, and ``synth`` draws the seeded inputs.
"""

__all__ = ["edge_ops", "synth"]


def __getattr__(name):
    if name in ("edge_ops", "synth"):
        import importlib

        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
