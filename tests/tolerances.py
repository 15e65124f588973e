"""Acceptance bands of the GPU parity tests, and the fp32 error analysis behind them.

The GPU computes in fp32 with its own summation order and the hardware
reciprocal square root; the oracle computes the exact value in fp64.  Where
the exact value of an output lies within a band of a rounding boundary of the
output format, both neighbours are correct roundings of a value the fp32
arithmetic may produce, so the strict check accepts either.  Everywhere else
the output must be bit-exact.  The bands below are first-order worst-case
bounds of the fp32 error, in units of u = 2^-24 (the fp32 unit roundoff), so
that a correct kernel always passes; the CPU tests in ``test_tolerances.py``
pin each band between its bound and twice its bound, so that a band too wide
to see a real slip fails there.

Error sources, each a relative error of at most:
  - one fp32 rounding (add, multiply, fma): u;
  - an fp32 constant rounded from its exact value: u/2;
  - ``rsqrtf``: 2 ulp, that is 4u at the bottom of a binade (CUDA's documented
    bound for the function);
  - ``ex2.approx.f32``: 2^-22 = 4u; ``rcp.approx.f32``: 2^-23 = 2u (the PTX ISA's
    stated accuracy of the approximate instructions; taken generously).
"""
from __future__ import annotations

import math

import numpy as np

U = 2.0 ** -24

# Largest reduction shapes of the kernels' fp32 sums of squares (a thread's
# sequential terms; the merges of its two alternating sums and of the two
# lanes of an fp32 pair; the shuffle tree of a warp; the combine over the
# warps of a row).  Every term is non-negative, so each addition adds at most
# u of the total to the relative error of the sum.
MAX_SEQ_TERMS = 32      # at most 4 vectors of 8 elements per running sum
MAX_TREE_LEVELS = 2 + 5  # the two merges, then a 32-lane xor tree
MAX_WARPS_PER_ROW = 16


def rms_norm_error_u(seq_terms=MAX_SEQ_TERMS, tree_levels=MAX_TREE_LEVELS,
                     warps=MAX_WARPS_PER_ROW):
    """Worst-case relative error, in u, of the fp32 normalized value
    x * r * (w + delta) with r = rsqrtf(fma(ss, 1/n, eps)).

      ss:          (seq_terms + tree_levels + warps - 1) u;
      r:           half of the error of its argument (ss, the rounding of 1/n
                   and of the fma: ss + 2u), plus rsqrtf's 4u;
      the output:  w + delta, x * r and the product with the weight: 3u.
    """
    ss = seq_terms + tree_levels + (warps - 1)
    return 0.5 * (ss + 2) + 4 + 3


# Relative band of every normalized output (RMSNorm rows and heads, the QK
# prologue's intermediate rounding, LayerNorm with its magnitude scale).
ETA_NORM = 2.0 ** -18

# Relative error bound of fp32 outputs against the exact value (at the pair
# norm for rotated channels): the benchmark spec's fp32 bar.
REL_F32 = 2e-6


def gate_error_coefficients(act):
    """(c0, c1): the fast gate's relative error is at most (c0 + c1 |v|) u, v the
    logistic argument (g for SiLU, 2z for tanh-GELU).

    t = e^-|v| comes from ex2.approx of -|v| log2(e).  A relative error e of
    that argument is an absolute error |v| e of the exponent, so t carries a
    relative error |v| e plus the instruction's 4u.  SiLU: e = 1.5u (the
    constant log2(e) and the product).  tanh-GELU: the exponent is formed as
    v log2(e) = K' g (1 + C g^2) with K' = 2 sqrt(2/pi) log2(e) rounded once:
    the constants K' and C (u/2 each), the products C g, (C g) g, K' g and
    the final product (u each), and the rounding of the sum 1 + C g^2 (u; it
    cannot cancel, since C g^2 >= 0): e = 6u.
    sigma = num / (1 + t) takes the add and rcp.approx (3u); the output
    g * u * sigma three products (3u).  Constant part: 4 + 3 + 3 = 10.
    """
    return (10.0, 1.5) if act == 0 else (10.0, 6.0)


# The gate bands: the coefficients above, the |v| term rounded up (SiLU 1.5 to
# 2, tanh-GELU 6 to 8).
GATE_BAND = {0: (10.0, 2.0), 1: (10.0, 8.0)}


def gate_eta(g, act):
    """Per-element relative band of the fast gates (bf16 / fp16 / FP8 outputs)."""
    g = np.asarray(g, np.float64)
    c0, c1 = GATE_BAND[act]
    if act == 0:
        v = g
    else:
        v = 2.0 * math.sqrt(2.0 / math.pi) * (g + 0.044715 * g ** 3)
    return (c0 + c1 * np.abs(v)) * U
