"""Parity with programmatic dependent launch switched off (EDGE_OPS_PDL=0).

The library reads the variable once per process, so a child pytest runs a
cross-section of the parity cases with it set: every kernel family, launched
without the programmatic-serialization attribute, must give the same results
as the oracle.  (The kernels' wait and trigger instructions are then no-ops.)
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))

SELECT = " or ".join([
    "test_benchmark_decode_step_matches_oracle",
    "test_runs_on_a_side_stream_and_in_a_cuda_graph",
    "test_positions_rewritten_by_the_preceding_kernel",
    "test_qk_norm_rope and (cfg1_f32 or cfg3_16_2_T333 or cfg4_bf16 or generic_odd_d37 or quad_f32_d128)",
    "test_rows and (cfg2_h2560_T64_direct or h2560_T700_ragged or generic_h37 or f16_h1024_T33)",
    "test_glu and (cfg2_T64 or generic_d37 or f32_accurate)",
    "test_layernorm and not fp8",
    "test_quantize_fp8",
    "test_qkv_rope_cache",
    "test_rope",
])


def test_parity_cases_with_dependent_launch_off():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, EDGE_OPS_PDL="0")
    # the child's cases would repeat the parent's lines in a stats dump
    env.pop("EDGE_OPS_REPORT_STATS", None)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(HERE, "test_gpu_parity.py"),
                        "-q", "-x", "-p", "no:cacheprovider", "-k", SELECT],
                       env=env, capture_output=True, text=True, timeout=1200)
    tail = (r.stdout[-3000:] + r.stderr[-2000:])
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " deselected" in r.stdout, tail
