"""The C ABI without a GPU: exports, and validation before any launch.

Every entry point validates all arguments before pointer arithmetic or a
launch ("thox-edge-ops v2", section 5.5).  So invalid calls can be made here
with made-up pointer values: no pointer is dereferenced and no kernel runs.
"""
import ctypes
import os
import re
import subprocess

import pytest

from memory_bound_decode_qk_gb300 import _build, edge_ops

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "edge_ops.h")

OK, NULL, DTYPE, SHAPE, ALIGN, ALIAS, UNSUP, CUDA, VALUE = range(9)
F32, F16, BF16, FP8 = 0, 1, 2, 3


@pytest.fixture(scope="module")
def L():
    _build.build()
    return edge_ops.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(edge_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("edge_qk_norm_rope", "edge_add_rmsnorm", "edge_rmsnorm", "edge_glu_act",
              "edge_status_str", "edge_version"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in declared_functions():
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r"\bT (edge_\w+)", out))
    assert set(declared_functions()) <= exported


def test_binding_names_match_header():
    assert set(edge_ops.EXPORTS) == set(declared_functions())


def test_version_and_status_strings(L):
    assert L.edge_version() == 100
    for s in range(9):
        assert L.edge_status_str(s)
    assert L.edge_status_str(42) == b"unknown status"
    assert L.edge_last_cuda_error() == 0


# Fake, suitably aligned device addresses: never dereferenced by validation.
X, R, W, O, O2 = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000


def rms(L, out=O, out_dt=BF16, x=X, w=W, dt=BF16, rows=4, hidden=64, eps=1e-6, off=0, inv=1.0):
    return L.edge_rmsnorm(out, out_dt, x, w, dt, rows, hidden, eps, off, inv, None)


def add(L, out=O, out_dt=BF16, x=X, r=R, w=W, dt=BF16, rows=4, hidden=64, eps=1e-6, off=0, inv=1.0):
    return L.edge_add_rmsnorm(out, out_dt, x, r, w, dt, rows, hidden, eps, off, inv, None)


def glu(L, out=O, out_dt=BF16, gu=X, dt=BF16, rows=4, d=64, act=0, inv=1.0):
    return L.edge_glu_act(out, out_dt, gu, dt, rows, d, act, inv, None)


QO, KO, Q, K, WQ, WK, POS, COS, SIN = (0x1000000, 0x2000000, 0x3000000, 0x4000000, 0x5000000,
                                       0x5100000, 0x6000000, 0x7000000, 0x8000000)


def qk(L, qo=QO, ko=KO, out_dt=BF16, q=Q, k=K, wq=WQ, wk=WK, dt=BF16, T=4, Hq=8, Hk=2, D=128,
       rot=64, layout=0, pos=POS, cos=COS, sin=SIN, P=4096, eps=1e-6, off=1, inv=1.0):
    return L.edge_qk_norm_rope(qo, ko, out_dt, q, k, wq, wk, dt, T, Hq, Hk, D, rot, layout, pos,
                               cos, sin, P, eps, off, inv, None)


def test_zero_rows_is_ok_and_launches_nothing(L):
    assert L.edge_rope(QO, KO, BF16, Q, K, BF16, 0, 8, 2, 128, 64, 0, POS, COS, SIN, 4096, 1.0,
                       None) == OK
    assert rms(L, rows=0) == OK
    assert L.edge_layernorm(O, BF16, X, W, None, BF16, 0, 64, 1e-5, 1.0, None) == OK
    assert L.edge_quantize_fp8(O, X, BF16, 0, 1.0, None) == OK
    assert add(L, rows=0) == OK
    assert glu(L, rows=0) == OK
    assert qk(L, T=0) == OK
    assert L.edge_copy(O, X, 0, None) == OK
    # no CUDA call was made: no sticky error recorded
    assert L.edge_last_cuda_error() == 0


@pytest.mark.parametrize("call,status", [
    (lambda L: rms(L, x=None), NULL),
    (lambda L: rms(L, out=None), NULL),
    (lambda L: add(L, r=None), NULL),
    (lambda L: glu(L, gu=None), NULL),
    (lambda L: qk(L, q=None), NULL),
    (lambda L: qk(L, k=None), NULL),
    (lambda L: qk(L, pos=None), NULL),
    (lambda L: qk(L, cos=None), NULL),
    (lambda L: rms(L, dt=FP8, out_dt=FP8), DTYPE),
    (lambda L: rms(L, dt=7), DTYPE),
    (lambda L: rms(L, dt=BF16, out_dt=F16), DTYPE),
    (lambda L: qk(L, dt=F32, out_dt=BF16), DTYPE),
    (lambda L: rms(L, rows=-1), SHAPE),
    (lambda L: rms(L, hidden=0), SHAPE),
    (lambda L: glu(L, d=0), SHAPE),
    (lambda L: qk(L, rot=65), SHAPE),
    (lambda L: qk(L, rot=130), SHAPE),
    (lambda L: qk(L, Hq=0), SHAPE),
    (lambda L: qk(L, P=-1), SHAPE),
    (lambda L: rms(L, rows=2 ** 62, hidden=2 ** 10), SHAPE),
    (lambda L: rms(L, eps=-1.0), VALUE),
    (lambda L: rms(L, eps=float("nan")), VALUE),
    (lambda L: rms(L, off=2), VALUE),
    (lambda L: rms(L, out_dt=FP8, inv=0.0), VALUE),
    (lambda L: rms(L, out_dt=FP8, inv=float("inf")), VALUE),
    (lambda L: glu(L, act=5), VALUE),
    (lambda L: qk(L, layout=2), VALUE),
    (lambda L: rms(L, x=X + 1), ALIGN),
    (lambda L: rms(L, out=O + 1), ALIGN),
    (lambda L: rms(L, dt=F32, out_dt=F32, x=X + 2), ALIGN),
    (lambda L: qk(L, pos=POS + 4), ALIGN),
    (lambda L: qk(L, cos=COS + 2), ALIGN),
    (lambda L: qk(L, D=4096, rot=64), UNSUP),
    (lambda L: L.edge_qk_norm_rope_ex(QO, KO, BF16, Q, K, WQ, WK, BF16, 4, 8, 2, 128, 64, 0, POS,
                                      COS, SIN, 4096, 1e-6, 1, 1.0, 2, None), VALUE),
    (lambda L: L.edge_rope(QO, KO, BF16, None, K, BF16, 4, 8, 2, 128, 64, 0, POS, COS, SIN,
                           4096, 1.0, None), NULL),
    (lambda L: L.edge_rope(QO, KO, BF16, Q, K, BF16, 4, 8, 2, 128, 63, 0, POS, COS, SIN,
                           4096, 1.0, None), SHAPE),
    (lambda L: L.edge_rope(Q + 2, KO, BF16, Q, K, BF16, 4, 8, 2, 128, 64, 0, POS, COS, SIN,
                           4096, 1.0, None), ALIAS),
    (lambda L: L.edge_layernorm(O, BF16, None, W, W + 4096, BF16, 4, 64, 1e-5, 1.0, None), NULL),
    (lambda L: L.edge_layernorm(O, BF16, X, W, W + 4096, BF16, 4, 64, -1.0, 1.0, None), VALUE),
    (lambda L: L.edge_layernorm(X + 2, BF16, X, W, W + 4096, BF16, 4, 64, 1e-5, 1.0, None), ALIAS),
    (lambda L: L.edge_layernorm(O, FP8, X, W, W + 4096, BF16, 4, 64, 1e-5, 0.0, None), VALUE),
    (lambda L: L.edge_quantize_fp8(O, X, BF16, -1, 1.0, None), SHAPE),
    (lambda L: L.edge_quantize_fp8(O, X, FP8, 16, 1.0, None), DTYPE),
    (lambda L: L.edge_quantize_fp8(O, X, BF16, 16, float("nan"), None), VALUE),
    (lambda L: L.edge_quantize_fp8(X + 8, X, BF16, 16, 1.0, None), ALIAS),
    (lambda L: L.edge_quantize_fp8(O, X + 1, BF16, 16, 1.0, None), ALIGN),
    (lambda L: L.edge_qkv_rope_cache(QO, KO, KO + 65536, Q, WQ, WK, BF16, 4, 8, 2, 128, 64, 0,
                                     POS, COS, SIN, 4096, None, 16, 1e-6, 0, 1, None), NULL),
    (lambda L: L.edge_qkv_rope_cache(QO, KO, KO, Q, WQ, WK, BF16, 4, 8, 2, 128, 64, 0, POS, COS,
                                     SIN, 4096, POS + 4096, 16, 1e-6, 0, 1, None), ALIAS),
    (lambda L: L.edge_qkv_rope_cache(QO, KO, KO + 65536, Q, WQ, WK, BF16, 4, 8, 2, 128, 64, 0,
                                     POS, COS, SIN, 4096, POS + 4096, 16, 1e-6, 0, 2, None), VALUE),
    (lambda L: L.edge_qkv_rope_cache(QO, KO, KO + 65536, Q, WQ, WK, FP8, 4, 8, 2, 128, 64, 0,
                                     POS, COS, SIN, 4096, POS + 4096, 16, 1e-6, 0, 1, None), DTYPE),
    (lambda L: L.edge_copy(None, X, 16, None), NULL),
    (lambda L: L.edge_copy(O, None, 16, None), NULL),
    (lambda L: L.edge_copy(O, X, -1, None), SHAPE),
    (lambda L: L.edge_copy(X + 8, X, 16, None), ALIAS),
    (lambda L: L.edge_copy(X, X + 15, 16, None), ALIAS),
    (lambda L: rms(L, hidden=2 ** 25, rows=1), UNSUP),
    # one past each declared limit: rows of 2**24, heads of 2048, 2**31 - 1 units
    (lambda L: rms(L, hidden=2 ** 24 + 8, rows=1), UNSUP),
    (lambda L: add(L, hidden=2 ** 24 + 8, rows=1), UNSUP),
    (lambda L: L.edge_layernorm(O, BF16, X, W, None, BF16, 1, 2 ** 24 + 8, 1e-5, 1.0, None),
     UNSUP),
    (lambda L: qk(L, D=2050, rot=64), UNSUP),
    (lambda L: qk(L, T=2 ** 28, Hq=8, Hk=0, k=None), UNSUP),
    (lambda L: L.edge_rope(QO, KO, BF16, Q, K, BF16, 4, 8, 2, 2050, 64, 0, POS, COS, SIN,
                           4096, 1.0, None), UNSUP),
    (lambda L: L.edge_qkv_rope_cache(QO, KO, KO + 2 ** 20, Q, WQ, WK, BF16, 4, 8, 2, 2050, 64, 0,
                                     POS, COS, SIN, 4096, POS + 4096, 16, 1e-6, 0, 1, None),
     UNSUP),
])
def test_invalid_calls_are_rejected(L, call, status):
    assert call(L) == status


def test_aliasing_rules(L):
    n = 4 * 64 * 2  # bytes of x
    # partial overlaps of a written buffer are rejected before any launch
    assert rms(L, out=X + 2) == ALIAS
    assert rms(L, out=W - 16) == ALIAS                      # output runs into the weight
    assert rms(L, out_dt=FP8, out=X) == ALIAS               # FP8 output cannot be in place
    assert add(L, r=X) == ALIAS                             # residual is x
    assert add(L, r=X + n - 2) == ALIAS                     # residual overlaps x's tail
    assert add(L, out=R) == ALIAS                           # out overwrites the residual
    assert glu(L, out=X + 64) == ALIAS                      # output inside gate_up
    assert qk(L, qo=Q + 2) == ALIAS
    assert qk(L, ko=Q) == ALIAS                              # k_out writes over q
    assert qk(L, qo=KO) == ALIAS                             # both outputs in one buffer
    assert qk(L, qo=COS) == ALIAS                            # output over the cache
    assert qk(L, ko=POS) == ALIAS                            # output over positions
    assert qk(L, out_dt=FP8, qo=Q) == ALIAS                  # FP8 output cannot be in place


def test_fastdiv_matches_division(tmp_path):
    # the multiply-high division used to flatten indices (Granlund-Montgomery)
    src = tmp_path / "fd.cpp"
    src.write_text(r'''
#include "fastdiv.h"
#include <cstdio>
#include <cstdint>
int main() {
  uint32_t ds[] = {1, 2, 3, 5, 7, 28, 18, 40, 1216, 1280, 9728, 4096, 12345, 65535,
                   2147483647u, 2147483648u, 4294967295u};
  uint32_t ns[] = {0, 1, 2, 3, 27, 28, 29, 1215, 1216, 1217, 65535, 65536, 1u << 31,
                   (1u << 31) - 1, 4294967295u, 4294967294u, 123456789u};
  unsigned long bad = 0;
  for (uint32_t d : ds) {
    edge::FastDiv f = edge::make_fastdiv(d);
    for (uint32_t n : ns) bad += edge::fast_div(n, f) != n / d;
    uint64_t x = 88172645463325252ull;
    for (int i = 0; i < 200000; ++i) {
      x ^= x << 13; x ^= x >> 7; x ^= x << 17;
      uint32_t n = (uint32_t)x;
      bad += edge::fast_div(n, f) != n / d;
    }
  }
  for (uint32_t d = 1; d < 3000; ++d) {
    edge::FastDiv f = edge::make_fastdiv(d);
    for (uint32_t n = 0; n < 20000; n += 7) bad += edge::fast_div(n, f) != n / d;
  }
  std::printf("%lu\n", bad);
  return bad != 0;
}
''')
    exe = tmp_path / "fd"
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", os.path.join(ROOT, "memory_bound_decode_qk_gb300", "csrc"),
                    str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "0"


def test_binding_raises_without_fallback(monkeypatch, tmp_path):
    # the product path fails loudly when the library is missing
    monkeypatch.setattr(edge_ops, "_LIB", None)
    monkeypatch.setattr(edge_ops._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        edge_ops.lib()
