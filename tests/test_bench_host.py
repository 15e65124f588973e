"""Host-side logic of the benchmark that needs no GPU: the staleness check of
the stored ncu traffic record."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _copy_sources(tmp_path):
    csrc = tmp_path / "memory_bound_decode_qk_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = os.path.join(ROOT, "memory_bound_decode_qk_gb300", "csrc")
    for name in ("rows.cu", "edge_common.cuh"):
        shutil.copy(os.path.join(src, name), csrc / name)
    return csrc


def test_source_hash_ignores_comments_and_sees_code(tmp_path, monkeypatch):
    csrc = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.source_sha("rows_vec_kernel")
    rows = csrc / "rows.cu"
    text = rows.read_text()
    # a comment and a blank line added: no kernel changed
    rows.write_text("// a note\n\n" + text.replace("{", "{ /* x */", 1))
    assert bench.source_sha("rows_vec_kernel") == base
    # a constant changed: the record must go stale
    rows.write_text(text.replace("return v;", "return v + 0.0f;", 1))
    assert bench.source_sha("rows_vec_kernel") != base


def test_committed_traffic_record_matches_the_current_kernel():
    # the record under profiles/ was captured from the current code of the
    # dominant kernel, so the bench reports its traffic rather than null
    assert bench.traffic_for("rows_vec_kernel") is not None
