"""The optional per-case statistics dump (tests/case_stats.py), on the CPU."""
import numpy as np

import case_stats


def test_line_format_and_digits(tmp_path, monkeypatch):
    path = tmp_path / "a.txt"
    monkeypatch.setenv(case_stats.ENV, str(path))
    monkeypatch.setenv("PYTEST_CURRENT_TEST", "tests/x.py::test_y[c1] (call)")
    got = np.array([1, 2, 3, 4], np.uint16)
    case_stats.record("out", got, np.array([0, 0, 1, 3]), np.array([0.0, 1.0 / 3.0, 0.25, 0.0]))
    line = path.read_text().strip()
    assert line.startswith("tests/x.py::test_y[c1]::out n=4 sha=")
    assert "exact=2 one_ulp=1 max_ulp=3" in line
    # %.17g: the double round-trips exactly
    rel = float(line.split("max_rel=")[1])
    assert rel == 1.0 / 3.0 and "max_rel=0.33333333333333331" in line


def test_disabled_writes_nothing(tmp_path, monkeypatch):
    monkeypatch.delenv(case_stats.ENV, raising=False)
    assert not case_stats.enabled()
    case_stats.record("out", np.zeros(3, np.uint8))
    assert not list(tmp_path.iterdir())


def test_diff_of_two_runs(tmp_path, monkeypatch):
    a, b = tmp_path / "a.txt", tmp_path / "b.txt"
    monkeypatch.setenv("PYTEST_CURRENT_TEST", "t::case (call)")
    x = np.arange(8, dtype=np.uint16)
    for path, last in ((a, 7), (b, 6)):
        monkeypatch.setenv(case_stats.ENV, str(path))
        case_stats.record("q", x)
        case_stats.record("q", x)          # a second check of the same name
        y = x.copy()
        y[-1] = last
        case_stats.record("k", y)
    A, B = case_stats.load(str(a)), case_stats.load(str(b))
    assert set(A) == {"t::case::q", "t::case::q#2", "t::case::k"}
    shared, bad = case_stats.diff(A, B)
    assert shared == 3 and bad == ["t::case::k"]
    assert case_stats.main([str(a), str(a)]) == 0
    assert case_stats.main([str(a), str(b)]) == 1
