"""Optional per-case statistics of the parity checks, for diffing two runs.

With ``EDGE_OPS_REPORT_STATS=<file>`` in the environment, every output check of
the GPU parity tests appends one line to <file>: the case (pytest node id and
the check's name), the element count, a digest of the output's bits, how many
elements equal the oracle's rounding and how many sit one ulp from it, the
largest ulp distance, and the largest error relative to the magnitude scale,
printed with ``%.17g`` so that nothing is lost to formatting.  Two runs (two
machines, two builds, programmatic dependent launch on and off) are then
compared case by case:

    python tests/case_stats.py A.txt B.txt

prints the number of shared cases and every shared case whose line differs,
and exits 1 if any does.  (The ninfer PR's "Output" section describes the
same practice: a stats dump of every case at %.17g, diffed across two bases.)
"""
from __future__ import annotations

import hashlib
import os
import sys

import numpy as np

ENV = "EDGE_OPS_REPORT_STATS"


def enabled() -> bool:
    return bool(os.environ.get(ENV))


def case_id(name: str) -> str:
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    return f"{test}::{name}" if test else name


def format_line(case: str, got: np.ndarray, ulp: np.ndarray | None = None,
                rel: np.ndarray | None = None) -> str:
    got = np.ascontiguousarray(got)
    fields = [case, f"n={got.size}", "sha=" + hashlib.sha256(got.tobytes()).hexdigest()[:16]]
    if ulp is not None:
        ulp = np.asarray(ulp).ravel()
        fields += [f"exact={int(np.count_nonzero(ulp == 0))}",
                   f"one_ulp={int(np.count_nonzero(ulp == 1))}",
                   f"max_ulp={int(ulp.max()) if ulp.size else 0}"]
    if rel is not None:
        rel = np.asarray(rel, np.float64).ravel()
        fields.append("max_rel=%.17g" % (float(rel.max()) if rel.size else 0.0))
    return " ".join(fields)


def record(name: str, got: np.ndarray, ulp: np.ndarray | None = None,
           rel: np.ndarray | None = None) -> None:
    """Append the case's line to the stats file, if one is named."""
    path = os.environ.get(ENV)
    if not path:
        return
    with open(path, "a") as f:
        f.write(format_line(case_id(name), got, ulp, rel) + "\n")


def load(path: str) -> dict[str, str]:
    """Case -> the rest of its line; a case recorded twice gets #2, #3, ..."""
    out: dict[str, str] = {}
    with open(path) as f:
        for line in f:
            line = line.rstrip("\n")
            if not line:
                continue
            case, _, rest = line.partition(" ")
            key, k = case, 1
            while key in out:
                k += 1
                key = f"{case}#{k}"
            out[key] = rest
    return out


def diff(a: dict[str, str], b: dict[str, str]) -> tuple[int, list[str]]:
    shared = sorted(set(a) & set(b))
    return len(shared), [c for c in shared if a[c] != b[c]]


def main(argv: list[str]) -> int:
    if len(argv) != 2:
        print("usage: python tests/case_stats.py A.txt B.txt", file=sys.stderr)
        return 2
    a, b = load(argv[0]), load(argv[1])
    n, bad = diff(a, b)
    print(f"{n} shared cases, {len(bad)} differing "
          f"({len(a) - n} only in {argv[0]}, {len(b) - n} only in {argv[1]})")
    for c in bad:
        print(f"{c}\n  {a[c]}\n  {b[c]}")
    return 1 if bad else 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
