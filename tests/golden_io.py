"""Reader for the hand-worked fixtures in tests/golden (test helper only)."""
import glob
import os
from fractions import Fraction

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(path):
    secs, cur, oracle_only = {}, None, False
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line == "oracle_only":
                oracle_only = True
                continue
            parts = line.split()
            if parts[0] in ("A", "B", "C_relu", "C_norelu"):
                cur = parts[0]
                secs[cur] = []
                continue
            secs[cur].append([Fraction(x) for x in parts])
    out = {"name": os.path.basename(path), "oracle_only": oracle_only}
    for key in ("A", "B"):
        vals = np.array([[float(v) for v in row] for row in secs[key]], dtype=np.float64)
        h = vals.astype(np.float16)
        assert np.array_equal(h.astype(np.float64), vals), f"{path}: {key} not exact in binary16"
        out[key] = h
    for key in ("C_relu", "C_norelu"):
        out[key] = secs[key]
    return out


def all_fixtures():
    return [load(p) for p in sorted(glob.glob(os.path.join(GOLDEN_DIR, "*.txt")))
            if not p.endswith("README.txt")]
