"""Reader for the hand-computed fixtures in tests/golden/.

File format: '#' comment lines (the citation and the hand working), then
blocks headed "<name> <rows> <cols>" followed by that many rows of numbers.
"""
import glob
import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(path):
    blocks = {}
    with open(path, encoding="utf-8") as f:
        lines = [ln.strip() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]
    i = 0
    while i < len(lines):
        name, r, c = lines[i].split()
        r, c = int(r), int(c)
        rows = [[float(x) for x in lines[i + 1 + k].split()] for k in range(r)]
        for row in rows:
            if len(row) != c:
                raise ValueError(f"{path}: block {name} has a row of {len(row)} != {c}")
        blocks[name] = np.array(rows, dtype=np.float64).reshape(r, c)
        i += 1 + r
    return blocks


def all_cases():
    return sorted(glob.glob(os.path.join(GOLDEN_DIR, "hand_*.txt")))
