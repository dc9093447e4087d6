"""Reader for the hand-worked fixtures under tests/golden/.

A fixture file holds one or more ``case:`` blocks.  Scalars are ``key: value``
lines; matrices are a ``name:`` line followed by rows of numbers.  Lines that
start with ``#`` are comments (the worked arithmetic lives there).
"""

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_MATS = {"A", "B", "C0", "bias", "row_bias", "expect", "mag"}


def load(name):
    cases, cur, mat = [], None, None
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                mat = None if not line else mat
                continue
            if ":" in line and line.split(":")[0].strip() in _MATS | {
                    "case", "M N K", "alpha", "beta", "relu"}:
                key, _, val = line.partition(":")
                key, val = key.strip(), val.strip()
                if key == "case":
                    cur = {"name": val}
                    cases.append(cur)
                    mat = None
                elif key in _MATS:
                    cur[key] = []
                    mat = key
                elif key == "M N K":
                    cur["M"], cur["N"], cur["K"] = (int(x) for x in val.split())
                elif key == "relu":
                    cur["relu"] = bool(int(val))
                else:
                    cur[key] = float(val)
                continue
            if mat is None:
                raise ValueError("stray line in %s: %r" % (name, raw))
            cur[mat].append([float(x) for x in line.split()])
    for c in cases:
        for k in _MATS:
            if k in c:
                c[k] = np.array(c[k], dtype=np.float64)
        for k in ("bias", "row_bias"):
            if k in c:
                c[k] = c[k].reshape(-1)
    return cases
