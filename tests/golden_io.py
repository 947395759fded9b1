"""Readers for the small text fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_keyed(name):
    """'key: numbers' lines -> {key: float64 array}; '#' starts a comment."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, vals = line.split(":", 1)
            out[key.strip()] = np.array([float(x) for x in vals.split()], dtype=np.float64)
    return out


def read_codes(name):
    """'<fmt> <hex code> <value>' lines -> list of (fmt, code, value)."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            fmt, code, val = line.split()
            rows.append((fmt, int(code, 16), float(val)))
    return rows
