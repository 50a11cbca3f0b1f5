"""Readers for the hand-derived fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.strip()
    return out


def floats(s):
    return np.array([float(t) for t in s.split()], np.float64)


def codes(spec, n):
    if spec.startswith("range("):
        a, b = spec[6:-1].split(",")
        return np.arange(int(a), int(b))
    if spec.startswith("const("):
        return np.full(n, int(spec[6:-1]))
    return np.array([int(t) for t in spec.split()])
