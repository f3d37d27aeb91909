"""Reader for the small text fixtures under tests/golden/ ("key: v1 v2 ..." lines)."""

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            out[key.strip()] = val.split()
    return out


def ints(d, key):
    return np.array([int(x) for x in d[key]], dtype=np.int64)


def floats(d, key):
    return np.array([float(x) for x in d[key]], dtype=np.float32)
