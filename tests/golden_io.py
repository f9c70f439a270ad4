"""Readers for the hand-derived text fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.strip() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]


def blocks(name):
    """Fixture of named blocks: a header line (starts with a letter) followed by rows of numbers."""
    out, key = {}, None
    for ln in _lines(name):
        if ln[0].isalpha():
            key = ln
            out[key] = []
        else:
            out[key].append(ln.split())
    return out


def csv_rows(name):
    rows = [ln.split(",") for ln in _lines(name)]
    return rows[0], rows[1:]


def as_array(rows, dtype):
    if dtype is np.uint8:
        return np.array([[int(v, 16) for v in r] for r in rows], dtype=np.uint8)
    return np.array([[float(v) for v in r] for r in rows]).astype(dtype)
