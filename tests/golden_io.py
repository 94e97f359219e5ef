"""Readers for the hand-worked fixtures in tests/golden/ (comments start with '#')."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.rstrip("\n") for ln in f if ln.strip() and not ln.startswith("#")]


def read_fixture(name):
    """Key/value lines; a line 'mask' starts a 0/1 matrix that runs to the end."""
    out, mask = {}, None
    for ln in _lines(name):
        if mask is not None:
            mask.append([c == "1" for c in ln.strip()])
            continue
        if ln.strip() == "mask":
            mask = []
            continue
        key, *vals = ln.split()
        out[key] = vals
    if mask is not None:
        out["mask"] = np.array(mask, dtype=bool)
    return out


def read_cases(name):
    """Lines 'case <scores> | <k> | <expected indices>'."""
    cases = []
    for ln in _lines(name):
        assert ln.startswith("case ")
        scores, k, exp = ln[5:].split("|")
        cases.append((np.array([float(x) for x in scores.split()]), int(k),
                      [int(x) for x in exp.split()]))
    return cases
