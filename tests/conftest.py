"""Shared pytest configuration: the ``gpu`` marker and fixture helpers."""

import math
import os
import re
import sys
from fractions import Fraction

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built libsaf")


_TOKEN = re.compile(r"^(-?)(?:(\d+(?:/\d+)?)\*)?(ln\(([^)]*)\)|[-\d./]+)$")


def _value(tok: str) -> float:
    """Parse '3/4', '-1', 'ln(5/2)', '-3/4*ln(3)' into a float."""
    m = _TOKEN.match(tok)
    if not m:
        raise ValueError(f"bad golden token {tok!r}")
    sign, coef, body, lnarg = m.groups()
    c = Fraction(coef) if coef else Fraction(1)
    if lnarg is not None:
        v = float(c) * math.log(Fraction(lnarg))
    else:
        v = float(c * Fraction(body))
    return -v if sign else v


def load_golden(name: str) -> dict:
    """Read a tests/golden/*.txt fixture into {key: np.ndarray}."""
    rows: dict = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, vals = (s.strip() for s in line.split("=", 1))
            arr = [_value(t) for t in vals.split()]
            m = re.match(r"^(\w+)\[(\d+)\]$", key)
            if m:
                rows.setdefault(m.group(1), {})[int(m.group(2))] = arr
            else:
                rows[key] = np.array(arr)
    out = {}
    for k, v in rows.items():
        out[k] = np.array([v[i] for i in sorted(v)]) if isinstance(v, dict) else v
    return out


@pytest.fixture
def golden():
    return load_golden

TESTS = os.path.join(ROOT, "tests")
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)
