import os
import sys
from fractions import Fraction

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size case, minutes of oracle time")


def pytest_runtest_setup(item):
    # A GPU test never passes or skips silently without a device: it fails.
    if "gpu" in item.keywords:
        import torch
        if not torch.cuda.is_available():
            pytest.fail("test marked gpu but no CUDA device is visible")


def read_golden(name):
    """Parse a golden text fixture: 'key: values' lines and matrix blocks
    ('key:' followed by rows).  Values may be ints, floats or p/q rationals."""
    out, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if ":" in line:
                key, rest = line.split(":", 1)
                rest = rest.strip()
                if rest:
                    out[key.strip()] = [Fraction(v) for v in rest.split()]
                    cur = None
                else:
                    cur = key.strip()
                    out[cur] = []
            else:
                out[cur].append([Fraction(v) for v in line.split()])
    return out


def as_f64(vals):
    return np.array([[float(v) for v in row] for row in vals]) if vals and isinstance(
        vals[0], list) else np.array([float(v) for v in vals])
