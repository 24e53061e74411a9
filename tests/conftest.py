import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_path(name):
    return os.path.join(GOLDEN, name)


def read_golden(name):
    """Parse a golden fixture: '#' comment lines, then 'key: value' lines
    whose values are whitespace-separated numbers (ints or floats or 0x hex)."""
    out = {}
    with open(golden_path(name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            vals = []
            for tok in v.split():
                if tok.startswith("0x"):
                    vals.append(int(tok, 16))
                elif any(c in tok for c in ".eE") and not tok.lstrip("-").isdigit():
                    vals.append(float(tok))
                else:
                    vals.append(int(tok))
            out[k.strip()] = vals
    return out
