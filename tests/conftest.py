import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_addoption(parser):
    parser.addoption("--bounds-checked", action="store_true", default=False,
                     help="run every library call through libmxfp8_bc.so, the build with index "
                          "checks on every computed global access (a failed check sets the "
                          "device status the tests assert on)")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload parity")
    if config.getoption("--bounds-checked"):
        import mxfp8_precision_gemms_gb300 as m
        from mxfp8_precision_gemms_gb300 import _build
        m.LIB_PATH, m._lib = _build.build(bounds_check=True), None


def read_golden(name):
    """Parse a tests/golden/*.txt fixture: '# ...' comments, 'key value' lines."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, _, val = line.partition(" ")
            out[key] = val.strip()
    return out


def read_golden_table(name):
    rows = []
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def pow2_or_float(s):
    if s.startswith("2^"):
        return 2.0 ** int(s[2:])
    return float(s)
