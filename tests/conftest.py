import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled library")
    config.addinivalue_line("markers", "slow: long-running full-size case")


def read_fixture(name):
    """Parse a golden text fixture: '#' comments, then lines 'key v1 v2 ...'."""
    data = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            data.setdefault(key, []).append([float(v) for v in vals])
    return {k: (v[0] if len(v) == 1 else v) for k, v in data.items()}


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.lib()
    return oracle


def bf16_bits(values) -> np.ndarray:
    """Float values that are exactly representable in BF16 -> their bit patterns."""
    v = np.asarray(values, dtype=np.float32)
    bits = v.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (bits >> 16).astype(np.uint16)
