import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def read_golden(name):
    """Parses a whitespace-separated fixture, skipping '#' comment lines."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def golden_kv(name):
    return {r[0]: r[1:] for r in read_golden(name)}


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def ordered_bits(t):
    """Maps float tensors (CPU) to integers whose differences count ulps."""
    import torch
    if t.dtype == torch.float32:
        i = t.contiguous().view(torch.int32).to(torch.int64)
        mag = i & 0x7FFFFFFF
    else:
        i = t.contiguous().view(torch.int16).to(torch.int64)
        mag = i & 0x7FFF
    return torch.where(i < 0, -mag, mag)


def ulp_distance(a, b):
    """Elementwise distance in units in the last place of a's dtype."""
    return (ordered_bits(a) - ordered_bits(b.to(a.dtype))).abs()


def gpu_ready():
    import torch
    return torch.cuda.is_available()
