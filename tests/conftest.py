import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU")
    config.addinivalue_line("markers", "slow: long-running (full-size shapes)")


def read_golden(name):
    """Parse a ``key: v1 v2 ...`` fixture (``#`` starts a comment line)."""
    out = {}
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                key, val = line.split(":", 1)
                out[key.strip()] = val.split()
            else:
                rows.append(line.split())
    if rows:
        out["_rows"] = rows
    return out


@pytest.fixture(scope="session")
def cuda_lib():
    """The compiled CUDA library, built in-tree.  GPU tests only.

    Skips when no GPU is visible (the CPU-only container); on a machine with a
    GPU a missing or broken extension is an error, never a fallback.
    """
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device visible")
    from fp4_weight_only_gb300 import binding

    binding.load()   # raises if the library cannot be built or loaded
    return binding
