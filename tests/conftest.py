import json
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")


def load_fixture(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def fixture_names(prefix):
    return sorted(n for n in os.listdir(GOLDEN) if n.startswith(prefix) and n.endswith(".json"))


def fixture_array(entry):
    """A fixture tensor as float64, first rounded to the dtype the page declares."""
    a = np.array(entry["data"], dtype=np.float64).reshape(entry["shape"])
    if entry["dtype"] == "float32":
        a = a.astype(np.float32).astype(np.float64)
    elif entry["dtype"] == "int64":
        a = a.astype(np.int64)
    return a


def page_close(got, expected):
    """Agreement with values the pages print (fp32 results printed to ~8 digits)."""
    got = np.asarray(got, dtype=np.float64)
    return np.abs(got - expected) <= 2e-6 + 1e-6 * np.abs(expected)


def gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.lib()
    return oracle
