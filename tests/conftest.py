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


# Parity bars: fp32 |y - ref| <= 1e-6 + 1e-5 |ref|; fp16/bf16 <= 1e-2 + 1e-2 |ref|.
TOL = {"float32": (1e-6, 1e-5), "float16": (1e-2, 1e-2), "bfloat16": (1e-2, 1e-2)}


def assert_parity(got, ref, dtype, what=""):
    """Element-wise comparison of a CUDA result (torch tensor) with oracle values."""
    import torch
    g = got.detach().to("cpu").to(torch.float64).numpy() if hasattr(got, "detach") else got
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    atol, rtol = TOL[dtype]
    err = np.abs(g - ref)
    bad = ~(err <= atol + rtol * np.abs(ref))
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err, -1)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside {atol} + {rtol}|ref| "
                             f"(worst at {i}: got {g[i]!r}, ref {ref[i]!r})")


@pytest.fixture(scope="session")
def gs_cuda():
    """The CUDA library, built for this machine; fails loudly when it cannot load."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without a CUDA device")
    from spatial_transformer_sampling_gb300 import build as gsbuild
    gsbuild.build()
    import spatial_transformer_sampling_gb300 as gs
    gs.load_library()
    return gs
