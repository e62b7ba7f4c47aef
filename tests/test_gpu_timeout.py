"""The bounded device-side wait runs out, on purpose and safely.

Every pipelined kernel waits on mbarriers with a time limit, after which it
records GS_ERR_TIMEOUT in the library's device error word and returns instead
of hanging.  gs_test_bounded_wait_expires arms an mbarrier for bytes that no
copy will deliver and waits on it with a 1 ms limit, so the wait must expire:
the kernel returns, gs_device_status reports GS_ERR_TIMEOUT once and GS_OK on
the next call, and an operator call afterwards still matches the oracle."""
import time

import pytest
import torch

from conftest import assert_parity
from spatial_transformer_sampling_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

GS_OK, GS_ERR_TIMEOUT = 0, 8


def test_bounded_wait_expires_and_the_context_stays_usable(gs_cuda, oracle_mod):
    L = gs_cuda.load_library()
    torch.cuda.synchronize()
    assert gs_cuda.gs_device_status() == GS_OK
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    assert L.gs_test_bounded_wait_expires(1_000_000, stream) == GS_OK
    torch.cuda.synchronize()            # the kernel returned
    waited = time.perf_counter() - t0
    assert waited >= 1e-3, waited       # it did wait for the limit
    assert gs_cuda.gs_device_status() == GS_ERR_TIMEOUT
    assert gs_cuda.gs_device_status() == GS_OK   # reading the word cleared it

    g = wl.rng(4242)
    theta = wl.as_dtype(wl.identity_theta(2, 2) + g.normal(0, 0.1, (2, 2, 3)), "float32")
    X = wl.as_dtype(g.normal(size=(2, 8, 40, 36)), "float32")
    size = (2, 8, 33, 35)
    Y = gs_cuda.gs_affine_sample(theta.cuda(), size, X.cuda(), "linear", "border", 1)
    assert gs_cuda.gs_device_status() == GS_OK
    ref = oracle_mod.affine_sample(wl.widened(theta), size, wl.widened(X), "linear", "border", 1)
    assert_parity(Y, ref, "float32", "fused affine sample after an expired wait")
