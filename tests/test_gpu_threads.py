"""First calls from several host threads at once.

The library's only host-side state is per-device setup done by the first call
that needs it (kernel shared-memory limits, the error word's and the static
scratch's device addresses), kept in atomics.  A fresh process starts eight
threads that all make their first calls together, each on its own CUDA stream,
through the fused 2-D path, both 3-D kernels (gather and TMA-staged boxes),
the staged Resize kernel, and the staged, channel-last and fp32 windowed
DeformConv kernels; every result is then compared with the oracle."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, threading
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
import oracle
import spatial_transformer_sampling_gb300 as gs
from spatial_transformer_sampling_gb300 import workloads as wl
from conftest import assert_parity

gs.load_library()
dev = torch.device("cuda:0")
torch.cuda.set_device(dev)
T = 8
g = wl.rng(1234)
cases = []
for t in range(T):
    th2 = wl.as_dtype(wl.identity_theta(2, 2) + g.normal(0, 0.1, (2, 2, 3)), "bfloat16")
    X2 = wl.as_dtype(g.normal(size=(2, 4, 40, 36)), "bfloat16")
    th3 = wl.as_dtype(wl.identity_theta(1, 3) + g.normal(0, 0.1, (1, 3, 4)), "float32")
    X3 = wl.as_dtype(g.normal(size=(1, 2, 12, 13, 14)), "float32")
    Xr = wl.as_dtype(g.normal(size=(1, 3, 20, 24)), "bfloat16")
    Xd = wl.as_dtype(g.normal(size=(1, 16, 9, 10)), "bfloat16")
    Wd = wl.as_dtype(g.normal(0, 0.05, size=(16, 16, 3, 3)), "bfloat16")
    Od = wl.as_dtype(g.normal(0, 1, size=(1, 18, 9, 10)), "bfloat16")
    # widths in whole 16-byte runs: the TMA 3-D kernel, the staged bf16 and the
    # windowed fp32 DeformConv
    X3b = wl.as_dtype(g.normal(size=(1, 2, 12, 13, 16)), "float32")
    Xs = wl.as_dtype(g.normal(size=(1, 16, 9, 16)), "bfloat16")
    Os = wl.as_dtype(g.normal(0, 1, size=(1, 18, 9, 16)), "bfloat16")
    Xf = wl.as_dtype(g.normal(size=(1, 16, 9, 16)), "float32")
    Wf = wl.as_dtype(g.normal(0, 0.05, size=(16, 16, 3, 3)), "float32")
    Of = wl.as_dtype(g.normal(0, 1, size=(1, 18, 9, 16)), "float32")
    cases.append((th2, X2, th3, X3, Xr, Xd, Wd, Od, X3b, Xs, Os, Xf, Wf, Of))
results = [None] * T
start = threading.Barrier(T)

def work(t):
    th2, X2, th3, X3, Xr, Xd, Wd, Od, X3b, Xs, Os, Xf, Wf, Of = [c.to(dev) for c in cases[t]]
    s = torch.cuda.Stream(dev)
    torch.cuda.synchronize(dev)
    start.wait()
    with torch.cuda.stream(s):
        r = (gs.gs_affine_sample(th2, (2, 4, 30, 34), X2, "linear", "border", 1),
             gs.gs_affine_sample(th3, (1, 2, 10, 11, 12), X3, "linear", "zeros", 0),
             gs.gs_resize(Xr, scales=(1, 1, 2, 2), mode="linear"),
             gs.gs_deform_conv(Xd, Wd, Od, pads=(1, 1, 1, 1), workspace="auto"),
             gs.gs_affine_sample(th3, (1, 2, 10, 11, 12), X3b, "linear", "zeros", 0),
             gs.gs_deform_conv(Xs, Wd, Os, pads=(1, 1, 1, 1)),
             gs.gs_deform_conv(Xf, Wf, Of, pads=(1, 1, 1, 1)))
    s.synchronize()
    results[t] = [y.cpu() for y in r]

threads = [threading.Thread(target=work, args=(t,)) for t in range(T)]
for th in threads: th.start()
for th in threads: th.join()
assert gs.gs_device_status() == 0
for t in range(T):
    th2, X2, th3, X3, Xr, Xd, Wd, Od, X3b, Xs, Os, Xf, Wf, Of = [wl.widened(c) for c in cases[t]]
    y2, y3, yr, yd, y3b, ys, yf = results[t]
    assert_parity(y2, oracle.affine_sample(th2, (2, 4, 30, 34), X2, "linear", "border", 1),
                  "bfloat16", f"thread {t} affine 2-D")
    assert_parity(y3, oracle.affine_sample(th3, (1, 2, 10, 11, 12), X3, "linear", "zeros", 0),
                  "float32", f"thread {t} affine 3-D")
    assert_parity(yr, oracle.resize(Xr, scales=(1, 1, 2, 2), mode="linear"),
                  "bfloat16", f"thread {t} resize")
    assert_parity(yd, oracle.deform_conv(Xd, Wd, Od, pads=(1, 1, 1, 1)), "bfloat16",
                  f"thread {t} deform")
    assert_parity(y3b, oracle.affine_sample(th3, (1, 2, 10, 11, 12), X3b, "linear", "zeros", 0),
                  "float32", f"thread {t} affine 3-D, staged boxes")
    assert_parity(ys, oracle.deform_conv(Xs, Wd, Os, pads=(1, 1, 1, 1)), "bfloat16",
                  f"thread {t} deform, staged")
    assert_parity(yf, oracle.deform_conv(Xf, Wf, Of, pads=(1, 1, 1, 1)), "float32",
                  f"thread {t} deform fp32, windowed")
print("threads ok")
"""


def test_first_calls_from_eight_host_threads(gs_cuda, oracle_mod):
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
