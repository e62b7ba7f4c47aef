"""GridSample at spatial ranks 4 to 6 on the GPU against the oracle.

GridSample - version 20 defines the operator for an X of any rank r+2; ranks 4
to 6 run on the rank-general kernel.  Seeded inputs, element by element: fp32
|y - ref| <= 1e-6 + 1e-5|ref|, fp16/bf16 <= 1e-2 + 1e-2|ref|, nearest bit for
bit.  Output planes span several 256-position tiles with a ragged tail.
"""
import itertools
import zlib

import numpy as np
import pytest
import torch

from conftest import assert_parity
from spatial_transformer_sampling_gb300 import workloads as wl
from test_gpu_sample_int import ITYPES, _int_tensor, check_int

pytestmark = pytest.mark.gpu

DTYPES = ["float32", "float16", "bfloat16"]
SHAPES = {
    4: ((2, 3, 4, 5, 3, 6), (5, 7, 6, 3)),          # 630 positions: 3 tiles, ragged
    5: ((2, 2, 3, 4, 3, 5, 2), (3, 4, 5, 3, 2)),     # 360
    6: ((1, 2, 3, 2, 4, 3, 2, 3), (2, 3, 4, 3, 2, 3)),   # 432
}
SWEEP = [(r, m, p, ac, dt)
         for r in (4, 5, 6) for m in ("linear", "nearest", "cubic")
         for p in ("zeros", "border", "reflection") for ac in (0, 1)
         for dt in (DTYPES if r == 4 else ["float32"])]


def exact(t):
    return wl.widened(t)


def _grid(g, n, out, r):
    grid = g.uniform(-1.4, 1.4, size=(n,) + out + (r,))
    flat = grid.reshape(-1, r)
    flat[:6] = np.array([-1.0, 1.0, 0.0, 7.3, -5.9, 2.0])[:, None]   # landmarks, far out
    return grid


@pytest.mark.parametrize("r,mode,pad,ac,dtype", SWEEP)
def test_grid_sample_rank_nd_sweep(gs_cuda, oracle_mod, r, mode, pad, ac, dtype):
    g = wl.rng(zlib.crc32(repr((r, mode, pad, ac, "nd")).encode()))
    xs, out = SHAPES[r]
    Xt = wl.as_dtype(g.normal(size=xs), dtype)
    Gt = wl.as_dtype(_grid(g, xs[0], out, r), dtype)
    Y = gs_cuda.gs_grid_sample(Xt.cuda(), Gt.cuda(), mode, pad, ac)
    assert tuple(Y.shape) == xs[:2] + out
    assert gs_cuda.gs_device_status() == 0
    ref = oracle_mod.grid_sample(exact(Xt), exact(Gt), mode, pad, ac)
    if mode == "nearest":
        np.testing.assert_array_equal(exact(Y), ref)
    else:
        assert_parity(Y, ref, dtype, f"r={r} {mode} {pad} ac={ac} {dtype}")


@pytest.mark.parametrize("r", [4, 5, 6])
@pytest.mark.parametrize("mode", ["linear", "nearest", "cubic"])
def test_rank_nd_static_entry_matches(gs_cuda, oracle_mod, r, mode):
    """gs_grid_sample_static and gs_grid_sample_ws take the same kernel at these ranks
    (the channel-last path is 2-D only): identical outputs."""
    g = wl.rng(31 + r)
    xs, out = SHAPES[r]
    Xt = wl.as_dtype(g.normal(size=xs), "float32").cuda()
    Gt = wl.as_dtype(_grid(g, xs[0], out, r), "float32").cuda()
    Y = gs_cuda.gs_grid_sample(Xt, Gt, mode, "reflection", 0)
    Ys = gs_cuda.gs_grid_sample_static(Xt, Gt, mode, "reflection", 0)
    Yw = gs_cuda.gs_grid_sample(Xt, Gt, mode, "reflection", 0, workspace="auto")
    assert torch.equal(Y, Ys) and torch.equal(Y, Yw)


@pytest.mark.parametrize("pad", ["zeros", "border", "reflection"])
@pytest.mark.parametrize("mode", ["linear", "nearest", "cubic"])
@pytest.mark.parametrize("ac", [0, 1])
def test_rank4_single_pixel_axes(gs_cuda, oracle_mod, pad, mode, ac):
    g = wl.rng(41)
    X = g.normal(size=(2, 2, 1, 5, 1, 4))
    grid = wl.as_dtype(g.uniform(-2, 2, size=(2, 3, 1, 4, 5, 4)), "float32")
    Y = gs_cuda.gs_grid_sample(wl.as_dtype(X, "float32").cuda(), grid.cuda(), mode, pad, ac)
    ref = oracle_mod.grid_sample(X.astype(np.float32).astype(np.float64), exact(grid), mode, pad, ac)
    assert_parity(Y, ref, "float32", "rank 4 with 1-pixel axes")


def test_rank_nd_empty_outputs(gs_cuda):
    X = torch.zeros((2, 3, 2, 2, 2, 2), device="cuda")
    assert gs_cuda.gs_grid_sample(X, torch.zeros((2, 3, 0, 2, 2, 4), device="cuda")).shape == \
        (2, 3, 3, 0, 2, 2)
    X = torch.zeros((0, 3, 2, 2, 2, 2, 2), device="cuda")
    assert gs_cuda.gs_grid_sample(X, torch.zeros((0, 1, 1, 1, 1, 1, 5), device="cuda")).shape == \
        (0, 3, 1, 1, 1, 1, 1)


def test_rank_beyond_six_is_rejected(gs_cuda):
    X = torch.zeros((1, 1) + (2,) * 7, device="cuda")
    grid = torch.zeros((1,) + (2,) * 7 + (7,), device="cuda")
    with pytest.raises(gs_cuda.GsError, match="GS_ERR_RANK"):
        gs_cuda.gs_grid_sample(X, grid)


@pytest.mark.parametrize("pad", ["zeros", "border", "reflection"])
def test_rank4_constant_and_separable_inputs(gs_cuda, pad):
    """Weights per axis sum to 1 (every mode), so a constant X stays constant wherever
    every tap is in range; with border padding everywhere."""
    g = wl.rng(51)
    X = torch.full((1, 2, 4, 3, 5, 4), 1.75, device="cuda")
    grid = wl.as_dtype(g.uniform(-3, 3, size=(1, 4, 3, 5, 6, 4)), "float32").cuda()
    for mode in ("linear", "cubic"):
        Y = gs_cuda.gs_grid_sample(X, grid, mode, "border", 1)
        torch.testing.assert_close(Y, torch.full_like(Y, 1.75), rtol=0, atol=4e-6)


@pytest.mark.parametrize("r,mode,pad,ac,dtype",
                         [(4, m, p, ac, dt) for m in ("linear", "nearest", "cubic")
                          for p in ("zeros", "border", "reflection") for ac in (0, 1)
                          for dt in ("uint8", "int16")])
def test_integer_x_rank4(gs_cuda, oracle_mod, r, mode, pad, ac, dtype):
    g = wl.rng(zlib.crc32(repr((r, mode, pad, ac, dtype, "nd-int")).encode()))
    xs = (2, 2, 3, 4, 3, 5)
    out = (3, 4, 5, 6)
    Xt, X64 = _int_tensor(g, xs, dtype)
    Gt = wl.as_dtype(g.uniform(-1.25, 1.25, size=(xs[0],) + out + (r,)), "float32")
    Y = gs_cuda.gs_grid_sample_int(Xt.cuda(), Gt.cuda(), mode, pad, ac)
    assert Y.dtype == Xt.dtype and tuple(Y.shape) == xs[:2] + out
    assert gs_cuda.gs_device_status() == 0
    check_int(oracle_mod, Y, X64, exact(Gt), mode, pad, ac, dtype)
