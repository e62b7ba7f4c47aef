"""GridSample through gs_grid_sample_ws (channel-last workspace path) on the GPU.

Against the oracle element by element on seeded inputs (same bars as the NCHW
path: fp32 |y - ref| <= 1e-6 + 1e-5|ref|, half types 1e-2 + 1e-2|ref|, nearest
bit for bit), and value for value against gs_grid_sample, whose taps, weights
and order of accumulation it shares.  Shapes span several 128-position blocks
with a ragged tail, several workspace chunks, channel counts that leave a
ragged last pass, and out-of-range taps under zeros padding.
"""
import itertools
import zlib

import numpy as np
import pytest
import torch

from conftest import assert_parity
from spatial_transformer_sampling_gb300 import GsError
from spatial_transformer_sampling_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DTYPES = ["float32", "float16", "bfloat16"]


def exact(t):
    return wl.widened(t)


def _grid(g, n, out, lo=-1.4, hi=1.4):
    grid = g.uniform(lo, hi, size=(n,) + out + (2,))
    flat = grid.reshape(-1, 2)
    flat[:6] = np.array([-1.0, 1.0, 0.0, 7.3, -5.9, 2.0])[:, None]   # landmarks and far-out values
    return grid


def _check(Y, ref, mode, dtype, what):
    if mode == "nearest":
        np.testing.assert_array_equal(exact(Y), ref.astype(np.float64), err_msg=what)
    else:
        assert_parity(Y, ref, dtype, what)


SWEEP = list(itertools.product(("linear", "nearest", "cubic"), ("zeros", "border", "reflection"),
                               (0, 1), DTYPES))


@pytest.mark.parametrize("mode,pad,ac,dtype", SWEEP)
def test_workspace_sweep(gs_cuda, oracle_mod, mode, pad, ac, dtype):
    g = wl.rng(zlib.crc32(repr(("ws", mode, pad, ac)).encode()))
    C = 24 if dtype == "float32" else 40          # one ragged pass of the 64-channel loop
    xs, out = (3, C, 19, 23), (29, 37)            # 1073 positions: 9 blocks, ragged tail
    Xt = wl.as_dtype(g.normal(size=xs), dtype)
    Gt = wl.as_dtype(_grid(g, xs[0], out), dtype)
    Xd, Gd = Xt.cuda(), Gt.cuda()
    Y = gs_cuda.gs_grid_sample_ws(Xd, Gd, "auto", mode, pad, ac)
    ref = oracle_mod.grid_sample(exact(Xt), exact(Gt), mode, pad, ac)
    _check(Y, ref, mode, dtype, f"ws {mode} {pad} ac={ac} {dtype}")
    Y0 = gs_cuda.gs_grid_sample(Xd, Gd, mode, pad, ac)
    assert torch.equal(Y, Y0)


# channel counts: one 16-byte vector per pixel, several passes, ragged passes
CHANNELS = {"float32": (4, 64, 68, 136), "float16": (8, 64, 72, 200), "bfloat16": (8, 128, 136)}


@pytest.mark.parametrize("dtype,C", [(d, c) for d in DTYPES for c in CHANNELS[d]])
@pytest.mark.parametrize("mode", ["linear", "cubic"])
def test_workspace_channel_counts(gs_cuda, oracle_mod, dtype, C, mode):
    g = wl.rng(zlib.crc32(repr(("wsC", dtype, C, mode)).encode()))
    xs, out = (2, C, 11, 9), (13, 21)
    Xt = wl.as_dtype(g.normal(size=xs), dtype)
    Gt = wl.as_dtype(_grid(g, xs[0], out, -1.2, 1.2), dtype)
    Y = gs_cuda.gs_grid_sample_ws(Xt.cuda(), Gt.cuda(), "auto", mode, "zeros", 0)
    ref = oracle_mod.grid_sample(exact(Xt), exact(Gt), mode, "zeros", 0)
    _check(Y, ref, mode, dtype, f"ws C={C} {mode} {dtype}")


@pytest.mark.parametrize("slots", [1, 2, 3, 4, 5, 6, 12])
def test_workspace_chunks(gs_cuda, oracle_mod, slots):
    """One slot: copy and sample alternate image by image.  k >= 2 slots: two
    buffers of k // 2 images, each launch sampling one chunk while copying the
    next (5 images: ragged last chunk)."""
    g = wl.rng(40 + slots)
    xs, out = (5, 32, 17, 15), (20, 19)
    Xt = wl.as_dtype(g.normal(size=xs), "float32")
    Gt = wl.as_dtype(_grid(g, xs[0], out), "float32")
    slot = xs[1] * (xs[2] * xs[3] + 1) * 4     # a zero pixel, then the image
    ws = torch.empty(slots * slot + 8, dtype=torch.uint8, device="cuda")
    Xd, Gd = Xt.cuda(), Gt.cuda()
    Y = gs_cuda.gs_grid_sample_ws(Xd, Gd, ws, "cubic", "reflection", 1)
    ref = oracle_mod.grid_sample(exact(Xt), exact(Gt), "cubic", "reflection", 1)
    assert_parity(Y, ref, "float32", f"{slots} slots")
    assert torch.equal(Y, gs_cuda.gs_grid_sample(Xd, Gd, "cubic", "reflection", 1))


@pytest.mark.parametrize("dtype", DTYPES)
def test_workspace_small_output_large_input(gs_cuda, oracle_mod, dtype):
    """Few output positions per image, many copy tiles: each sampling block
    also copies many tiles of the next chunk."""
    g = wl.rng(61)
    xs, out = (4, 16, 64, 70), (5, 7)
    Xt = wl.as_dtype(g.normal(size=xs), dtype)
    Gt = wl.as_dtype(_grid(g, xs[0], out), dtype)
    for ws in ("auto", torch.empty(2 * 16 * (64 * 70 + 1) * 4, dtype=torch.uint8, device="cuda")):
        Y = gs_cuda.gs_grid_sample_ws(Xt.cuda(), Gt.cuda(), ws, "linear", "zeros", 0)
        ref = oracle_mod.grid_sample(exact(Xt), exact(Gt), "linear", "zeros", 0)
        assert_parity(Y, ref, dtype, "small output, large input")


def test_workspace_too_small_or_ineligible_takes_the_gather(gs_cuda, oracle_mod):
    g = wl.rng(77)
    Xt = wl.as_dtype(g.normal(size=(2, 6, 9, 10)), "float32")     # 24 bytes per pixel: no vectors
    Gt = wl.as_dtype(_grid(g, 2, (7, 8)), "float32")
    ref = oracle_mod.grid_sample(exact(Xt), exact(Gt), "linear", "zeros", 0)
    assert gs_cuda.gs_grid_sample_workspace_size(Xt.shape, (7, 8), torch.float32) == 0
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    Y = gs_cuda.gs_grid_sample_ws(Xt.cuda(), Gt.cuda(), ws, "linear", "zeros", 0)
    assert_parity(Y, ref, "float32", "ineligible C")
    Xt = wl.as_dtype(g.normal(size=(2, 8, 9, 10)), "float32")
    ref = oracle_mod.grid_sample(exact(Xt), exact(Gt), "linear", "zeros", 0)
    small = torch.empty(8 * (9 * 10 + 1) * 4 - 16, dtype=torch.uint8, device="cuda")
    Y = gs_cuda.gs_grid_sample_ws(Xt.cuda(), Gt.cuda(), small, "linear", "zeros", 0)
    assert_parity(Y, ref, "float32", "workspace below one image")
    Y = gs_cuda.gs_grid_sample_ws(Xt.cuda(), Gt.cuda(), None, "linear", "zeros", 0)
    assert_parity(Y, ref, "float32", "no workspace")


def test_workspace_alignment_is_checked(gs_cuda):
    X = torch.zeros((1, 8, 4, 4), device="cuda")
    grid = torch.zeros((1, 3, 3, 2), device="cuda")
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(GsError, match="misaligned"):
        gs_cuda.gs_grid_sample_ws(X, grid, ws[4:], "linear", "zeros", 0)


def test_workspace_ranks_1_and_3_take_the_gather(gs_cuda, oracle_mod):
    g = wl.rng(78)
    for xs, out in (((2, 8, 37), (45,)), ((1, 8, 5, 6, 7), (4, 5, 6))):
        r = len(out)
        Xt = wl.as_dtype(g.normal(size=xs), "float32")
        Gt = wl.as_dtype(g.uniform(-1.2, 1.2, size=(xs[0],) + out + (r,)), "float32")
        Y = gs_cuda.gs_grid_sample_ws(Xt.cuda(), Gt.cuda(), "auto", "linear", "border", 0)
        ref = oracle_mod.grid_sample(exact(Xt), exact(Gt), "linear", "border", 0)
        assert_parity(Y, ref, "float32", f"rank {r} with workspace")


def test_workspace_empty_inputs(gs_cuda):
    X = torch.zeros((0, 8, 4, 4), device="cuda")
    grid = torch.zeros((0, 3, 3, 2), device="cuda")
    assert gs_cuda.gs_grid_sample_ws(X, grid, "auto").shape == (0, 8, 3, 3)
    X = torch.zeros((2, 8, 4, 4), device="cuda")
    grid = torch.zeros((2, 0, 3, 2), device="cuda")
    assert gs_cuda.gs_grid_sample_ws(X, grid, "auto").shape == (2, 8, 0, 3)


@pytest.mark.parametrize("dtype", ["float32", "float16"])
@pytest.mark.parametrize("mode", ["cubic", "nearest", "linear"])
def test_full_size_gs2d_cubic_with_workspace(gs_cuda, oracle_mod, dtype, mode):
    w = wl.WORKLOADS["gs2d_cubic"]
    inp = wl.make_grid_sample_inputs(w)
    Xt, Gt = wl.as_dtype(inp["X"], dtype), wl.as_dtype(inp["grid"], dtype)
    Xd, Gd = Xt.cuda(), Gt.cuda()
    Y = gs_cuda.gs_grid_sample_ws(Xd, Gd, "auto", mode, w.padding_mode, w.align_corners,
                                  w.cubic_coeff_a)
    torch.cuda.synchronize()
    g = wl.rng(3)
    idx = np.unique(np.concatenate([g.integers(0, Y.numel(), 20000), [0, Y.numel() - 1]]))
    ref = oracle_mod.grid_sample_at(exact(Xt), exact(Gt), idx, mode, w.padding_mode,
                                    w.align_corners, w.cubic_coeff_a)
    got = Y.reshape(-1)[torch.from_numpy(idx).cuda()]
    _check(got, ref, mode, dtype, f"gs2d {mode} {dtype} with workspace, sampled")
    # at any size: the same values as the NCHW gather
    assert torch.equal(Y, gs_cuda.gs_grid_sample(Xd, Gd, mode, w.padding_mode, w.align_corners,
                                                 w.cubic_coeff_a))


@pytest.mark.parametrize("dtype", DTYPES)
def test_workspace_unaligned_input(gs_cuda, oracle_mod, dtype):
    """X one element past a 16-byte boundary: the copy reads it element by element."""
    g = wl.rng(62)
    xs, out = (2, 16, 12, 16), (9, 11)      # H*W a multiple of every vector width
    Xt = wl.as_dtype(g.normal(size=xs), dtype)
    Gt = wl.as_dtype(_grid(g, xs[0], out), dtype)
    n = int(np.prod(xs))
    buf = torch.empty(n + 8, dtype=Xt.dtype, device="cuda")
    Xd = buf[1:n + 1].view(xs)
    Xd.copy_(Xt.cuda())
    assert Xd.data_ptr() % 16 != 0
    Y = gs_cuda.gs_grid_sample_ws(Xd, Gt.cuda(), "auto", "linear", "reflection", 1)
    ref = oracle_mod.grid_sample(exact(Xt), exact(Gt), "linear", "reflection", 1)
    assert_parity(Y, ref, dtype, "unaligned X")
    assert torch.equal(Y, gs_cuda.gs_grid_sample(Xd, Gt.cuda(), "linear", "reflection", 1))
