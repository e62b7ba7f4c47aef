"""GridSample, AffineGrid and the fused AffineGrid+GridSample on the GPU against
the oracle, element by element on seeded inputs.

Sizes span several 256-position tiles with a ragged tail.  Bars: fp32
|y - ref| <= 1e-6 + 1e-5|ref|; fp16/bf16 <= 1e-2 + 1e-2|ref|; nearest is
compared bit for bit (its outputs are copies of X or 0).  The full-size
workloads are checked on sampled outputs the oracle computes one by one,
through the same library call the bench times.
"""
import itertools
import zlib

import numpy as np
import pytest
import torch

from conftest import (assert_parity, fixture_array, fixture_names, load_fixture, page_close)
from spatial_transformer_sampling_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DTYPES = ["float32", "float16", "bfloat16"]


def dev(a, dtype):
    return wl.as_dtype(a, dtype).cuda()


def exact(t):
    return wl.widened(t)


# ------------------------------------------------------------- page examples

@pytest.mark.parametrize("name", fixture_names("gridsample__"))
def test_page_examples_grid_sample(gs_cuda, oracle_mod, name):
    fx = load_fixture(name)
    a = fx["attributes"]
    X = fixture_array(fx["inputs"]["X"])
    grid = fixture_array(fx["inputs"]["Grid"])
    mode, pad, ac = a.get("mode", "linear"), a.get("padding_mode", "zeros"), a.get("align_corners", 0)
    Y = gs_cuda.gs_grid_sample(dev(X, "float32"), dev(grid, "float32"), mode, pad, ac)
    ref = oracle_mod.grid_sample(X, grid, mode, pad, ac)
    assert_parity(Y, ref, "float32", fx["citation"])
    assert page_close(exact(Y), fixture_array(fx["outputs"]["Y"])).all(), fx["citation"]


@pytest.mark.parametrize("name", fixture_names("affinegrid__"))
def test_page_examples_affine_grid(gs_cuda, oracle_mod, name):
    fx = load_fixture(name)
    theta = fixture_array(fx["inputs"]["theta"])
    size = fixture_array(fx["inputs"]["size"])
    ac = fx["attributes"].get("align_corners", 0)
    G = gs_cuda.gs_affine_grid(dev(theta, "float32"), size, ac)
    assert_parity(G, oracle_mod.affine_grid(theta, size, ac), "float32", fx["citation"])
    assert page_close(exact(G), fixture_array(fx["outputs"]["grid"])).all(), fx["citation"]


# ------------------------------------------------------- small seeded sweeps

SHAPES = {1: ((2, 3, 37), (301,)), 2: ((2, 3, 19, 23), (29, 37)), 3: ((2, 2, 7, 9, 11), (5, 13, 17))}
SWEEP = list(itertools.product((1, 2, 3), ("linear", "nearest", "cubic"),
                               ("zeros", "border", "reflection"), (0, 1), DTYPES))


def _sweep_grid(g, n, out, r):
    grid = g.uniform(-1.4, 1.4, size=(n,) + out + (r,))
    flat = grid.reshape(-1, r)
    flat[:6] = np.array([-1.0, 1.0, 0.0, 7.3, -5.9, 2.0])[:, None]   # landmarks and far-out values
    return grid


@pytest.mark.parametrize("r,mode,pad,ac,dtype", SWEEP)
def test_grid_sample_sweep(gs_cuda, oracle_mod, r, mode, pad, ac, dtype):
    g = wl.rng(zlib.crc32(repr((r, mode, pad, ac)).encode()))
    xs, out = SHAPES[r]
    Xt = wl.as_dtype(g.normal(size=xs), dtype)
    Gt = wl.as_dtype(_sweep_grid(g, xs[0], out, r), dtype)
    Y = gs_cuda.gs_grid_sample(Xt.cuda(), Gt.cuda(), mode, pad, ac)
    ref = oracle_mod.grid_sample(exact(Xt), exact(Gt), mode, pad, ac)
    if mode == "nearest":
        np.testing.assert_array_equal(exact(Y), ref.astype(np.float64))
    else:
        assert_parity(Y, ref, dtype, f"r={r} {mode} {pad} ac={ac} {dtype}")


AFFINE_SWEEP = list(itertools.product((2, 3), ("linear", "nearest", "cubic"),
                                      ("zeros", "border", "reflection"), (0, 1), DTYPES))
AFFINE_SHAPES = {2: ((3, 3, 21, 17), (3, 3, 26, 31)), 3: ((2, 2, 9, 7, 11), (2, 2, 6, 10, 13))}


@pytest.mark.parametrize("r,mode,pad,ac,dtype", AFFINE_SWEEP)
def test_affine_sample_sweep(gs_cuda, oracle_mod, r, mode, pad, ac, dtype):
    g = wl.rng(zlib.crc32(repr((r, mode, pad, ac, 7)).encode()))
    xs, size = AFFINE_SHAPES[r]
    theta = wl.identity_theta(xs[0], r) + g.normal(0, 0.25, size=(xs[0], r, r + 1))
    theta[-1] *= 1.7   # one image zoomed out past the borders
    Tt = wl.as_dtype(theta, dtype)
    Xt = wl.as_dtype(g.normal(size=xs), dtype)
    Y = gs_cuda.gs_affine_sample(Tt.cuda(), size, Xt.cuda(), mode, pad, ac)
    ref = oracle_mod.affine_sample(exact(Tt), size, exact(Xt), mode, pad, ac)
    if mode == "nearest":
        assert_nearest_affine(oracle_mod, Y, ref, Tt, size, xs, ac)
    else:
        assert_parity(Y, ref, dtype, f"affine r={r} {mode} {pad} ac={ac} {dtype}")


def assert_nearest_affine(oracle_mod, Y, ref, Tt, size, xs, ac):
    """Nearest on an affine map: bit copies away from half-integer positions.

    Where the exact position is k + 1/2 but the map's coefficients are not
    dyadic (e.g. a 1/37 scale), neither the fp64 oracle nor the fixed-point
    kernel forms the tie exactly, and each rounds it by its own rounding
    error; within 1e-7 px of a tie only membership in X (or 0) is checked.
    """
    r = len(xs) - 2
    grid = oracle_mod.affine_grid(exact(Tt), size, ac)
    tie = np.zeros(grid.shape[:-1], dtype=bool)
    for d in range(r):
        n = xs[2 + d]
        gd = grid[..., r - 1 - d]
        x = (gd + 1) / 2 * (n - 1) if ac else ((gd + 1) * n - 1) / 2
        tie |= np.abs(x - np.floor(x) - 0.5) < 1e-7
    tie = np.broadcast_to(tie[:, None], ref.shape)
    got = exact(Y)
    np.testing.assert_array_equal(got[~tie], ref[~tie])
    return tie


@pytest.mark.parametrize("r,ac,dtype", list(itertools.product((2, 3), (0, 1), DTYPES)))
def test_affine_grid_random(gs_cuda, oracle_mod, r, ac, dtype):
    g = wl.rng(50 + r + 10 * ac)
    size = (3, 2, 17, 23) if r == 2 else (2, 2, 5, 9, 7)
    Tt = wl.as_dtype(g.normal(size=(size[0], r, r + 1)) * 2, dtype)
    G = gs_cuda.gs_affine_grid(Tt.cuda(), size, ac)
    assert_parity(G, oracle_mod.affine_grid(exact(Tt), size, ac), dtype, "affine_grid")


# ------------------------------------------------------------- closed forms

@pytest.mark.parametrize("r,mode,ac,dtype",
                         list(itertools.product((2, 3), ("linear", "nearest", "cubic"), (0, 1),
                                                DTYPES)))
def test_identity_theta_reproduces_X_bit_exactly(gs_cuda, r, mode, ac, dtype):
    g = wl.rng(61)
    xs = (3, 4, 33, 45) if r == 2 else (2, 3, 9, 17, 13)
    Xt = dev(g.normal(size=xs), dtype)
    Tt = dev(wl.identity_theta(xs[0], r), dtype)
    for pad in ("zeros", "border", "reflection"):
        Y = gs_cuda.gs_affine_sample(Tt, xs, Xt, mode, pad, ac)
        assert torch.equal(Y, Xt), (mode, pad, ac, dtype)


@pytest.mark.parametrize("dtype", ["float32", "float16"])
@pytest.mark.parametrize("ac", [0, 1])
@pytest.mark.parametrize("pad", ["zeros", "border", "reflection"])
def test_nearest_half_integer_ties_are_bit_exact(gs_cuda, oracle_mod, dtype, ac, pad):
    """Grid values whose unnormalised position is exactly k + 1/2 (ties to the even index)."""
    n = 8
    k = np.arange(-3, n + 2)
    x = k + 0.5
    gv = (2 * x + 1) / n - 1 if ac == 0 else 2 * x / (n - 1) - 1
    gv = gv.astype(np.float32).astype(np.float64)
    X = wl.rng(71).normal(size=(1, 2, n))
    Xt = wl.as_dtype(X, dtype)
    Gt = wl.as_dtype(gv.reshape(1, -1, 1), dtype)
    Y = gs_cuda.gs_grid_sample(Xt.cuda(), Gt.cuda(), "nearest", pad, ac)
    np.testing.assert_array_equal(exact(Y), oracle_mod.grid_sample(exact(Xt), exact(Gt), "nearest",
                                                                   pad, ac))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("mode", ["linear", "cubic"])
def test_grid_sample_affine_grid_composition(gs_cuda, oracle_mod, dtype, mode):
    """gs_affine_grid feeds gs_grid_sample, the unfused composition: the grid is
    rounded to the I/O dtype in between (the unfused reading), so the sampling stage
    is compared with the oracle's GridSample on that rounded grid, and the grid with
    the oracle's AffineGrid."""
    g = wl.rng(81)
    X = g.normal(size=(2, 3, 20, 24))
    theta = wl.identity_theta(2, 2) + g.normal(0, 0.2, size=(2, 2, 3))
    size = (2, 3, 18, 22)
    Tt, Xt = wl.as_dtype(theta, dtype), wl.as_dtype(X, dtype)
    G = gs_cuda.gs_affine_grid(Tt.cuda(), size, 1)
    G_ref = oracle_mod.affine_grid(exact(Tt), size, 1)
    assert_parity(G, G_ref, dtype, "grid")
    Y = gs_cuda.gs_grid_sample(Xt.cuda(), G, mode, "border", 1)
    ref = oracle_mod.grid_sample(exact(Xt), exact(G), mode, "border", 1)
    assert_parity(Y, ref, dtype, f"sampling the rounded grid ({mode}, {dtype})")


# ------------------------------------------------------------- edge cases

def test_empty_inputs_return_empty_outputs(gs_cuda):
    X = torch.zeros((0, 3, 5, 5), device="cuda")
    grid = torch.zeros((0, 4, 4, 2), device="cuda")
    assert gs_cuda.gs_grid_sample(X, grid).shape == (0, 3, 4, 4)
    X = torch.zeros((2, 0, 5, 5), device="cuda")
    grid = torch.zeros((2, 4, 4, 2), device="cuda")
    assert gs_cuda.gs_grid_sample(X, grid).shape == (2, 0, 4, 4)
    X = torch.zeros((2, 3, 5, 5), device="cuda")
    assert gs_cuda.gs_grid_sample(X, torch.zeros((2, 0, 4, 2), device="cuda")).shape == (2, 3, 0, 4)


@pytest.mark.parametrize("pad", ["zeros", "border", "reflection"])
@pytest.mark.parametrize("mode", ["linear", "nearest", "cubic"])
@pytest.mark.parametrize("ac", [0, 1])
def test_degenerate_single_pixel_axes(gs_cuda, oracle_mod, pad, mode, ac):
    g = wl.rng(91)
    X = g.normal(size=(2, 3, 1, 6))
    grid = g.uniform(-2, 2, size=(2, 5, 7, 2))
    Y = gs_cuda.gs_grid_sample(dev(X, "float32"), dev(grid, "float32"), mode, pad, ac)
    assert_parity(Y, oracle_mod.grid_sample(X, wl.widened(wl.as_dtype(grid, "float32")), mode, pad,
                                            ac), "float32", "1-pixel axis")
    theta = wl.identity_theta(2, 2) + g.normal(0, 0.3, size=(2, 2, 3))
    size = (2, 3, 1, 9)   # single-row output: the base position is 0
    Y = gs_cuda.gs_affine_sample(dev(theta, "float32"), size, dev(X, "float32"), mode, pad, ac)
    ref = oracle_mod.affine_sample(wl.widened(wl.as_dtype(theta, "float32")), size, X, mode, pad, ac)
    assert_parity(Y, ref, "float32", "1-pixel output axis")


@pytest.mark.parametrize("pad", ["zeros", "border", "reflection"])
@pytest.mark.parametrize("mode", ["linear", "cubic"])
def test_far_out_and_non_finite_grid_values(gs_cuda, oracle_mod, pad, mode):
    """Far-out finite values match the oracle; NaN, inf and 1e30 stay in bounds and give
    finite output (the operator leaves their result open)."""
    # values where the fp64 oracle is itself exact (|g| well below 2^50 for these n)
    vals = np.array([1e10, -1e10, 3.0e7, -3.0e7, 4097.25, -65536.5, 7.75, -9.1])
    X = wl.rng(101).normal(size=(1, 2, 11, 13))
    grid = np.stack(np.meshgrid(vals, vals[::-1]), -1)[None]
    Gt = wl.as_dtype(grid, "float32")
    Y = gs_cuda.gs_grid_sample(dev(X, "float32"), Gt.cuda(), mode, pad, 0)
    assert_parity(Y, oracle_mod.grid_sample(X, exact(Gt), mode, pad, 0), "float32", "far out")
    bad = torch.tensor([[[[float("nan"), 0.0], [float("inf"), -float("inf")]],
                         [[1e30, -1e30], [3e38, 0.5]]]], device="cuda")
    Y = gs_cuda.gs_grid_sample(dev(X, "float32"), bad, mode, pad, 0)
    assert torch.isfinite(Y).all()
    theta = torch.tensor([[[float("nan"), 0, 0], [0, 1e30, 0]]], device="cuda")
    Y = gs_cuda.gs_affine_sample(theta, (1, 2, 5, 6), dev(X, "float32"), mode, pad, 0)
    assert torch.isfinite(Y).all()


def test_maximum_extent(gs_cuda, oracle_mod):
    n = 1 << 20
    g = wl.rng(111)
    Xt = wl.as_dtype(g.normal(size=(1, 2, n)), "float32")
    grid = g.uniform(-1.1, 1.1, size=(1, 4099, 1))
    for mode, pad in (("linear", "zeros"), ("cubic", "reflection"), ("nearest", "border")):
        Gt = wl.as_dtype(grid, "float32")
        Y = gs_cuda.gs_grid_sample(Xt.cuda(), Gt.cuda(), mode, pad, 1)
        ref = oracle_mod.grid_sample(exact(Xt), exact(Gt), mode, pad, 1)
        if mode == "nearest":
            np.testing.assert_array_equal(exact(Y), ref)
        else:
            # at n = 2^20 one fp32 grid ulp is ~0.06 px; compare against the
            # oracle on the same rounded grid, which is what both sides see
            assert_parity(Y, ref, "float32", f"n=2^20 {mode}")


# --------------------------------------------------- full-size workloads

def _sample_idx(total, k=20000, seed=0):
    g = wl.rng(seed)
    idx = np.unique(np.concatenate([g.integers(0, total, k), [0, total - 1]]))
    return idx


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_full_size_stn2d(gs_cuda, oracle_mod, dtype):
    w = wl.WORKLOADS["stn2d"]
    inp = wl.make_affine_sample_inputs(w)
    Tt, Xt = wl.as_dtype(inp["theta"], dtype), wl.as_dtype(inp["X"], dtype)
    Xd = Xt.cuda()
    Y = gs_cuda.gs_affine_sample(Tt.cuda(), inp["size"], Xd, w.mode, w.padding_mode,
                                 w.align_corners)
    torch.cuda.synchronize()
    idx = _sample_idx(Y.numel(), seed=1)
    ref = oracle_mod.affine_sample_at(exact(Tt), inp["size"], exact(Xt), idx, w.mode,
                                      w.padding_mode, w.align_corners)
    assert_parity(Y.reshape(-1)[torch.from_numpy(idx).cuda()], ref, dtype, "stn2d sampled")
    # at any size: linear + border output lies within each slab's range of X
    lo = Xd.float().amin(dim=(2, 3), keepdim=True)
    hi = Xd.float().amax(dim=(2, 3), keepdim=True)
    Yf = Y.float()
    slack = 1e-6 if dtype == "float32" else 2e-2
    assert bool(((Yf >= lo - slack) & (Yf <= hi + slack)).all())


@pytest.mark.parametrize("dtype", ["float32", "float16"])
@pytest.mark.parametrize("mode", ["cubic", "nearest"])
def test_full_size_gs2d_cubic_and_nearest(gs_cuda, oracle_mod, dtype, mode):
    w = wl.WORKLOADS["gs2d_cubic"]
    inp = wl.make_grid_sample_inputs(w)
    Xt, Gt = wl.as_dtype(inp["X"], dtype), wl.as_dtype(inp["grid"], dtype)
    Y = gs_cuda.gs_grid_sample(Xt.cuda(), Gt.cuda(), mode, w.padding_mode, w.align_corners,
                               w.cubic_coeff_a)
    torch.cuda.synchronize()
    idx = _sample_idx(Y.numel(), seed=2)
    ref = oracle_mod.grid_sample_at(exact(Xt), exact(Gt), idx, mode, w.padding_mode,
                                    w.align_corners, w.cubic_coeff_a)
    got = Y.reshape(-1)[torch.from_numpy(idx).cuda()]
    if mode == "nearest":
        np.testing.assert_array_equal(exact(got), ref)
    else:
        assert_parity(got, ref, dtype, f"gs2d {mode} sampled")


def test_full_size_stn3d(gs_cuda, oracle_mod):
    w = wl.WORKLOADS["stn3d"]
    inp = wl.make_affine_sample_inputs(w)
    Tt, Xt = wl.as_dtype(inp["theta"], "float32"), wl.as_dtype(inp["X"], "float32")
    Y = gs_cuda.gs_affine_sample(Tt.cuda(), inp["size"], Xt.cuda(), w.mode, w.padding_mode,
                                 w.align_corners)
    torch.cuda.synchronize()
    idx = _sample_idx(Y.numel(), seed=3)
    ref = oracle_mod.affine_sample_at(exact(Tt), inp["size"], exact(Xt), idx, w.mode,
                                      w.padding_mode, w.align_corners)
    assert_parity(Y.reshape(-1)[torch.from_numpy(idx).cuda()], ref, "float32", "stn3d sampled")


def test_full_size_gs2d_small(gs_cuda, oracle_mod):
    w = wl.WORKLOADS["gs2d_small"]
    inp = wl.make_grid_sample_inputs(w)
    Xt, Gt = wl.as_dtype(inp["X"], "float32"), wl.as_dtype(inp["grid"], "float32")
    Y = gs_cuda.gs_grid_sample(Xt.cuda(), Gt.cuda(), w.mode, w.padding_mode, w.align_corners)
    assert_parity(Y, oracle_mod.grid_sample(exact(Xt), exact(Gt), w.mode, w.padding_mode,
                                            w.align_corners), "float32", "gs2d_small")


# ------------------------------------------------ fused 2-D footprint cases

def _footprint_thetas(n):
    """identity-ish, pushed off the bottom, pushed off the top and rotated, zoomed out."""
    base = [[[1.02, 0.03, 0.01], [-0.02, 0.98, 0.02]],
            [[1.0, 0.05, 0.1], [0.06, 1.0, 0.6]],
            [[0.95, -0.2, -0.05], [0.25, 1.05, -0.7]],
            [[2.5, 0.0, 0.0], [0.0, 2.5, 0.0]]]
    return np.array([base[i % 4] for i in range(n)])


@pytest.mark.parametrize("mode", ["linear", "nearest", "cubic"])
@pytest.mark.parametrize("pad", ["zeros", "border", "reflection"])
@pytest.mark.parametrize("ac", [0, 1])
@pytest.mark.parametrize("dtype", DTYPES)
def test_affine_footprint_cases(gs_cuda, oracle_mod, mode, pad, ac, dtype):
    """Bands pushed off either edge, rotated, zoomed out; a ragged tile tail."""
    g = wl.rng(zlib.crc32(repr((mode, pad, ac, dtype, "footprint")).encode()))
    xs = (4, 5, 40, 32)            # 5 channels: not a multiple of the ring depth
    size = (4, 5, 37, 48)          # 1776 positions: a ragged last tile
    Tt = wl.as_dtype(_footprint_thetas(4), dtype)
    Xt = wl.as_dtype(g.normal(size=xs), dtype)
    Y = gs_cuda.gs_affine_sample(Tt.cuda(), size, Xt.cuda(), mode, pad, ac)
    ref = oracle_mod.affine_sample(exact(Tt), size, exact(Xt), mode, pad, ac)
    if mode == "nearest":
        tie = assert_nearest_affine(oracle_mod, Y, ref, Tt, size, xs, ac)
        assert tie.any()   # the zoomed image puts a whole row on exact ties
    else:
        assert_parity(Y, ref, dtype, f"footprint {mode} {pad} ac={ac} {dtype}")


@pytest.mark.parametrize("pad", ["zeros", "border", "reflection"])
@pytest.mark.parametrize("mode", ["linear", "nearest", "cubic"])
def test_affine_blocks_that_gather_from_global(gs_cuda, oracle_mod, pad, mode):
    """Blocks whose input rows overflow the shared-memory ring (a 12x zoom-out
    of a 300 x 256 image) and a map whose positions need fp64 (a translation
    of millions of pixels) both gather from global memory."""
    g = wl.rng(zlib.crc32(repr((pad, mode, "band-gather")).encode()))
    xs = (2, 2, 300, 256)
    size = (2, 2, 40, 64)
    theta = np.array([[[12.0, 0.5, 0.0], [0.3, 11.0, 0.1]],
                      [[1.0, 0.0, 3.0e6], [0.0, 1.0, -2.0e6]]])
    Tt, Xt = wl.as_dtype(theta, "float32"), wl.as_dtype(g.normal(size=xs), "float32")
    Y = gs_cuda.gs_affine_sample(Tt.cuda(), size, Xt.cuda(), mode, pad, 0)
    assert gs_cuda.gs_device_status() == 0
    ref = oracle_mod.affine_sample(exact(Tt), size, exact(Xt), mode, pad, 0)
    if mode == "nearest":
        assert_nearest_affine(oracle_mod, Y, ref, Tt, size, xs, 0)
    else:
        assert_parity(Y, ref, "float32", f"gather {mode} {pad}")


@pytest.mark.parametrize("mode", ["linear", "cubic"])
def test_affine_tall_input_zoomed_and_transposed(gs_cuda, oracle_mod, mode):
    g = wl.rng(17)
    xs = (2, 3, 420, 32)
    size = (2, 3, 30, 40)
    theta = np.array([[[1.5, 0.0, 0.0], [0.0, 1.5, 0.0]], [[0.3, 1.2, 0.1], [1.3, 0.2, -0.1]]])
    Tt, Xt = wl.as_dtype(theta, "float32"), wl.as_dtype(g.normal(size=xs), "float32")
    for pad in ("zeros", "border", "reflection"):
        Y = gs_cuda.gs_affine_sample(Tt.cuda(), size, Xt.cuda(), mode, pad, 0)
        assert_parity(Y, oracle_mod.affine_sample(exact(Tt), size, exact(Xt), mode, pad, 0),
                      "float32", f"tall {mode} {pad}")
        assert gs_cuda.gs_device_status() == 0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("mode", ["linear", "nearest"])
def test_output_pairs_match_single_outputs(gs_cuda, oracle_mod, dtype, mode):
    """Even output widths with Y aligned to two elements take adjacent output
    pairs per thread (packed FMA, one store per pair); a Y one element off that
    alignment takes one output at a time.  Same bits either way."""
    w = wl.WORKLOADS["stn2d"]
    inp = wl.make_affine_sample_inputs(w, x_shape=(6, 5, 128, 128), out_spatial=(50, 128))
    Tt, Xt = wl.as_dtype(inp["theta"], dtype).cuda(), wl.as_dtype(inp["X"], dtype).cuda()
    size = (6, 5, 50, 128)
    Y1 = gs_cuda.gs_affine_sample(Tt, size, Xt, mode, "border", 1)
    buf = torch.empty(Y1.numel() + 1, dtype=Y1.dtype, device="cuda")
    Y2 = buf[1:].view(size)
    gs_cuda.gs_affine_sample(Tt, size, Xt, mode, "border", 1, out=Y2)
    assert torch.equal(Y1, Y2)
    ref = oracle_mod.affine_sample(exact(Tt), size, exact(Xt), mode, "border", 1)
    if mode == "nearest":
        assert_nearest_affine(oracle_mod, Y1, ref, Tt.cpu(), size, (6, 5, 128, 128), 1)
    else:
        assert_parity(Y1, ref, dtype, f"pairs {dtype}")


def test_results_do_not_depend_on_input_alignment(gs_cuda):
    """An X view offset by one element gives bit-identical results."""
    w = wl.WORKLOADS["stn2d"]
    inp = wl.make_affine_sample_inputs(w, x_shape=(8, 6, 128, 128))
    for dtype in ("float32", "bfloat16"):
        Tt, Xt = dev(inp["theta"], dtype), dev(inp["X"], dtype)
        base = torch.empty(Xt.numel() + 8, dtype=Xt.dtype, device="cuda")
        Xm = base[1:1 + Xt.numel()].view_as(Xt)
        Xm.copy_(Xt)
        size = (8, 6, 128, 128)
        Yb = gs_cuda.gs_affine_sample(Tt, size, Xt, "linear", "border", 1)
        Yg = gs_cuda.gs_affine_sample(Tt, size, Xm, "linear", "border", 1)
        assert torch.equal(Yb, Yg), dtype


# ------------------------------------------------ fused 3-D footprint cases

def _footprint_thetas_3d(n):
    base = [[[1.02, 0.03, -0.05, 0.01], [-0.04, 0.98, 0.06, 0.02], [0.05, -0.03, 1.01, -0.03]],
            [[1.0, 0.05, 0.0, 0.1], [0.06, 1.0, 0.0, 0.6], [0.0, 0.1, 1.0, -0.7]],
            [[0.95, -0.2, 0.1, -0.05], [0.25, 1.05, -0.1, -0.3], [-0.1, 0.15, 0.9, 0.2]],
            [[2.5, 0.0, 0.0, 0.0], [0.0, 2.5, 0.0, 0.0], [0.0, 0.0, 2.5, 0.0]]]
    return np.array([base[i % 4] for i in range(n)])


@pytest.mark.parametrize("mode", ["linear", "nearest"])
@pytest.mark.parametrize("pad", ["zeros", "border", "reflection"])
@pytest.mark.parametrize("ac", [0, 1])
@pytest.mark.parametrize("dtype", DTYPES)
def test_affine3d_footprint_cases(gs_cuda, oracle_mod, mode, pad, ac, dtype):
    """Rows of 16-byte multiples: several tiles, ragged in depth and rows."""
    g = wl.rng(zlib.crc32(repr((mode, pad, ac, dtype, "footprint3")).encode()))
    xs = (4, 3, 12, 10, 16)
    size = (4, 3, 20, 30, 24)
    Tt = wl.as_dtype(_footprint_thetas_3d(4), dtype)
    Xt = wl.as_dtype(g.normal(size=xs), dtype)
    Y = gs_cuda.gs_affine_sample(Tt.cuda(), size, Xt.cuda(), mode, pad, ac)
    assert gs_cuda.gs_device_status() == 0
    ref = oracle_mod.affine_sample(exact(Tt), size, exact(Xt), mode, pad, ac)
    if mode == "nearest":
        assert_nearest_affine(oracle_mod, Y, ref, Tt, size, xs, ac)
    else:
        assert_parity(Y, ref, dtype, f"3d footprint {mode} {pad} ac={ac} {dtype}")


@pytest.mark.parametrize("pad", ["zeros", "border", "reflection"])
def test_affine3d_box_too_large_gathers_instead(gs_cuda, oracle_mod, pad):
    g = wl.rng(23)
    xs = (1, 2, 40, 40, 32)            # a zoomed-out tile needs the whole 205 KB volume
    size = (1, 2, 10, 12, 16)
    theta = np.array([[[1.6, 0.0, 0.0, 0.0], [0.0, 1.6, 0.0, 0.0], [0.0, 0.0, 1.6, 0.0]]])
    Tt, Xt = wl.as_dtype(theta, "float32"), wl.as_dtype(g.normal(size=xs), "float32")
    Y = gs_cuda.gs_affine_sample(Tt.cuda(), size, Xt.cuda(), "linear", pad, 1)
    assert gs_cuda.gs_device_status() == 0
    assert_parity(Y, oracle_mod.affine_sample(exact(Tt), size, exact(Xt), "linear", pad, 1),
                  "float32", f"3d gather fallback {pad}")


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_affine3d_batch_matches_per_image_calls(gs_cuda, oracle_mod, dtype):
    """More 8 x 8 x 16 output tiles than the persistent grid (two blocks per
    SM) holds, with a partial last round: blocks take several tiles of
    different images in turn.  The batched call must give the bits of one call
    per image (fewer tiles than blocks, one tile each) and agree with the
    oracle on sampled outputs."""
    grid = 2 * torch.cuda.get_device_properties(0).multi_processor_count
    tiles_per_image = 4 * 4 * 4                      # output (32, 32, 64)
    n = next(k for k in range(2, 200)
             if k * tiles_per_image > grid and 0 < (k * tiles_per_image) % grid <= grid // 3)
    C = 7
    g = wl.rng(29)
    xs = (n, C, 32, 32, 64)
    size = (n, C, 32, 32, 64)
    theta = np.tile(np.eye(3, 4), (n, 1, 1)) + g.normal(0.0, 0.05, size=(n, 3, 4))
    Tt, Xt = wl.as_dtype(theta, dtype), wl.as_dtype(g.normal(size=xs), dtype)
    Td, Xd = Tt.cuda(), Xt.cuda()
    Y = gs_cuda.gs_affine_sample(Td, size, Xd, "linear", "zeros", 0)
    assert gs_cuda.gs_device_status() == 0
    for i in range(n):
        Yi = gs_cuda.gs_affine_sample(Td[i:i + 1].contiguous(), (1,) + size[1:],
                                      Xd[i:i + 1].contiguous(), "linear", "zeros", 0)
        assert torch.equal(Y[i], Yi[0]), f"image {i} differs from its own call"
    idx = _sample_idx(Y.numel(), k=5000, seed=4)
    ref = oracle_mod.affine_sample_at(exact(Tt), size, exact(Xt), idx, "linear", "zeros", 0)
    assert_parity(Y.reshape(-1)[torch.from_numpy(idx).cuda()], ref, dtype,
                  f"3d batch {dtype}")
