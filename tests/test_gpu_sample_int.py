"""GridSample with integer X (uint8, int8, uint16, int16) on the GPU against the
oracle.  The oracle interpolates the exact integer values in fp64; the cast at the
end (truncation toward zero, saturated at the type's range) is compared exactly
wherever the fp64 value is farther from an integer than the kernel's fp32
rounding can move it, and within one unit (the two integers around it) elsewhere.
Nearest-mode outputs are copies and must be bit-exact everywhere."""
import itertools
import zlib

import numpy as np
import pytest
import torch

from spatial_transformer_sampling_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ITYPES = {"uint8": torch.uint8, "int8": torch.int8, "int16": torch.int16}
if hasattr(torch, "uint16"):
    ITYPES["uint16"] = torch.uint16


def _int_tensor(g, shape, dtype):
    lo, hi = {"uint8": (0, 255), "int8": (-128, 127), "uint16": (0, 65535),
              "int16": (-32768, 32767)}[dtype]
    a = g.integers(lo, hi + 1, size=shape, dtype=np.int64)
    if dtype == "uint16":   # build through int32: torch has few uint16 conversions
        t = torch.from_numpy(a.astype(np.int32)).to(torch.uint16)
    else:
        t = torch.from_numpy(a).to(ITYPES[dtype])
    return t, a.astype(np.float64)


def _as_int64(t):
    return t.to(torch.int32).to(torch.int64).numpy() if t.dtype == getattr(torch, "uint16", None) \
        else t.to(torch.int64).numpy()


def check_int(oracle_mod, Y, X64, grid64, mode, pad, ac, dtype, r, coverage=True):
    v = oracle_mod.grid_sample(X64, grid64, mode, pad, ac)
    exp = oracle_mod.cast_to_integer(v, dtype)
    got = _as_int64(Y.cpu())
    if mode == "nearest":
        np.testing.assert_array_equal(got, exp)
        return
    # fp32 error bound: one rounding per tap and per axis combine (plus the weight
    # products), each at most one ulp of |sum w X| <= max|X| * sum|w|
    taps = (2 if mode == "linear" else 4) ** r
    wsum = 1.0 if mode == "linear" else 1.6 ** r
    band = (taps + r) * 2.0 ** -23 * np.abs(X64).max() * wsum + 1e-6
    lo, hi = oracle_mod.INT_RANGES[dtype]
    near = np.abs(v - np.round(v)) <= band
    clear = ~near | (v <= lo - band) | (v >= hi + band)   # clearly saturated
    np.testing.assert_array_equal(got[clear], exp[clear])
    lo_exp = oracle_mod.cast_to_integer(v - band, dtype)
    hi_exp = oracle_mod.cast_to_integer(v + band, dtype)
    assert ((got >= np.minimum(lo_exp, hi_exp)) & (got <= np.maximum(lo_exp, hi_exp))).all()
    if coverage and band < 0.05:
        assert clear.mean() > 0.5   # the exact comparison covers most outputs
    return band


SWEEP = [(r, m, p, ac, dt, gdt) for r in (1, 2, 3) for m in ("linear", "nearest", "cubic")
         for p in ("zeros", "border", "reflection") for ac in (0, 1) for dt in ITYPES
         for gdt in ("float32", "float16", "bfloat16")
         if (r == 2 or (p == "zeros" and ac == 0)) and (gdt == "float32" or (m == "linear" and p == "border"))]


@pytest.mark.parametrize("r,mode,pad,ac,dtype,gdt", SWEEP)
def test_integer_x_sweep(gs_cuda, oracle_mod, r, mode, pad, ac, dtype, gdt):
    g = wl.rng(zlib.crc32(repr((r, mode, pad, ac, dtype, gdt, "int")).encode()))
    xs = {1: (2, 3, 29), 2: (2, 3, 13, 17), 3: (1, 2, 7, 8, 9)}[r]
    out = {1: (31,), 2: (11, 19), 3: (5, 6, 7)}[r]
    Xt, X64 = _int_tensor(g, xs, dtype)
    grid = g.uniform(-1.25, 1.25, size=(xs[0],) + out + (r,))
    Gt = wl.as_dtype(grid, gdt)
    Y = gs_cuda.gs_grid_sample_int(Xt.cuda(), Gt.cuda(), mode, pad, ac)
    assert Y.dtype == Xt.dtype and tuple(Y.shape) == xs[:2] + out
    assert gs_cuda.gs_device_status() == 0
    check_int(oracle_mod, Y, X64, wl.widened(Gt), mode, pad, ac, dtype, r)


@pytest.mark.parametrize("dtype", list(ITYPES))
def test_integer_x_cubic_overshoot_saturates(gs_cuda, oracle_mod, dtype):
    """A step between the type's extremes: cubic weights ring past both ends next to it."""
    lo, hi = oracle_mod.INT_RANGES[dtype]
    step = np.broadcast_to(np.arange(12) >= 6, (12, 12))
    X64 = np.where(step, hi, lo).astype(np.float64)[None, None]
    Xt = torch.from_numpy(X64.astype(np.int64))
    Xt = Xt.to(torch.int32).to(ITYPES[dtype]) if dtype == "uint16" else Xt.to(ITYPES[dtype])
    grid = wl.rng(4).uniform(-0.9, 0.9, size=(1, 20, 20, 2))
    Gt = wl.as_dtype(grid, "float32")
    Y = gs_cuda.gs_grid_sample_int(Xt.cuda(), Gt.cuda(), "cubic", "border", 0)
    v = oracle_mod.grid_sample(X64, wl.widened(Gt), "cubic", "border", 0)
    assert (v > hi).any() and (v < lo).any()
    # most outputs sit on the flat sides, exactly on lo or hi: no coverage bar here
    band = check_int(oracle_mod, Y, X64, wl.widened(Gt), "cubic", "border", 0, dtype, 2,
                     coverage=False)
    got = _as_int64(Y.cpu())
    assert (got[v > hi + band] == hi).all() and (got[v < lo - band] == lo).all()
    assert (v > hi + band).any() and (v < lo - band).any()


def test_integer_x_at_pixel_centres_is_a_copy(gs_cuda, oracle_mod):
    """Grid points on pixel centres (power-of-two extents, so the grid values are
    exact in fp32): every weight is 0 or 1 and the copy is exact."""
    g = wl.rng(9)
    Xt, X64 = _int_tensor(g, (1, 2, 4, 8), "uint8")
    ys, xs = np.meshgrid(np.arange(4), np.arange(8), indexing="ij")
    grid = np.stack([(2 * xs + 1) / 8 - 1, (2 * ys + 1) / 4 - 1], axis=-1)[None]
    Gt = wl.as_dtype(grid, "float32")
    for mode in ("linear", "cubic"):
        Y = gs_cuda.gs_grid_sample_int(Xt.cuda(), Gt.cuda(), mode, "zeros", 0)
        np.testing.assert_array_equal(_as_int64(Y.cpu()), X64.astype(np.int64))
