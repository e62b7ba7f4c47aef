"""Resize on the GPU against the oracle, element by element on seeded inputs:
the Resize page's worked examples, sweeps over modes, coordinate maps,
nearest modes, antialias, exclude_outside, tf_crop_and_resize, axes and
keep_aspect_ratio_policy for 1-, 2- and 3-D resizes (with identity axes
batched in front), edge cases, and the full-size workloads on sampled
outputs."""
import itertools
import zlib

import numpy as np
import pytest
import torch

from conftest import assert_parity, fixture_array, fixture_names, load_fixture, page_close
from spatial_transformer_sampling_gb300 import GsError
from spatial_transformer_sampling_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DTYPES = ["float32", "float16", "bfloat16"]


def _fixture_kwargs(fx):
    ins = fx["inputs"]
    kw = dict(fx["attributes"])
    if "scales" in ins:
        kw["scales"] = [float(v) for v in fixture_array(ins["scales"])]
    if "sizes" in ins:
        kw["sizes"] = [int(v) for v in fixture_array(ins["sizes"])]
    if "roi" in ins:
        kw["roi"] = [float(v) for v in fixture_array(ins["roi"])]
    return kw


@pytest.mark.parametrize("name", fixture_names("resize__"))
def test_page_examples_resize(gs_cuda, oracle_mod, name):
    fx = load_fixture(name)
    kw = _fixture_kwargs(fx)
    X = fixture_array(fx["inputs"]["X"])
    Y = gs_cuda.gs_resize(wl.as_dtype(X, "float32").cuda(), **kw)
    ref = oracle_mod.resize(X, **kw)
    assert_parity(Y, ref, "float32", fx["citation"])
    exp = fixture_array(fx["outputs"]["Y"])
    got = wl.widened(Y)[..., :exp.shape[-2], :exp.shape[-1]]
    assert got.shape == exp.shape
    assert page_close(got, exp).all(), fx["citation"]


def _f32(v):
    """The operator's scales and roi are float tensors: both sides get the float32 values."""
    return [float(np.float32(x)) for x in v]


def _run(gs_cuda, oracle_mod, X64, dtype, what, **kw):
    for k in ("scales", "roi"):
        if k in kw:
            kw[k] = _f32(kw[k])
    Xt = wl.as_dtype(X64, dtype)
    Y = gs_cuda.gs_resize(Xt.cuda(), **kw)
    assert gs_cuda.gs_device_status() == 0
    ref = oracle_mod.resize(wl.widened(Xt), **kw)
    if kw.get("mode", "nearest") == "nearest":
        np.testing.assert_array_equal(wl.widened(Y), ref, err_msg=what)
    else:
        assert_parity(Y, ref, dtype, what)


COORDS = ["half_pixel", "pytorch_half_pixel", "align_corners", "asymmetric"]
SWEEP = [(m, c, aa, ex, dt) for m in ("nearest", "linear", "cubic") for c in COORDS
         for aa in (0, 1) for ex in (0, 1) for dt in DTYPES
         if not (m == "nearest" and (aa or ex)) and (dt == "float32" or (aa == 0 and ex == 0))]


@pytest.mark.parametrize("mode,coord,aa,ex,dtype", SWEEP)
def test_resize_2d_sweep(gs_cuda, oracle_mod, mode, coord, aa, ex, dtype):
    g = wl.rng(zlib.crc32(repr((mode, coord, aa, ex, dtype)).encode()))
    X = g.normal(size=(2, 3, 19, 23))
    for scales in ([1, 1, 1.7, 2.3], [1, 1, 0.45, 0.6], [1, 1, 3.0, 0.31]):
        _run(gs_cuda, oracle_mod, X, dtype, f"2d {mode} {coord} aa={aa} ex={ex} {scales}",
             scales=scales, mode=mode, coordinate_transformation_mode=coord, antialias=aa,
             exclude_outside=ex, cubic_coeff_a=-0.5 if ex else -0.75)
    _run(gs_cuda, oracle_mod, X, dtype, f"2d sizes {mode} {coord}", sizes=[2, 3, 40, 7], mode=mode,
         coordinate_transformation_mode=coord, antialias=aa, exclude_outside=ex)


@pytest.mark.parametrize("nearest_mode", ["round_prefer_floor", "round_prefer_ceil", "floor", "ceil"])
@pytest.mark.parametrize("coord", COORDS)
def test_resize_nearest_modes_are_bit_exact(gs_cuda, oracle_mod, nearest_mode, coord):
    g = wl.rng(zlib.crc32(repr((nearest_mode, coord)).encode()))
    X = g.normal(size=(1, 4, 8, 12))
    # scales 2 and 0.5 put many source coordinates on exact halves
    for scales in ([1, 1, 2.0, 0.5], [1, 1, 0.5, 4.0], [1, 1, 1.5, 2.5]):
        _run(gs_cuda, oracle_mod, X, "float32", f"nearest {nearest_mode} {coord} {scales}",
             scales=scales, mode="nearest", coordinate_transformation_mode=coord,
             nearest_mode=nearest_mode)


@pytest.mark.parametrize("mode", ["nearest", "linear", "cubic"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_resize_1d_and_3d(gs_cuda, oracle_mod, mode, dtype):
    g = wl.rng(zlib.crc32(repr((mode, dtype, "13d")).encode()))
    X1 = g.normal(size=(3, 2, 37))
    _run(gs_cuda, oracle_mod, X1, dtype, f"1d {mode}", scales=[1, 1, 2.6], mode=mode)
    X3 = g.normal(size=(2, 2, 7, 9, 11))
    _run(gs_cuda, oracle_mod, X3, dtype, f"3d {mode}", sizes=[2, 2, 13, 5, 17], mode=mode)
    _run(gs_cuda, oracle_mod, X3, dtype, f"3d aa {mode}", scales=[1, 1, 0.5, 0.7, 0.4],
         mode=mode, antialias=1)


def test_resize_identity_axes_in_front_are_batched(gs_cuda, oracle_mod):
    g = wl.rng(77)
    X = g.normal(size=(2, 3, 4, 5, 6))
    # only the last two axes change; the three in front become slices
    _run(gs_cuda, oracle_mod, X, "float32", "batched", scales=[1, 1, 1, 1.5, 0.5], mode="linear")
    # the channel axis is resized with two identity axes behind it: three trailing axes
    _run(gs_cuda, oracle_mod, X[0], "float32", "channel axis", scales=[1, 2.0, 1, 1], mode="linear")
    # four resized axes are not supported
    with pytest.raises(GsError, match="unsupported"):
        gs_cuda.gs_resize(torch.zeros((2, 3, 4, 5), device="cuda"), scales=[2, 2, 2, 2],
                          mode="linear")


@pytest.mark.parametrize("dtype", DTYPES)
def test_resize_crop_and_extrapolation(gs_cuda, oracle_mod, dtype):
    g = wl.rng(5)
    X = g.normal(size=(2, 3, 10, 12))
    for roi in ([0, 0, 0.1, 0.2, 1, 1, 0.8, 0.9], [0, 0, -0.3, 0.5, 1, 1, 0.7, 1.6]):
        for mode in ("nearest", "linear", "cubic"):
            _run(gs_cuda, oracle_mod, X, dtype, f"crop {roi} {mode}", sizes=[2, 3, 7, 9], roi=roi,
                 mode=mode, coordinate_transformation_mode="tf_crop_and_resize",
                 extrapolation_value=-2.5)
    _run(gs_cuda, oracle_mod, X, dtype, "crop axes", sizes=[5, 6], axes=[3, 2],
         roi=[0.2, 0.1, 0.9, 0.6], mode="linear",
         coordinate_transformation_mode="tf_crop_and_resize")


STAGED = [(m, c, dt) for m in ("nearest", "linear", "cubic")
          for c in COORDS + ["tf_crop_and_resize"] for dt in DTYPES]


@pytest.mark.parametrize("mode,coord,dtype", STAGED)
def test_resize_staged_rows_match_the_row_kernel(gs_cuda, oracle_mod, mode, coord, dtype):
    """Inputs whose rows are whole 16-byte chunks take the staged row kernel
    (each slice's input rows bulk-copied into shared memory first); the same
    input one element off 16-byte alignment takes the plain row kernel.  Both
    match the oracle, and each other bit for bit."""
    g = wl.rng(zlib.crc32(repr((mode, coord, dtype, "staged")).encode()))
    X = g.normal(size=(3, 5, 21, 40))
    Xt = wl.as_dtype(X, dtype)
    cases = [dict(scales=_f32([1, 1, 1.7, 2.3])), dict(scales=_f32([1, 1, 0.45, 0.6])),
             dict(sizes=[3, 5, 63, 16]), dict(scales=_f32([1, 1, 1, 2.0]))]
    for case in cases:
        kw = dict(case, mode=mode, coordinate_transformation_mode=coord)
        if coord == "tf_crop_and_resize":
            kw.update(roi=_f32([0, 0, -0.2, 0.1, 1, 1, 0.9, 1.3]), extrapolation_value=-3.5)
        Y1 = gs_cuda.gs_resize(Xt.cuda(), **kw)
        buf = torch.empty(Xt.numel() + 1, dtype=Xt.dtype, device="cuda")
        Xu = buf[1:].view(Xt.shape)
        Xu.copy_(Xt.cuda())
        Y2 = gs_cuda.gs_resize(Xu, **kw)
        assert gs_cuda.gs_device_status() == 0
        what = f"staged {mode} {coord} {dtype} {case}"
        assert torch.equal(Y1, Y2), what
        ref = oracle_mod.resize(wl.widened(Xt), **kw)
        if mode == "nearest":
            np.testing.assert_array_equal(wl.widened(Y1), ref, err_msg=what)
        else:
            assert_parity(Y1, ref, dtype, what)


@pytest.mark.parametrize("policy", ["stretch", "not_larger", "not_smaller"])
def test_resize_keep_aspect_ratio(gs_cuda, oracle_mod, policy):
    X = wl.rng(6).normal(size=(1, 2, 9, 14))
    for sizes in ([20, 20], [4, 30], [9, 3]):
        _run(gs_cuda, oracle_mod, X, "float32", f"keep {policy} {sizes}", sizes=sizes, axes=[2, 3],
             mode="linear", keep_aspect_ratio_policy=policy)


def test_resize_edge_cases(gs_cuda, oracle_mod):
    g = wl.rng(8)
    # a single input pixel, a single output pixel, and an empty output
    _run(gs_cuda, oracle_mod, g.normal(size=(1, 2, 1, 1)), "float32", "1px in", sizes=[1, 2, 5, 4],
         mode="cubic")
    _run(gs_cuda, oracle_mod, g.normal(size=(1, 2, 6, 7)), "float32", "1px out", sizes=[1, 2, 1, 1],
         mode="linear", coordinate_transformation_mode="align_corners")
    _run(gs_cuda, oracle_mod, g.normal(size=(1, 2, 6, 7)), "float32", "1px out pytorch",
         sizes=[1, 2, 1, 1], mode="linear", coordinate_transformation_mode="pytorch_half_pixel")
    Y = gs_cuda.gs_resize(torch.zeros((1, 2, 6, 7), device="cuda"), sizes=[1, 2, 0, 3])
    assert Y.shape == (1, 2, 0, 3)
    # large output tiles with ragged tails along every axis
    _run(gs_cuda, oracle_mod, g.normal(size=(1, 1, 33, 70)), "float32", "ragged",
         sizes=[1, 1, 97, 301], mode="cubic")


@pytest.mark.parametrize("name,dtype", [("resize2d_up", "float32"), ("resize2d_up", "bfloat16"),
                                        ("resize2d_aa", "float32")])
def test_full_size_resize_workloads(gs_cuda, oracle_mod, name, dtype):
    """The bench workloads at full size; the oracle recomputes two whole slices."""
    w = wl.WORKLOADS[name]
    X = wl.make_resize_inputs(w)["X"]
    Xt = wl.as_dtype(X, dtype)
    kw = dict(scales=_f32(w.extra["scales"]), mode=w.mode, antialias=w.extra["antialias"])
    Y = gs_cuda.gs_resize(Xt.cuda(), **kw)
    assert tuple(Y.shape) == (w.x_shape[0], w.x_shape[1]) + tuple(w.out_spatial)
    for n, c in ((0, 0), (w.x_shape[0] - 1, w.x_shape[1] - 1)):
        ref = oracle_mod.resize(wl.widened(Xt[n:n + 1, c:c + 1]), **kw)
        assert_parity(Y[n:n + 1, c:c + 1], ref, dtype, f"{name} slice {n},{c}")


@pytest.mark.parametrize("dtype", ["float16", "bfloat16"])
def test_resize_pairs_match_single_outputs(gs_cuda, oracle_mod, dtype):
    """16-bit Resize with an even output width writes pairs of outputs; Y two
    bytes off a pair boundary takes the single-output staged loop instead.  The
    same bits either way (each pair lane rounds as fmaf), and the oracle's."""
    g = wl.rng(zlib.crc32(repr(("pairs", dtype)).encode()))
    Xt = wl.as_dtype(g.normal(size=(2, 7, 24, 32)), dtype)
    kw = dict(scales=_f32([1, 1, 2.0, 1.5]), mode="linear")
    Y1 = gs_cuda.gs_resize(Xt.cuda(), **kw)
    buf = torch.empty(Y1.numel() + 1, dtype=Y1.dtype, device="cuda")
    Y2 = buf[1:].view(Y1.shape)
    gs_cuda.gs_resize(Xt.cuda(), out=Y2, **kw)
    assert gs_cuda.gs_device_status() == 0
    assert torch.equal(Y1, Y2)
    assert_parity(Y1, oracle_mod.resize(wl.widened(Xt), **kw), dtype, f"pairs {dtype}")
