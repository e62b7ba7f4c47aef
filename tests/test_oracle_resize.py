"""The Resize oracle against what the Resize page and the mathematics fix.

Pins (all CPU):
  - the 37 worked examples of the Resize - 18 page, element by element
    (`_resize_upsample_sizes_nearest_not_smaller` states 8x8 and prints 7 rows:
    the stated extent is checked and the printed rows compared);
  - closed forms: sizes equal to the input give X back for every mode and
    coordinate map; nearest x2 with the asymmetric map is a plain repeat;
    antialiased linear at scale 1/2 (half_pixel) is the [1,3,3,1]/8 filter
    in the interior; linear align_corners resizing of a ramp gives the ramp;
  - invariants: a constant input stays constant for every mode, with and
    without antialias and exclude_outside; Resize of a separable (outer
    product) input is the outer product of the 1-D resizes;
  - tf_crop_and_resize with the whole roi [0, 1] and the input's sizes is the
    identity, and a crop outside the input is extrapolation_value.
"""
import itertools

import numpy as np
import pytest

from conftest import fixture_array, fixture_names, load_fixture, page_close


def fixture_call(oracle_mod, name):
    fx = load_fixture(name)
    ins = fx["inputs"]
    kw = dict(fx["attributes"])
    if "scales" in ins:
        kw["scales"] = fixture_array(ins["scales"])
    if "sizes" in ins:
        kw["sizes"] = fixture_array(ins["sizes"]).astype(np.int64)
    if "roi" in ins:
        kw["roi"] = fixture_array(ins["roi"])
    return fx, oracle_mod.resize(fixture_array(ins["X"]), **kw)


@pytest.mark.parametrize("name", fixture_names("resize__"))
def test_resize_page_example(oracle_mod, name):
    fx, got = fixture_call(oracle_mod, name)
    exp = fixture_array(fx["outputs"]["Y"])
    stated = fx.get("stated_spatial_shape")
    if stated:
        assert list(got.shape[-2:]) == stated, (fx["citation"], got.shape)
        got = got[..., :exp.shape[-2], :exp.shape[-1]]
    assert got.shape == exp.shape, (fx["citation"], got.shape, exp.shape)
    assert page_close(got, exp).all(), (fx["citation"], got, exp)


COORDS = ["half_pixel", "pytorch_half_pixel", "align_corners", "asymmetric"]


@pytest.mark.parametrize("mode", ["nearest", "linear", "cubic"])
@pytest.mark.parametrize("coord", COORDS)
def test_same_size_is_identity(oracle_mod, mode, coord):
    X = np.random.default_rng(1).normal(size=(2, 3, 5, 7))
    for antialias, excl in ((0, 0), (1, 0), (0, 1)):
        Y = oracle_mod.resize(X, sizes=[2, 3, 5, 7], mode=mode, coordinate_transformation_mode=coord,
                              antialias=antialias, exclude_outside=excl)
        np.testing.assert_allclose(Y, X, rtol=0, atol=1e-15)


def test_nearest_double_asymmetric_is_repeat(oracle_mod):
    X = np.random.default_rng(2).normal(size=(1, 2, 4, 3))
    Y = oracle_mod.resize(X, scales=[1, 1, 2, 2], mode="nearest",
                          coordinate_transformation_mode="asymmetric", nearest_mode="floor")
    np.testing.assert_array_equal(Y, X.repeat(2, axis=2).repeat(2, axis=3))


def test_antialias_linear_half_is_1331_filter(oracle_mod):
    x = np.random.default_rng(3).normal(size=16)
    Y = oracle_mod.resize(x[None, :], scales=[1, 0.5], mode="linear", antialias=1)[0]
    # output i sits at input 2i + 0.5: taps 2i-1 .. 2i+2 with weights 1, 3, 3, 1 (/8)
    for i in range(1, 7):
        ref = (x[2 * i - 1] + 3 * x[2 * i] + 3 * x[2 * i + 1] + x[2 * i + 2]) / 8
        assert abs(Y[i] - ref) < 1e-14
    # at the edges the missing taps read the edge value
    assert abs(Y[0] - (x[0] + 3 * x[0] + 3 * x[1] + x[2]) / 8) < 1e-14


def test_linear_align_corners_keeps_a_ramp(oracle_mod):
    x = 0.3 + 1.7 * np.arange(9, dtype=np.float64)
    Y = oracle_mod.resize(x, sizes=[25], mode="linear", coordinate_transformation_mode="align_corners")
    np.testing.assert_allclose(Y, 0.3 + 1.7 * np.linspace(0, 8, 25), rtol=0, atol=1e-13)


@pytest.mark.parametrize("mode,antialias,excl", [("nearest", 0, 0), ("linear", 0, 0), ("linear", 1, 0),
                                                  ("cubic", 0, 0), ("cubic", 1, 0), ("cubic", 0, 1),
                                                  ("cubic", 1, 1)])
def test_constant_stays_constant(oracle_mod, mode, antialias, excl):
    X = np.full((1, 1, 9, 13), 2.5)
    for scales in ([1, 1, 0.37, 0.61], [1, 1, 2.3, 1.7]):
        Y = oracle_mod.resize(X, scales=scales, mode=mode, antialias=antialias, exclude_outside=excl,
                              cubic_coeff_a=-0.5)
        np.testing.assert_allclose(Y, 2.5, rtol=0, atol=1e-13)


@pytest.mark.parametrize("mode,coord,antialias", list(itertools.product(
    ["nearest", "linear", "cubic"], COORDS, [0, 1])))
def test_separable_input_gives_separable_output(oracle_mod, mode, coord, antialias):
    g = np.random.default_rng(4)
    u, v = g.normal(size=6), g.normal(size=11)
    X = np.outer(u, v)[None, None]
    kw = dict(mode=mode, coordinate_transformation_mode=coord, antialias=antialias)
    Y = oracle_mod.resize(X, sizes=[1, 1, 4, 17], **kw)
    yu = oracle_mod.resize(u, sizes=[4], **kw)
    yv = oracle_mod.resize(v, sizes=[17], **kw)
    np.testing.assert_allclose(Y[0, 0], np.outer(yu, yv), rtol=1e-13, atol=1e-13)


def test_crop_and_resize_whole_roi_is_identity(oracle_mod):
    X = np.random.default_rng(5).normal(size=(1, 2, 6, 5))
    Y = oracle_mod.resize(X, sizes=[1, 2, 6, 5], roi=[0, 0, 0, 0, 1, 1, 1, 1], mode="linear",
                          coordinate_transformation_mode="tf_crop_and_resize")
    np.testing.assert_allclose(Y, X, rtol=0, atol=1e-14)
    Z = oracle_mod.resize(X, sizes=[1, 2, 3, 3], roi=[0, 0, 1.5, 0, 1, 1, 2.5, 1], mode="linear",
                          coordinate_transformation_mode="tf_crop_and_resize",
                          extrapolation_value=-7.0)
    assert (Z == -7.0).all()


def test_scale_output_extent_is_floored(oracle_mod):
    shape = oracle_mod.resize_shape((1, 1, 7, 10), scales=[1, 1, 0.5, 1.55])[0]
    assert shape == (1, 1, 3, 15)
