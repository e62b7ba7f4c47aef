"""The oracle against the values the operator pages print for their worked examples.

Fixtures under tests/golden/ transcribe each example (inputs, attributes,
expected output) with its citation.  Defaults for attributes an example does
not set come from the pages' Attributes sections: GridSample mode=linear,
padding_mode=zeros, align_corners=0; AffineGrid align_corners=0; DeformConv
stride 1, dilation 1, group 1, offset_group 1, B = 0, mask = 1.
"""
import numpy as np
import pytest

from conftest import fixture_array, fixture_names, load_fixture, page_close


@pytest.mark.parametrize("name", fixture_names("affinegrid__"))
def test_affine_grid_page_example(oracle_mod, name):
    fx = load_fixture(name)
    theta = fixture_array(fx["inputs"]["theta"])
    size = fixture_array(fx["inputs"]["size"])
    got = oracle_mod.affine_grid(theta, size, fx["attributes"].get("align_corners", 0))
    exp = fixture_array(fx["outputs"]["grid"])
    assert got.shape == exp.shape
    assert page_close(got, exp).all(), fx["citation"]


@pytest.mark.parametrize("name", fixture_names("gridsample__"))
def test_grid_sample_page_example(oracle_mod, name):
    fx = load_fixture(name)
    a = fx["attributes"]
    X = fixture_array(fx["inputs"]["X"])
    grid = fixture_array(fx["inputs"]["Grid"])
    got = oracle_mod.grid_sample(X, grid, a.get("mode", "linear"), a.get("padding_mode", "zeros"),
                                 a.get("align_corners", 0))
    exp = fixture_array(fx["outputs"]["Y"])
    assert got.shape == exp.shape
    assert page_close(got, exp).all(), (fx["citation"], got, exp)


def test_grid_sample_page_examples_cover_every_mode_and_padding():
    seen = set()
    for name in fixture_names("gridsample__"):
        a = load_fixture(name)["attributes"]
        seen.add((a.get("mode", "linear"), a.get("padding_mode", "zeros"), a.get("align_corners", 0)))
    modes = {s[0] for s in seen}
    pads = {s[1] for s in seen}
    assert modes == {"linear", "nearest", "cubic"} and pads == {"zeros", "border", "reflection"}


@pytest.mark.parametrize("name", fixture_names("deformconv__"))
def test_deform_conv_page_example(oracle_mod, name):
    fx = load_fixture(name)
    a = fx["attributes"]
    ins = fx["inputs"]
    got = oracle_mod.deform_conv(
        fixture_array(ins["X"]), fixture_array(ins["W"]), fixture_array(ins["offset"]),
        fixture_array(ins["B"]) if "B" in ins else None,
        fixture_array(ins["mask"]) if "mask" in ins else None,
        kernel_shape=a.get("kernel_shape"), pads=a.get("pads"), strides=a.get("strides"),
        dilations=a.get("dilations"), group=a.get("group", 1),
        offset_group=a.get("offset_group", 1))
    exp = fixture_array(fx["outputs"]["Y"])
    assert got.shape == exp.shape
    assert page_close(got, exp).all(), (fx["citation"], got, exp)


def _resize_source_coords(mode, n_in, n_out, length_resized, scale):
    """Resize's coordinate_transformation_mode maps (Resize - 18, Attributes)."""
    xr = np.arange(n_out, dtype=np.float64)
    if mode == "half_pixel":
        return (xr + 0.5) / scale - 0.5
    if mode == "align_corners":
        return xr * (n_in - 1) / (length_resized - 1)
    if mode == "asymmetric":
        return xr / scale
    raise ValueError(mode)


def resize_via_grid_sample_names():
    """Resize examples that are plain separable linear / cubic interpolation (no
    antialias, no crop, all axes given): those GridSample can reproduce."""
    out = []
    for n in fixture_names("resize__"):
        fx = load_fixture(n)
        a = fx["attributes"]
        if (a.get("mode") in ("linear", "cubic") and not a.get("antialias")
                and "axes" not in a and "roi" not in fx["inputs"]
                and a.get("coordinate_transformation_mode", "half_pixel")
                in ("half_pixel", "align_corners", "asymmetric")):
            out.append(n)
    return out


@pytest.mark.parametrize("name", resize_via_grid_sample_names())
def test_resize_examples_through_grid_sample(oracle_mod, name):
    """Resize (no antialias) is GridSample on a separable grid with edge-clamped taps.

    Each output coordinate's source position x (Resize's own map) is written
    as a GridSample grid value with align_corners=0, g = (2x+1)/n - 1, and
    sampled with padding_mode=border.  This pins the Keys cubic weights at
    a = -0.75 (and a = -0.5 through the exclude_outside examples, compared at
    points whose four taps all lie inside, where renormalisation is a no-op),
    the cubic tap order, and the per-tap border clamp at an unclamped
    coordinate.  With scales given, the resized length is input * scale,
    unfloored, as the align_corners examples require.
    """
    fx = load_fixture(name)
    a = fx["attributes"]
    X = fixture_array(fx["inputs"]["X"])
    exp = fixture_array(fx["outputs"]["Y"])
    H, W = X.shape[2:]
    Ho, Wo = exp.shape[2:]
    if "scales" in fx["inputs"]:
        sc = fixture_array(fx["inputs"]["scales"])
        sh, sw, lh, lw = sc[2], sc[3], H * sc[2], W * sc[3]
    else:
        sh, sw, lh, lw = Ho / H, Wo / W, Ho, Wo
    mode = a.get("coordinate_transformation_mode", "half_pixel")
    ys = _resize_source_coords(mode, H, Ho, lh, sh)
    xs = _resize_source_coords(mode, W, Wo, lw, sw)
    grid = np.zeros((1, Ho, Wo, 2))
    grid[0, :, :, 0] = ((2 * xs + 1) / W - 1)[None, :]
    grid[0, :, :, 1] = ((2 * ys + 1) / H - 1)[:, None]
    got = oracle_mod.grid_sample(X, grid, a["mode"], "border", 0, a.get("cubic_coeff_a", -0.75))
    ok = page_close(got, exp)
    if a.get("exclude_outside"):
        inner = ((ys >= 1) & (ys < H - 2))[:, None] & ((xs >= 1) & (xs < W - 2))[None, :]
        assert inner.any()
        ok = ok[0, 0][inner]
    assert ok.all(), (fx["citation"], got, exp)
