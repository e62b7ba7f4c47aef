"""The Python binding checks the shapes the C ABI does not receive (grid, theta,
offset, mask, B, out) before any device work, so these run on the CPU: a bad
shape raises ValueError naming the tensor, a good one gets as far as the
device check ("libgs takes CUDA tensors")."""
import pytest
import torch

import spatial_transformer_sampling_gb300 as gs


def z(*shape, dtype=torch.float32):
    return torch.zeros(shape, dtype=dtype)


def raises_shape(what, fn, *args, **kw):
    with pytest.raises(ValueError, match=what):
        fn(*args, **kw)


def reaches_device_check(fn, *args, **kw):
    with pytest.raises(ValueError, match="CUDA"):
        fn(*args, **kw)


SAMPLERS = [gs.gs_grid_sample, gs.gs_grid_sample_ws, gs.gs_grid_sample_static]


@pytest.mark.parametrize("fn", SAMPLERS)
def test_grid_sample_wrappers_check_grid_and_out(fn):
    X = z(2, 3, 8, 9)
    reaches_device_check(fn, X, z(2, 5, 6, 2))
    raises_shape("grid", fn, X, z(1, 5, 6, 2))           # smaller batch
    raises_shape("grid", fn, X, z(2, 5, 6, 3))           # wrong last extent
    raises_shape("grid", fn, X, z(2, 30, 2))             # fewer dimensions than X
    raises_shape("grid", fn, X, z(2, 5, 6, 7, 2))        # more dimensions than X
    raises_shape("out", fn, X, z(2, 5, 6, 2), out=z(2, 3, 5, 5))
    raises_shape("out", fn, X, z(2, 5, 6, 2), out=z(2, 2, 5, 6))
    reaches_device_check(fn, X, z(2, 5, 6, 2), out=z(2, 3, 5, 6))


def test_grid_sample_int_checks_grid_and_out():
    X = z(2, 3, 8, 9, dtype=torch.uint8)
    raises_shape("grid", gs.gs_grid_sample_int, X, z(3, 5, 6, 2))
    raises_shape("out", gs.gs_grid_sample_int, X, z(2, 5, 6, 2),
                 out=z(2, 3, 6, 5, dtype=torch.uint8))
    with pytest.raises(ValueError, match="contiguous CUDA"):
        gs.gs_grid_sample_int(X, z(2, 5, 6, 2))


def test_grid_sample_rejects_x_without_spatial_axes():
    raises_shape("X must be", gs.gs_grid_sample, z(2, 3), z(2, 2))


def test_affine_sample_checks_theta_size_and_out():
    X = z(2, 3, 8, 9)
    f = gs.gs_affine_sample
    reaches_device_check(f, z(2, 2, 3), (2, 3, 5, 6), X)
    raises_shape("theta", f, z(1, 2, 3), (2, 3, 5, 6), X)
    raises_shape("theta", f, z(2, 3, 4), (2, 3, 5, 6), X)
    raises_shape("size", f, z(2, 2, 3), (2, 4, 5, 6), X)
    raises_shape("size", f, z(2, 2, 3), (2, 3, 5), X)
    raises_shape("out", f, z(2, 2, 3), (2, 3, 5, 6), X, out=z(2, 3, 6, 5))


def test_affine_grid_checks_theta_and_out():
    f = gs.gs_affine_grid
    reaches_device_check(f, z(2, 3, 4), (2, 1, 4, 5, 6))
    raises_shape("theta", f, z(2, 2, 3), (2, 1, 4, 5, 6))
    raises_shape("theta", f, z(3, 2, 3), (2, 1, 5, 6))
    raises_shape("out", f, z(2, 2, 3), (2, 1, 5, 6), out=z(2, 6, 5, 2))


def test_deform_conv_checks_every_tensor_shape():
    f = gs.gs_deform_conv
    X, W = z(2, 4, 8, 8), z(6, 4, 3, 3)
    off, mask, B = z(2, 18, 8, 8), z(2, 9, 8, 8), z(6)
    kw = dict(pads=(1, 1, 1, 1))
    reaches_device_check(f, X, W, off, B, mask, **kw)
    raises_shape("offset", f, X, W, z(1, 18, 8, 8), **kw)
    raises_shape("offset", f, X, W, z(2, 18, 6, 6), **kw)
    raises_shape("offset", f, X, W, off, offset_group=2, **kw)
    raises_shape("mask", f, X, W, off, None, z(2, 9, 7, 8), **kw)
    raises_shape("B", f, X, W, off, z(5), **kw)
    raises_shape("W", f, X, z(6, 3, 3, 3), off, **kw)
    raises_shape("W", f, X, W, off, group=2, **kw)
    raises_shape("out", f, X, W, off, out=z(2, 6, 8, 7), **kw)
    raises_shape("4-D", f, z(4, 8, 8), W, off, **kw)
    reaches_device_check(f, X, z(6, 2, 3, 3), off, group=2, **kw)
