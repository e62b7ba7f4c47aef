"""The C ABI without a GPU: the library builds, loads, exports every entry point
include/gs.h declares, and rejects bad arguments on the host (before any
CUDA call, so these run on a machine with no GPU)."""
import ctypes
import os
import re

import pytest

import spatial_transformer_sampling_gb300 as gs
from spatial_transformer_sampling_gb300 import build as gsbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "gs.h")


@pytest.fixture(scope="module")
def L():
    gsbuild.build()
    return gs.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gs_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gs_affine_grid", "gs_grid_sample", "gs_affine_sample", "gs_deform_conv"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(gs.EXPORTED_SYMBOLS) <= set(declared_functions())


def test_version_and_status_strings(L):
    assert L.gs_version().decode().count(".") == 2
    assert gs.gs_status_str(0) == "ok"
    assert "shape" in gs.gs_status_str(3)


def _i64(v):
    return (ctypes.c_int64 * len(v))(*v)


FAKE = 0x10000   # a non-null, aligned pointer value; never dereferenced on these paths


def _gsample(L, x_shape, out, r=2, dt=0, mode=0, pad=0, ac=0, a=-0.75, X=FAKE, grid=FAKE, Y=FAKE,
             entry="gs_grid_sample"):
    if entry == "gs_grid_sample_ws":   # no workspace: checks as gs_grid_sample
        return L.gs_grid_sample_ws(X, _i64(x_shape), r, grid, _i64(out), dt, mode, pad, ac, a,
                                   None, 0, Y, None)
    return getattr(L, entry)(X, _i64(x_shape), r, grid, _i64(out), dt, mode, pad, ac, a, Y, None)


ENTRIES = ["gs_grid_sample", "gs_grid_sample_ws", "gs_grid_sample_static"]


@pytest.mark.parametrize("kwargs,status", [
    (dict(mode=3), 5), (dict(pad=-1), 5), (dict(ac=2), 5), (dict(dt=9), 4),
    (dict(r=7, x_shape=[1, 1] + [2] * 7, out=[2] * 7), 2), (dict(r=0), 2),
    (dict(X=None), 1), (dict(Y=None), 1), (dict(grid=None), 1),
    (dict(X=FAKE + 2), 6), (dict(dt=1, Y=FAKE + 1), 6),
    (dict(x_shape=[1, 1, 1 << 21, 2]), 3), (dict(x_shape=[1, 1, -1, 2]), 3),
    (dict(x_shape=[1, 1, 1 << 16, 1 << 16]), 3), (dict(x_shape=[1, 1, 0, 4]), 3),
    (dict(mode=2, a=float("nan")), 5),
])
@pytest.mark.parametrize("entry", ENTRIES)
def test_grid_sample_rejects_bad_arguments(L, kwargs, status, entry):
    args = dict(x_shape=[2, 3, 4, 5], out=[3, 3], entry=entry)
    args.update(kwargs)
    assert _gsample(L, **args) == status


@pytest.mark.parametrize("x_shape,out", [([0, 3, 4, 5], [3, 3]), ([2, 0, 4, 5], [3, 3]),
                                         ([2, 3, 4, 5], [0, 3])])
@pytest.mark.parametrize("entry", ENTRIES)
def test_empty_tensors_return_ok_without_a_launch(L, x_shape, out, entry):
    assert _gsample(L, x_shape, out, X=None, grid=None, Y=None, entry=entry) == 0


@pytest.mark.parametrize("r", [4, 5, 6])
@pytest.mark.parametrize("entry", ENTRIES)
def test_ranks_four_to_six_are_accepted(L, r, entry):
    # an empty output passes every check and returns without a launch
    xs = [2, 3] + [4] * r
    assert _gsample(L, xs, [0] + [3] * (r - 1), X=None, grid=None, Y=None, r=r, entry=entry) == 0
    # a bad extent at the innermost axis is still caught
    assert _gsample(L, [2, 3] + [4] * (r - 1) + [-1], [3] * r, r=r, entry=entry) == 3


def test_affine_sample_from_host_checks(L):
    f = L.gs_affine_sample_from_host
    streams = (ctypes.c_void_p * 3)(None, None, None)
    size, xs = _i64([2, 3, 4, 4]), _i64([2, 3, 4, 4])

    def call(r=2, size=size, xs=xs, theta_h=FAKE, X_h=FAKE, Y_h=FAKE, theta_d=FAKE, X_d=FAKE,
             Y_d=FAKE, streams=streams):
        return f(theta_h, size, r, X_h, xs, 0, 0, 0, 0, -0.75, Y_h, theta_d, X_d, Y_d, 2, streams)

    assert call(r=1) == 2 and call(r=4) == 2                                  # rank
    assert call(size=_i64([2, 4, 4, 4])) == 3                                  # C mismatch
    assert call(streams=None) == 1 and call(X_h=None) == 1 and call(theta_d=None) == 1
    assert call(Y_d=None) == 1 and call(Y_h=None) == 1
    assert call(X_d=FAKE + 2) == 6                                             # misaligned
    # an empty batch returns before any pointer is needed
    assert call(size=_i64([0, 3, 4, 4]), xs=_i64([0, 3, 4, 4]), theta_h=None, X_h=None, Y_h=None,
                theta_d=None, X_d=None, Y_d=None, streams=None) == 0


def test_static_scratch_rejects_an_image_slot_beyond_its_size(L):
    # (512*513 + 1) * 64 fp32 elements exceed the 64 MiB scratch: refused on the host
    assert _gsample(L, [1, 64, 512, 513], [4, 4], entry="gs_grid_sample_static") == 3


def test_affine_sample_checks(L):
    f = L.gs_affine_sample
    assert f(FAKE, _i64([2, 3, 4, 4]), 1, FAKE, _i64([2, 3, 4]), 0, 0, 0, 0, -0.75, FAKE, None) == 2
    assert f(FAKE, _i64([2, 4, 4, 4]), 2, FAKE, _i64([2, 3, 4, 4]), 0, 0, 0, 0, -0.75, FAKE, None) == 3
    assert f(None, _i64([2, 3, 4, 4]), 2, FAKE, _i64([2, 3, 4, 4]), 0, 0, 0, 0, -0.75, FAKE, None) == 1
    assert f(FAKE, _i64([0, 3, 4, 4]), 2, None, _i64([0, 3, 4, 4]), 0, 0, 0, 0, -0.75, None, None) == 0


def test_affine_grid_checks(L):
    f = L.gs_affine_grid
    assert f(FAKE, 0, 1, _i64([1, 1, 4]), 0, FAKE, None) == 2
    assert f(FAKE, 0, 2, _i64([1, 1, 4, 4]), 3, FAKE, None) == 5
    assert f(FAKE, 5, 2, _i64([1, 1, 4, 4]), 0, FAKE, None) == 4
    assert f(None, 0, 2, _i64([1, 1, 4, 4]), 0, FAKE, None) == 1
    assert f(None, 0, 2, _i64([0, 1, 4, 4]), 0, None, None) == 0


def _deform(L, x_shape=(1, 4, 8, 8), oC=4, kernel=(3, 3), pads=(1, 1, 1, 1), strides=(1, 1),
            dil=(1, 1), group=1, og=1, X=FAKE, ws=False):
    a = gs.deform_attrs(kernel, pads, strides, dil, group, og)
    if ws:   # no workspace: checks as gs_deform_conv
        return L.gs_deform_conv_ws(X, _i64(list(x_shape)), FAKE, oC, FAKE, None, None,
                                   ctypes.byref(a), 0, None, 0, FAKE, None)
    return L.gs_deform_conv(X, _i64(list(x_shape)), FAKE, oC, FAKE, None, None, ctypes.byref(a), 0,
                            FAKE, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(group=3), 5), (dict(og=3), 5), (dict(oC=6, group=4), 5), (dict(kernel=(0, 3)), 5),
    (dict(strides=(0, 1)), 5), (dict(dil=(1, 0)), 5), (dict(pads=(-1, 0, 0, 0)), 5),
    (dict(x_shape=(1, 4, 2, 2), pads=(0, 0, 0, 0)), 3), (dict(X=None), 1),
])
@pytest.mark.parametrize("ws", [False, True])
def test_deform_conv_rejects_bad_arguments(L, kwargs, status, ws):
    assert _deform(L, ws=ws, **kwargs) == status


def test_deform_conv_workspace_size_queries(L):
    n = ctypes.c_size_t(7)
    a = gs.deform_attrs((3, 3), (1, 1, 1, 1))
    # bf16, 3x3: the staged kernel takes the shape and wants no workspace
    assert L.gs_deform_conv_workspace_size(_i64([8, 64, 64, 64]), 64, ctypes.byref(a), 2,
                                           ctypes.byref(n)) == 0 and n.value == 0
    # bf16, 1x5 (a tap count the staged kernel does not take): the channel-last
    # path's packed W (64*64*5*2 bytes) + 8 slots of (64*64 + 1) * 64 * 2
    a5 = gs.deform_attrs((1, 5), (0, 2, 0, 2))
    assert L.gs_deform_conv_workspace_size(_i64([8, 64, 64, 64]), 64, ctypes.byref(a5), 2,
                                           ctypes.byref(n)) == 0
    assert n.value == 64 * 64 * 5 * 2 + 8 * (64 * 64 + 1) * 64 * 2
    assert L.gs_deform_conv_workspace_size(_i64([8, 64, 64, 64]), 64, ctypes.byref(a), 0,
                                           ctypes.byref(n)) == 0 and n.value == 0   # fp32
    assert L.gs_deform_conv_workspace_size(_i64([8, 64, 64, 64]), 64, ctypes.byref(a), 2,
                                           None) == 1
    bad = gs.deform_attrs((3, 3), (1, 1, 1, 1), group=3)
    assert L.gs_deform_conv_workspace_size(_i64([8, 64, 64, 64]), 64, ctypes.byref(bad), 2,
                                           ctypes.byref(n)) == 5


def test_deform_conv_null_attrs(L):
    assert L.gs_deform_conv(FAKE, _i64([1, 1, 4, 4]), FAKE, 1, FAKE, None, None, None, 0, FAKE,
                            None) == 1


# ------------------------------------------------------------------ Resize host logic

def _resize_shape_lib(x_shape, **kw):
    return gs.gs_resize_output_shape(tuple(x_shape), **kw)


@pytest.mark.parametrize("case", [
    dict(x=(1, 1, 4, 4), scales=[1, 1, 0.6, 0.6]),
    dict(x=(1, 1, 2, 4), scales=[1, 1, 0.6, 0.6]),
    dict(x=(2, 3, 7, 10), scales=[1, 1, 0.5, 1.55]),
    dict(x=(1, 1, 2, 2), sizes=[7, 8], axes=[2, 3], keep_aspect_ratio_policy="not_larger"),
    dict(x=(1, 1, 2, 2), sizes=[7, 8], axes=[2, 3], keep_aspect_ratio_policy="not_smaller"),
    dict(x=(1, 1, 2, 4), sizes=[1, 3], axes=[2, 3], keep_aspect_ratio_policy="not_smaller"),
    dict(x=(1, 1, 4, 4), sizes=[3, 3], axes=[3, 2], roi=[0.6, 0.4, 0.8, 0.6],
         coordinate_transformation_mode="tf_crop_and_resize"),
    dict(x=(1, 1, 4, 4), scales=[0.8, 0.5], axes=[-1, -2], roi=[0.2, 0.0, 0.9, 1.0],
         coordinate_transformation_mode="tf_crop_and_resize"),
    dict(x=(5, 9, 3), scales=[1, 2.5, 1 / 3]),
])
def test_resize_output_shape_matches_oracle(L, oracle_mod, case):
    case = dict(case)
    x = case.pop("x")
    got = _resize_shape_lib(x, **case)
    coord = case.get("coordinate_transformation_mode", "half_pixel")
    keep = case.get("keep_aspect_ratio_policy", "stretch")
    exp = oracle_mod.resize_shape(x, case.get("scales"), case.get("sizes"), case.get("roi"),
                                  case.get("axes"), coord, keep)[0]
    assert got == exp


def test_resize_rejects_bad_arguments_on_the_host(L):
    at = gs.resize_attrs()
    f32 = lambda *v: (ctypes.c_float * len(v))(*v)
    shape = _i64([1, 1, 4, 4])
    out = (ctypes.c_int64 * 4)()
    # both scales and sizes, neither, a zero scale, a repeated axis, a bad mode
    assert L.gs_resize_output_shape(4, shape, None, 0, f32(1, 1, 2, 2), _i64([1, 1, 8, 8]), None,
                                    ctypes.byref(at), out) == 5
    assert L.gs_resize_output_shape(4, shape, None, 0, None, None, None, ctypes.byref(at), out) == 5
    assert L.gs_resize_output_shape(4, shape, None, 0, f32(1, 1, 0, 2), None, None,
                                    ctypes.byref(at), out) == 5
    assert L.gs_resize_output_shape(4, shape, _i64([2, -2]), 2, f32(2, 2), None, None,
                                    ctypes.byref(at), out) == 3
    bad = gs.resize_attrs()
    bad.mode = 7
    assert L.gs_resize_output_shape(4, shape, None, 0, f32(1, 1, 2, 2), None, None,
                                    ctypes.byref(bad), out) == 5
    # four resized axes, and an antialiased downscale needing more than 64 taps
    four = _i64([2, 2, 4, 4])
    assert L.gs_resize(FAKE, 4, four, None, 0, f32(2, 1, 2, 2), None, None, ctypes.byref(at), 0,
                       FAKE, None) == 9
    aa = gs.resize_attrs(mode="cubic", antialias=1)
    big = _i64([1, 1, 1024, 1024])
    assert L.gs_resize(FAKE, 4, big, None, 0, f32(1, 1, 0.01, 0.01), None, None, ctypes.byref(aa),
                       0, FAKE, None) == 9
    # an empty output needs no pointers; an empty input with a nonempty output is a shape error
    assert L.gs_resize(None, 4, _i64([1, 1, 4, 4]), None, 0, None, _i64([1, 1, 0, 3]), None,
                       ctypes.byref(at), 0, None, None) == 0
    assert L.gs_resize(FAKE, 4, _i64([1, 1, 0, 4]), None, 0, None, _i64([1, 1, 3, 3]), None,
                       ctypes.byref(at), 0, FAKE, None) == 3


def test_integer_x_entry_rejects_bad_types_on_the_host(L):
    xs, out = _i64([1, 2, 4, 4]), _i64([3, 3])
    # X type not an integer code, grid type not a float code, bad rank
    assert L.gs_grid_sample_int(FAKE, 0, xs, 2, FAKE, 0, out, 0, 0, 0, -0.75, FAKE, None) == 4
    assert L.gs_grid_sample_int(FAKE, 16, xs, 2, FAKE, 9, out, 0, 0, 0, -0.75, FAKE, None) == 4
    assert L.gs_grid_sample_int(FAKE, 16, _i64([1, 2] + [4] * 7), 7, FAKE, 0, _i64([3] * 7), 0, 0,
                                0, -0.75, FAKE, None) == 2
    # misaligned int16 X
    assert L.gs_grid_sample_int(FAKE + 1, 19, xs, 2, FAKE, 0, out, 0, 0, 0, -0.75, FAKE, None) == 6
    # empty output: no launch, no pointers needed
    assert L.gs_grid_sample_int(None, 16, xs, 2, None, 0, _i64([0, 3]), 0, 0, 0, -0.75, None,
                                None) == 0


def test_bounded_wait_hook_rejects_limits_on_the_host(L):
    # 0 and more than a second are refused before anything is enqueued
    assert L.gs_test_bounded_wait_expires(0, None) == 5
    assert L.gs_test_bounded_wait_expires(1_000_000_001, None) == 5
