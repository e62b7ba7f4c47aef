"""Plain double-precision CPU oracle for the spatial-transformer sampling path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference legs of ``bench.py`` may import this package.  The
CUDA library never does, and this package imports nothing from it.

The arithmetic lives in ``oracle.c`` (scalar fp64 loops, one output element at
a time, in the order the operator pages state the method).  This module only
builds it with gcc, loads it with ctypes and marshals numpy float64 arrays.
Inputs in float32 / float16 / bfloat16 are widened to float64 exactly by the
caller before they reach here.
"""
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

MODES = {"linear": 0, "bilinear": 0, "nearest": 1, "cubic": 2, "bicubic": 2}
PADS = {"zeros": 0, "border": 1, "reflection": 2}

_lib = None
_lock = threading.Lock()

_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)


class _DeformAttrs(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int64 * 2), ("pads", ctypes.c_int64 * 4),
                ("strides", ctypes.c_int64 * 2), ("dilations", ctypes.c_int64 * 2),
                ("group", ctypes.c_int64), ("offset_group", ctypes.c_int64)]


def build(force=False):
    """Compile oracle.c into _build/liboracle.so with gcc (OpenMP over output elements)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_BUILD_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_variant(src_text, out_path):
    """Compile an edited copy of oracle.c (the tests plant mistakes this way)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                    "-ffp-contract=off", src, "-o", out_path, "-lm"], check=True)
    return out_path


class use_library:
    """Context manager: route every call through another build of oracle.c."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = lib()
        with _lock:
            _lib = _bind(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(L):
    """Declare the C signatures on a loaded build of oracle.c."""
    L.or_affine_grid.argtypes = [_f64p, ctypes.c_int, _i64p, ctypes.c_int, _f64p]
    L.or_grid_sample.argtypes = [_f64p, _i64p, ctypes.c_int, _f64p, _i64p, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_double, _f64p]
    L.or_grid_sample_at.argtypes = [_f64p, _i64p, ctypes.c_int, _f64p, _i64p, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_double, _i64p,
                                    ctypes.c_int64, _f64p]
    L.or_affine_sample.argtypes = [_f64p, _i64p, ctypes.c_int, _f64p, _i64p, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_double, _f64p]
    L.or_affine_sample_at.argtypes = [_f64p, _i64p, ctypes.c_int, _f64p, _i64p, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_double, _i64p,
                                      ctypes.c_int64, _f64p]
    L.or_deform_conv.argtypes = [_f64p, _i64p, _f64p, ctypes.c_int64, _f64p, _f64p, _f64p,
                                 ctypes.POINTER(_DeformAttrs), _f64p]
    L.or_deform_conv_at.argtypes = [_f64p, _i64p, _f64p, ctypes.c_int64, _f64p, _f64p, _f64p,
                                    ctypes.POINTER(_DeformAttrs), _i64p, ctypes.c_int64, _f64p]
    L.or_deform_out_extent.argtypes = [ctypes.c_int64] * 6
    L.or_deform_out_extent.restype = ctypes.c_int64
    L.or_resize_shape.argtypes = [ctypes.c_int, _i64p, _i64p, ctypes.c_int, _f64p, _i64p, _f64p,
                                  ctypes.c_int, ctypes.c_int, _i64p, _f64p, _f64p, _f64p, _f64p]
    L.or_resize.argtypes = [_f64p, ctypes.c_int, _i64p, _i64p, _f64p, _f64p, _f64p, _f64p,
                            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                            ctypes.c_int, ctypes.c_double, ctypes.c_int, _f64p]
    L.or_set_num_threads.argtypes = [ctypes.c_int]
    L.or_max_threads.restype = ctypes.c_int
    L.or_num_procs.restype = ctypes.c_int
    for f in ("or_affine_grid", "or_grid_sample", "or_grid_sample_at", "or_affine_sample",
              "or_affine_sample_at", "or_deform_conv", "or_deform_conv_at", "or_resize_shape",
              "or_resize"):
        getattr(L, f).restype = ctypes.c_int
    return L


def set_num_threads(n):
    lib().or_set_num_threads(int(n))


def max_threads():
    return int(lib().or_max_threads())


def num_procs():
    return int(lib().or_num_procs())


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i64(v):
    return np.ascontiguousarray(np.asarray(v, dtype=np.int64))


def _p(a, t=_f64p):
    return a.ctypes.data_as(t) if a is not None else None


def _check(rc):
    if rc != 0:
        raise ValueError("oracle rejected the arguments")


def affine_grid(theta, size, align_corners=0):
    """AffineGrid: theta (N, r, r+1), size (N, C, spatial...) -> grid (N, spatial..., r)."""
    theta = _f64(theta)
    size = _i64(size)
    r = theta.shape[1]
    assert theta.shape == (size[0], r, r + 1) and size.shape == (r + 2,)
    grid = np.empty(tuple(size[:1]) + tuple(size[2:]) + (r,), dtype=np.float64)
    _check(lib().or_affine_grid(_p(theta), r, _p(size, _i64p), int(align_corners), _p(grid)))
    return grid


def grid_sample(X, grid, mode="linear", padding_mode="zeros", align_corners=0,
                cubic_coeff_a=-0.75):
    """GridSample: X (N, C, in...), grid (N, out..., r) -> Y (N, C, out...)."""
    X, grid = _f64(X), _f64(grid)
    r = X.ndim - 2
    assert grid.ndim == r + 2 and grid.shape[-1] == r and grid.shape[0] == X.shape[0]
    xs = _i64(X.shape)
    out = _i64(grid.shape[1:-1])
    Y = np.empty(X.shape[:2] + grid.shape[1:-1], dtype=np.float64)
    _check(lib().or_grid_sample(_p(X), _p(xs, _i64p), r, _p(grid), _p(out, _i64p), MODES[mode],
                                PADS[padding_mode], int(align_corners), float(cubic_coeff_a),
                                _p(Y)))
    return Y


def grid_sample_at(X, grid, flat_idx, mode="linear", padding_mode="zeros", align_corners=0,
                   cubic_coeff_a=-0.75):
    """GridSample evaluated only at the given flat indices of Y."""
    X, grid = _f64(X), _f64(grid)
    r = X.ndim - 2
    xs = _i64(X.shape)
    out = _i64(grid.shape[1:-1])
    idx = _i64(flat_idx).ravel()
    vals = np.empty(idx.shape, dtype=np.float64)
    _check(lib().or_grid_sample_at(_p(X), _p(xs, _i64p), r, _p(grid), _p(out, _i64p),
                                   MODES[mode], PADS[padding_mode], int(align_corners),
                                   float(cubic_coeff_a), _p(idx, _i64p), idx.size, _p(vals)))
    return vals


def affine_sample(theta, size, X, mode="linear", padding_mode="zeros", align_corners=0,
                  cubic_coeff_a=-0.75):
    """GridSample(X, AffineGrid(theta, size)) with the grid kept in float64."""
    theta, X, size = _f64(theta), _f64(X), _i64(size)
    r = X.ndim - 2
    xs = _i64(X.shape)
    Y = np.empty(X.shape[:2] + tuple(size[2:]), dtype=np.float64)
    _check(lib().or_affine_sample(_p(theta), _p(size, _i64p), r, _p(X), _p(xs, _i64p),
                                  MODES[mode], PADS[padding_mode], int(align_corners),
                                  float(cubic_coeff_a), _p(Y)))
    return Y


def affine_sample_at(theta, size, X, flat_idx, mode="linear", padding_mode="zeros",
                     align_corners=0, cubic_coeff_a=-0.75):
    theta, X, size = _f64(theta), _f64(X), _i64(size)
    r = X.ndim - 2
    xs = _i64(X.shape)
    idx = _i64(flat_idx).ravel()
    vals = np.empty(idx.shape, dtype=np.float64)
    _check(lib().or_affine_sample_at(_p(theta), _p(size, _i64p), r, _p(X), _p(xs, _i64p),
                                     MODES[mode], PADS[padding_mode], int(align_corners),
                                     float(cubic_coeff_a), _p(idx, _i64p), idx.size, _p(vals)))
    return vals


def _deform_attrs(W, kernel_shape, pads, strides, dilations, group, offset_group):
    a = _DeformAttrs()
    ks = kernel_shape if kernel_shape is not None else W.shape[2:]
    a.kernel[:] = [int(k) for k in ks]
    a.pads[:] = [int(p) for p in (pads if pads is not None else [0, 0, 0, 0])]
    a.strides[:] = [int(s) for s in (strides if strides is not None else [1, 1])]
    a.dilations[:] = [int(d) for d in (dilations if dilations is not None else [1, 1])]
    a.group = int(group)
    a.offset_group = int(offset_group)
    return a


def deform_out_shape(x_shape, oC, attrs):
    L = lib()
    oH = L.or_deform_out_extent(x_shape[2], attrs.kernel[0], attrs.pads[0], attrs.pads[2],
                                attrs.strides[0], attrs.dilations[0])
    oW = L.or_deform_out_extent(x_shape[3], attrs.kernel[1], attrs.pads[1], attrs.pads[3],
                                attrs.strides[1], attrs.dilations[1])
    return (x_shape[0], oC, oH, oW)


def deform_conv(X, W, offset, B=None, mask=None, kernel_shape=None, pads=None, strides=None,
                dilations=None, group=1, offset_group=1):
    """DeformConv 2-D: X (N,C,H,W), W (oC,C/group,kH,kW), offset (N,og*kH*kW*2,oH,oW)."""
    X, W, offset = _f64(X), _f64(W), _f64(offset)
    B = _f64(B) if B is not None else None
    mask = _f64(mask) if mask is not None else None
    at = _deform_attrs(W, kernel_shape, pads, strides, dilations, group, offset_group)
    xs = _i64(X.shape)
    Y = np.empty(deform_out_shape(X.shape, W.shape[0], at), dtype=np.float64)
    _check(lib().or_deform_conv(_p(X), _p(xs, _i64p), _p(W), W.shape[0], _p(offset), _p(B),
                                _p(mask), ctypes.byref(at), _p(Y)))
    return Y


def deform_conv_at(X, W, offset, flat_idx, B=None, mask=None, kernel_shape=None, pads=None,
                   strides=None, dilations=None, group=1, offset_group=1):
    X, W, offset = _f64(X), _f64(W), _f64(offset)
    B = _f64(B) if B is not None else None
    mask = _f64(mask) if mask is not None else None
    at = _deform_attrs(W, kernel_shape, pads, strides, dilations, group, offset_group)
    xs = _i64(X.shape)
    idx = _i64(flat_idx).ravel()
    vals = np.empty(idx.shape, dtype=np.float64)
    _check(lib().or_deform_conv_at(_p(X), _p(xs, _i64p), _p(W), W.shape[0], _p(offset), _p(B),
                                   _p(mask), ctypes.byref(at), _p(idx, _i64p), idx.size,
                                   _p(vals)))
    return vals


RESIZE_MODES = {"nearest": 1, "linear": 0, "cubic": 2}
RESIZE_COORDS = {"half_pixel": 0, "pytorch_half_pixel": 1, "align_corners": 2, "asymmetric": 3,
                 "tf_crop_and_resize": 4}
RESIZE_NEAREST = {"round_prefer_floor": 0, "round_prefer_ceil": 1, "floor": 2, "ceil": 3}
RESIZE_KEEP = {"stretch": 0, "not_larger": 1, "not_smaller": 2}


def resize_shape(x_shape, scales=None, sizes=None, roi=None, axes=None,
                 coordinate_transformation_mode="half_pixel", keep_aspect_ratio_policy="stretch"):
    """Resize output extents and per-axis (scale, length_resized, roi_start, roi_end)."""
    xs = _i64(x_shape)
    rank = xs.size
    ax = _i64(axes) if axes is not None else None
    na = 0 if ax is None else ax.size
    sc = _f64(scales) if scales is not None else None
    sz = _i64(sizes) if sizes is not None else None
    ro = _f64(roi) if roi is not None else None
    out = np.empty(rank, dtype=np.int64)
    scale, lres, r0, r1 = (np.empty(rank, dtype=np.float64) for _ in range(4))
    _check(lib().or_resize_shape(rank, _p(xs, _i64p), _p(ax, _i64p), na, _p(sc), _p(sz, _i64p),
                                 _p(ro), RESIZE_COORDS[coordinate_transformation_mode],
                                 RESIZE_KEEP[keep_aspect_ratio_policy], _p(out, _i64p),
                                 _p(scale), _p(lres), _p(r0), _p(r1)))
    return tuple(int(v) for v in out), scale, lres, r0, r1


def resize(X, scales=None, sizes=None, roi=None, axes=None, mode="nearest",
           coordinate_transformation_mode="half_pixel", nearest_mode="round_prefer_floor",
           cubic_coeff_a=-0.75, exclude_outside=0, extrapolation_value=0.0, antialias=0,
           keep_aspect_ratio_policy="stretch"):
    """Resize - 18 on an N-D array (one of scales / sizes, for `axes` or all axes)."""
    X = _f64(X)
    out, scale, lres, r0, r1 = resize_shape(X.shape, scales, sizes, roi, axes,
                                            coordinate_transformation_mode,
                                            keep_aspect_ratio_policy)
    Y = np.empty(out, dtype=np.float64)
    if Y.size == 0:
        return Y
    xs = _i64(X.shape)
    os_ = _i64(out)
    _check(lib().or_resize(_p(X), X.ndim, _p(xs, _i64p), _p(os_, _i64p), _p(scale), _p(lres),
                           _p(r0), _p(r1), RESIZE_MODES[mode],
                           RESIZE_COORDS[coordinate_transformation_mode],
                           RESIZE_NEAREST[nearest_mode], float(cubic_coeff_a),
                           int(exclude_outside), float(extrapolation_value), int(antialias),
                           _p(Y)))
    return Y


INT_RANGES = {"uint8": (0, 255), "int8": (-128, 127), "uint16": (0, 65535), "int16": (-32768, 32767)}


def cast_to_integer(values, dtype):
    """GridSample - version 20, Outputs: integer X is interpolated in floating point and
    cast to the integer type at the end.  Reading: truncation toward zero, saturated at
    the type's range (cubic weights can overshoot it)."""
    lo, hi = INT_RANGES[dtype]
    v = np.clip(np.asarray(values, dtype=np.float64), lo, hi)
    return np.trunc(v).astype(np.int64)
