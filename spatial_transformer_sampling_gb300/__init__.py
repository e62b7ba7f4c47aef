"""GB300-native spatial-transformer sampling: thin Python binding of libgs.

The functions here carry the C ABI's names (include/gs.h) and only marshal
arguments: they check that tensors are contiguous CUDA tensors of one dtype,
allocate outputs with torch when none is given, and pass raw pointers plus the
current torch stream to the library.  Every step of the computation runs in
libgs's kernels.  There is no CPU fallback: if the library is missing or a
call fails, an exception is raised.

Operators (see the docstrings and include/gs.h):
  gs_affine_grid   AffineGrid
  gs_grid_sample   GridSample (rank 1-6; linear / nearest / cubic;
                   zeros / border / reflection; both align_corners)
  gs_affine_sample GridSample(X, AffineGrid(theta, size)) fused
  gs_deform_conv   DeformConv 2-D

Host-memory variants (gs_affine_sample_from_host, gs_grid_sample_from_host)
stream a batch from pinned host memory in chunks, overlapping the copies in
both directions with the kernels.
"""
import ctypes
import os

__all__ = ["gs_affine_grid", "gs_grid_sample", "gs_affine_sample", "gs_deform_conv",
           "gs_status_str", "gs_device_status", "GsError", "library_path", "load_library",
           "EXPORTED_SYMBOLS", "HostStreamer", "gs_affine_sample_from_host",
           "gs_grid_sample_from_host"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libgs.so")

EXPORTED_SYMBOLS = ("gs_affine_grid", "gs_grid_sample", "gs_affine_sample",
                    "gs_affine_sample_from_host", "gs_deform_conv",
                    "gs_resize", "gs_resize_output_shape", "gs_grid_sample_int", "gs_status_str",
                    "gs_device_status",
                    "gs_version")

MODES = {"linear": 0, "bilinear": 0, "nearest": 1, "cubic": 2, "bicubic": 2}
PADS = {"zeros": 0, "border": 1, "reflection": 2}
STATUS = {0: "GS_OK", 1: "GS_ERR_NULL", 2: "GS_ERR_RANK", 3: "GS_ERR_SHAPE", 4: "GS_ERR_DTYPE",
          5: "GS_ERR_ATTR", 6: "GS_ERR_ALIGN", 7: "GS_ERR_CUDA", 8: "GS_ERR_TIMEOUT",
          9: "GS_ERR_UNSUPPORTED"}

_lib = None


class GsError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({gs_status_str(status)})")


class ResizeAttrs(ctypes.Structure):
    """gs_resize_attrs (include/gs.h)."""
    _fields_ = [("mode", ctypes.c_int), ("coord", ctypes.c_int), ("nearest_mode", ctypes.c_int),
                ("cubic_coeff_a", ctypes.c_float), ("exclude_outside", ctypes.c_int),
                ("extrapolation_value", ctypes.c_float), ("antialias", ctypes.c_int),
                ("keep_aspect_ratio_policy", ctypes.c_int)]


RESIZE_COORDS = {"half_pixel": 0, "pytorch_half_pixel": 1, "align_corners": 2, "asymmetric": 3,
                 "tf_crop_and_resize": 4}
RESIZE_NEAREST = {"round_prefer_floor": 0, "round_prefer_ceil": 1, "floor": 2, "ceil": 3}
RESIZE_KEEP = {"stretch": 0, "not_larger": 1, "not_smaller": 2}


class DeformAttrs(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int64 * 2), ("pads", ctypes.c_int64 * 4),
                ("strides", ctypes.c_int64 * 2), ("dilations", ctypes.c_int64 * 2),
                ("group", ctypes.c_int64), ("offset_group", ctypes.c_int64)]


def library_path():
    return _LIB_PATH


def load_library(path=None):
    """Load libgs.so (built by spatial_transformer_sampling_gb300/build.py)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libgs.so not built ({p}); run __graft_entry__.build() first")
    L = ctypes.CDLL(p)
    vp, i64p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64)
    ci, cf = ctypes.c_int, ctypes.c_float
    L.gs_affine_grid.argtypes = [vp, ci, ci, i64p, ci, vp, vp]
    L.gs_grid_sample.argtypes = [vp, i64p, ci, vp, i64p, ci, ci, ci, ci, cf, vp, vp]
    L.gs_grid_sample_workspace_size.argtypes = [i64p, ci, i64p, ci, ctypes.POINTER(ctypes.c_size_t)]
    L.gs_grid_sample_ws.argtypes = [vp, i64p, ci, vp, i64p, ci, ci, ci, ci, cf, vp, ctypes.c_size_t,
                                    vp, vp]
    L.gs_grid_sample_static.argtypes = [vp, i64p, ci, vp, i64p, ci, ci, ci, ci, cf, vp, vp]
    L.gs_affine_sample.argtypes = [vp, i64p, ci, vp, i64p, ci, ci, ci, ci, cf, vp, vp]
    L.gs_affine_sample_from_host.argtypes = [vp, i64p, ci, vp, i64p, ci, ci, ci, ci, cf, vp, vp, vp,
                                             vp, ci, ctypes.POINTER(ctypes.c_void_p)]
    L.gs_deform_conv.argtypes = [vp, i64p, vp, ctypes.c_int64, vp, vp, vp,
                                 ctypes.POINTER(DeformAttrs), ci, vp, vp]
    L.gs_deform_conv_workspace_size.argtypes = [i64p, ctypes.c_int64, ctypes.POINTER(DeformAttrs),
                                                ci, ctypes.POINTER(ctypes.c_size_t)]
    L.gs_deform_conv_ws.argtypes = [vp, i64p, vp, ctypes.c_int64, vp, vp, vp,
                                    ctypes.POINTER(DeformAttrs), ci, vp, ctypes.c_size_t, vp, vp]
    L.gs_grid_sample_int.argtypes = [vp, ci, i64p, ci, vp, ci, i64p, ci, ci, ci, cf, vp, vp]
    f32p = ctypes.POINTER(ctypes.c_float)
    L.gs_resize_output_shape.argtypes = [ci, i64p, i64p, ci, f32p, i64p, f32p,
                                         ctypes.POINTER(ResizeAttrs), i64p]
    L.gs_resize.argtypes = [vp, ci, i64p, i64p, ci, f32p, i64p, f32p, ctypes.POINTER(ResizeAttrs),
                            ci, vp, vp]
    L.gs_status_str.argtypes = [ci]
    L.gs_status_str.restype = ctypes.c_char_p
    L.gs_device_status.argtypes = [vp]
    L.gs_test_bounded_wait_expires.argtypes = [ctypes.c_uint64, vp]
    L.gs_version.restype = ctypes.c_char_p
    for f in ("gs_affine_grid", "gs_grid_sample", "gs_grid_sample_workspace_size",
              "gs_grid_sample_ws", "gs_grid_sample_static", "gs_affine_sample",
              "gs_affine_sample_from_host", "gs_deform_conv",
              "gs_deform_conv_workspace_size", "gs_deform_conv_ws", "gs_device_status",
              "gs_resize_output_shape", "gs_resize", "gs_grid_sample_int",
              "gs_test_bounded_wait_expires"):
        getattr(L, f).restype = ci
    if path is None:
        _lib = L
    return L


def gs_status_str(status):
    return load_library().gs_status_str(int(status)).decode()


def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    codes = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
    if t.dtype not in codes:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def _check_tensors(*ts):
    ref = next(t for t in ts if t is not None)
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("libgs takes CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("libgs takes contiguous tensors")
        if t.dtype != ref.dtype or t.device != ref.device:
            raise ValueError("all tensors of one call share dtype and device")
    return ref


def _shape_error(what, got, want):
    raise ValueError(f"{what} has shape {tuple(got)}, expected {tuple(want)}")


def _check_sample_shapes(X, grid, out):
    """The C ABI receives X's shape and the output extents only, and trusts that
    grid is (N, out..., r) and out is (N, C, out...): check both here.  Shapes
    only, so that it runs before (and without) any device work."""
    if X.dim() < 3:
        raise ValueError(f"X must be (N, C, spatial...), got {tuple(X.shape)}")
    r = X.dim() - 2
    if grid.dim() != X.dim() or grid.shape[0] != X.shape[0] or grid.shape[-1] != r:
        raise ValueError(f"grid has shape {tuple(grid.shape)}, expected (N={X.shape[0]}, "
                         f"{r} output extents, {r}) for X of shape {tuple(X.shape)}")
    want = list(X.shape[:2]) + list(grid.shape[1:-1])
    if out is not None and list(out.shape) != want:
        _shape_error("out", out.shape, want)
    return r, list(grid.shape[1:-1])


def _i64(vals):
    arr = (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])
    return arr


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(t):
    return ctypes.c_void_p(_torch().cuda.current_stream(t.device).cuda_stream)


def _ok(status, where):
    if status != 0:
        raise GsError(status, where)


def gs_affine_grid(theta, size, align_corners=0, out=None):
    """AffineGrid: theta (N, r, r+1) -> grid (N, spatial..., r); size = (N, C, spatial...)."""
    torch = _torch()
    size = [int(s) for s in size]
    r = len(size) - 2
    if list(theta.shape) != [size[0], r, r + 1]:
        _shape_error("theta", theta.shape, (size[0], r, r + 1))
    if out is not None and list(out.shape) != [size[0]] + size[2:] + [r]:
        _shape_error("out", out.shape, [size[0]] + size[2:] + [r])
    _check_tensors(theta, out)
    if out is None:
        out = torch.empty([size[0]] + size[2:] + [r], dtype=theta.dtype, device=theta.device)
    _ok(load_library().gs_affine_grid(_ptr(theta), _dtype_code(theta), r, _i64(size),
                                      int(align_corners), _ptr(out), _stream(theta)),
        "gs_affine_grid")
    return out


def gs_grid_sample(X, grid, mode="linear", padding_mode="zeros", align_corners=0,
                   cubic_coeff_a=-0.75, out=None, workspace=None):
    """GridSample: X (N, C, in...), grid (N, out..., r) -> Y (N, C, out...).

    ``workspace``: None calls gs_grid_sample; a device tensor (any dtype, used as
    raw bytes) or "auto" (one of the size gs_grid_sample_workspace_size asks
    for, from torch's allocator) calls gs_grid_sample_ws."""
    torch = _torch()
    r, out_sp = _check_sample_shapes(X, grid, out)
    _check_tensors(X, grid, out)
    if out is None:
        out = torch.empty(list(X.shape[:2]) + out_sp, dtype=X.dtype, device=X.device)
    if workspace is not None:
        return gs_grid_sample_ws(X, grid, workspace, mode, padding_mode, align_corners,
                                 cubic_coeff_a, out)
    _ok(load_library().gs_grid_sample(_ptr(X), _i64(X.shape), r, _ptr(grid), _i64(out_sp),
                                      _dtype_code(X), MODES[mode], PADS[padding_mode],
                                      int(align_corners), float(cubic_coeff_a), _ptr(out),
                                      _stream(X)), "gs_grid_sample")
    return out


def _int_code(t):
    torch = _torch()
    codes = {torch.uint8: 16, torch.int8: 17, torch.int16: 19}
    if hasattr(torch, "uint16"):
        codes[torch.uint16] = 18
    if t.dtype not in codes:
        raise TypeError(f"unsupported integer dtype {t.dtype}")
    return codes[t.dtype]


def gs_grid_sample_int(X, grid, mode="linear", padding_mode="zeros", align_corners=0,
                       cubic_coeff_a=-0.75, out=None):
    """GridSample with an integer X (uint8, int8, uint16, int16) and a float grid: fp32
    intermediates, truncated toward zero and saturated at the end (gs_grid_sample_int)."""
    torch = _torch()
    r, out_sp = _check_sample_shapes(X, grid, out)
    for t in (X, grid, out):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("libgs takes contiguous CUDA tensors")
    if out is not None and out.dtype != X.dtype:
        raise ValueError("out must have X's dtype")
    if out is None:
        out = torch.empty(list(X.shape[:2]) + out_sp, dtype=X.dtype, device=X.device)
    _ok(load_library().gs_grid_sample_int(_ptr(X), _int_code(X), _i64(X.shape), r, _ptr(grid),
                                          _dtype_code(grid), _i64(out_sp), MODES[mode],
                                          PADS[padding_mode], int(align_corners),
                                          float(cubic_coeff_a), _ptr(out), _stream(X)),
        "gs_grid_sample_int")
    return out


def gs_grid_sample_workspace_size(x_shape, out_spatial, dtype):
    """Workspace bytes gs_grid_sample_ws asks for (0: the shape never uses one)."""
    torch = _torch()
    code = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[dtype]
    n = ctypes.c_size_t(0)
    _ok(load_library().gs_grid_sample_workspace_size(_i64(x_shape), len(x_shape) - 2,
                                                     _i64(out_spatial), code, ctypes.byref(n)),
        "gs_grid_sample_workspace_size")
    return int(n.value)


def gs_grid_sample_ws(X, grid, workspace="auto", mode="linear", padding_mode="zeros",
                      align_corners=0, cubic_coeff_a=-0.75, out=None):
    """gs_grid_sample with a device workspace (see gs_grid_sample_ws in gs.h)."""
    torch = _torch()
    r, out_sp = _check_sample_shapes(X, grid, out)
    _check_tensors(X, grid, out)
    if out is None:
        out = torch.empty(list(X.shape[:2]) + out_sp, dtype=X.dtype, device=X.device)
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError(f"workspace must be a tensor, None or 'auto', not {workspace!r}")
        nbytes = gs_grid_sample_workspace_size(X.shape, out_sp, X.dtype)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=X.device) if nbytes else None
    if workspace is not None:
        if not workspace.is_cuda or workspace.device != X.device or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on X's device")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    else:
        ws_ptr, ws_bytes = None, 0
    _ok(load_library().gs_grid_sample_ws(_ptr(X), _i64(X.shape), r, _ptr(grid), _i64(out_sp),
                                         _dtype_code(X), MODES[mode], PADS[padding_mode],
                                         int(align_corners), float(cubic_coeff_a), ws_ptr,
                                         ws_bytes, _ptr(out), _stream(X)), "gs_grid_sample_ws")
    return out


def gs_grid_sample_static(X, grid, mode="linear", padding_mode="zeros", align_corners=0,
                          cubic_coeff_a=-0.75, out=None):
    """gs_grid_sample with its scratch in the library's static device memory
    (gs_grid_sample_static in gs.h), for callers that cannot allocate device
    memory at the call: the C entry point allocates nothing.  Pass ``out`` to keep
    this wrapper from allocating the output with torch.  Concurrent calls race on
    the one scratch; the first call on a device should precede any stream capture."""
    torch = _torch()
    r, out_sp = _check_sample_shapes(X, grid, out)
    _check_tensors(X, grid, out)
    if out is None:
        out = torch.empty(list(X.shape[:2]) + out_sp, dtype=X.dtype, device=X.device)
    _ok(load_library().gs_grid_sample_static(_ptr(X), _i64(X.shape), r, _ptr(grid),
                                             _i64(out_sp), _dtype_code(X), MODES[mode],
                                             PADS[padding_mode], int(align_corners),
                                             float(cubic_coeff_a), _ptr(out), _stream(X)),
        "gs_grid_sample_static")
    return out


STATIC_WORKSPACE_BYTES = 64 << 20   # GS_STATIC_WORKSPACE_BYTES in gs.h


def gs_affine_sample(theta, size, X, mode="linear", padding_mode="zeros", align_corners=0,
                     cubic_coeff_a=-0.75, out=None):
    """GridSample(X, AffineGrid(theta, size)) in one kernel; size = (N, C, out...)."""
    torch = _torch()
    size = [int(s) for s in size]
    r = X.dim() - 2
    if len(size) != X.dim() or size[:2] != list(X.shape[:2]):
        raise ValueError(f"size {tuple(size)} must be (N, C, out...) with X's N and C "
                         f"(X has shape {tuple(X.shape)})")
    if list(theta.shape) != [size[0], r, r + 1]:
        _shape_error("theta", theta.shape, (size[0], r, r + 1))
    if out is not None and list(out.shape) != size:
        _shape_error("out", out.shape, size)
    _check_tensors(X, theta, out)
    if out is None:
        out = torch.empty(list(X.shape[:2]) + size[2:], dtype=X.dtype, device=X.device)
    _ok(load_library().gs_affine_sample(_ptr(theta), _i64(size), r, _ptr(X), _i64(X.shape),
                                        _dtype_code(X), MODES[mode], PADS[padding_mode],
                                        int(align_corners), float(cubic_coeff_a), _ptr(out),
                                        _stream(X)), "gs_affine_sample")
    return out


def deform_attrs(kernel_shape, pads=None, strides=None, dilations=None, group=1, offset_group=1):
    a = DeformAttrs()
    a.kernel[:] = [int(k) for k in kernel_shape]
    a.pads[:] = [int(p) for p in (pads if pads is not None else (0, 0, 0, 0))]
    a.strides[:] = [int(s) for s in (strides if strides is not None else (1, 1))]
    a.dilations[:] = [int(d) for d in (dilations if dilations is not None else (1, 1))]
    a.group = int(group)
    a.offset_group = int(offset_group)
    return a


def deform_out_hw(H, W, a):
    oH = (H + a.pads[0] + a.pads[2] - a.dilations[0] * (a.kernel[0] - 1) - 1) // a.strides[0] + 1
    oW = (W + a.pads[1] + a.pads[3] - a.dilations[1] * (a.kernel[1] - 1) - 1) // a.strides[1] + 1
    return oH, oW


def _check_deform_shapes(X, W, offset, B, mask, out, a, oH, oW):
    """The C ABI receives X's shape, oC and the attributes only, and trusts the
    other tensors' shapes: check them here (shapes only, no device work)."""
    N, C = X.shape[0], X.shape[1]
    oC = W.shape[0]
    K = int(a.kernel[0]) * int(a.kernel[1])
    og, grp = int(a.offset_group), int(a.group)
    if grp < 1 or C % grp:
        raise ValueError(f"group {grp} does not divide C = {C}")
    want_w = (oC, C // grp, int(a.kernel[0]), int(a.kernel[1]))
    if tuple(W.shape) != want_w:
        _shape_error("W", W.shape, want_w)
    if oH < 1 or oW < 1:
        return   # the library rejects or skips these before touching memory
    if tuple(offset.shape) != (N, og * K * 2, oH, oW):
        _shape_error("offset", offset.shape, (N, og * K * 2, oH, oW))
    if B is not None and tuple(B.shape) != (oC,):
        _shape_error("B", B.shape, (oC,))
    if mask is not None and tuple(mask.shape) != (N, og * K, oH, oW):
        _shape_error("mask", mask.shape, (N, og * K, oH, oW))
    if out is not None and tuple(out.shape) != (N, oC, oH, oW):
        _shape_error("out", out.shape, (N, oC, oH, oW))


def gs_deform_conv(X, W, offset, B=None, mask=None, kernel_shape=None, pads=None, strides=None,
                   dilations=None, group=1, offset_group=1, out=None, workspace=None):
    """DeformConv 2-D: X (N,C,H,W), W (oC,C/group,kH,kW), offset (N,og*kH*kW*2,oH,oW).

    ``workspace``: None calls gs_deform_conv; a device tensor (raw bytes) or
    "auto" (the size gs_deform_conv_workspace_size asks for, from torch's
    allocator) calls gs_deform_conv_ws."""
    torch = _torch()
    if X.dim() != 4 or W.dim() != 4:
        raise ValueError(f"X and W must be 4-D, got {tuple(X.shape)} and {tuple(W.shape)}")
    a = deform_attrs(kernel_shape if kernel_shape is not None else W.shape[2:], pads, strides,
                     dilations, group, offset_group)
    oH, oW = deform_out_hw(X.shape[2], X.shape[3], a)
    _check_deform_shapes(X, W, offset, B, mask, out, a, oH, oW)
    _check_tensors(X, W, offset, B, mask, out)
    if out is None:
        out = torch.empty((X.shape[0], W.shape[0], oH, oW), dtype=X.dtype, device=X.device)
    L = load_library()
    if workspace is None:
        _ok(L.gs_deform_conv(_ptr(X), _i64(X.shape), _ptr(W), int(W.shape[0]), _ptr(offset),
                             _ptr(B), _ptr(mask), ctypes.byref(a), _dtype_code(X), _ptr(out),
                             _stream(X)), "gs_deform_conv")
        return out
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError(f"workspace must be a tensor, None or 'auto', not {workspace!r}")
        nbytes = gs_deform_conv_workspace_size(X.shape, int(W.shape[0]), a, X.dtype)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=X.device) if nbytes else None
    if workspace is not None:
        if not workspace.is_cuda or workspace.device != X.device or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous tensor on X's device")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    else:
        ws_ptr, ws_bytes = None, 0
    _ok(L.gs_deform_conv_ws(_ptr(X), _i64(X.shape), _ptr(W), int(W.shape[0]), _ptr(offset),
                            _ptr(B), _ptr(mask), ctypes.byref(a), _dtype_code(X), ws_ptr, ws_bytes,
                            _ptr(out), _stream(X)), "gs_deform_conv_ws")
    return out


def gs_deform_conv_workspace_size(x_shape, oC, attrs, dtype):
    """Workspace bytes gs_deform_conv_ws asks for (0: the call never uses one).
    ``attrs`` is a DeformAttrs (see deform_attrs)."""
    torch = _torch()
    code = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[dtype]
    n = ctypes.c_size_t(0)
    _ok(load_library().gs_deform_conv_workspace_size(_i64(x_shape), int(oC), ctypes.byref(attrs),
                                                     code, ctypes.byref(n)),
        "gs_deform_conv_workspace_size")
    return int(n.value)


def gs_deform_conv_ws(X, W, offset, B=None, mask=None, workspace="auto", **kw):
    """gs_deform_conv with a device workspace (see gs_deform_conv_ws in gs.h)."""
    return gs_deform_conv(X, W, offset, B, mask, workspace=workspace, **kw)


def resize_attrs(mode="nearest", coordinate_transformation_mode="half_pixel",
                 nearest_mode="round_prefer_floor", cubic_coeff_a=-0.75, exclude_outside=0,
                 extrapolation_value=0.0, antialias=0, keep_aspect_ratio_policy="stretch"):
    """gs_resize_attrs from the Resize operator's attribute names (the operator's defaults)."""
    return ResizeAttrs(MODES[mode], RESIZE_COORDS[coordinate_transformation_mode],
                       RESIZE_NEAREST[nearest_mode], float(cubic_coeff_a), int(exclude_outside),
                       float(extrapolation_value), int(antialias),
                       RESIZE_KEEP[keep_aspect_ratio_policy])


def _resize_vectors(x_shape, scales, sizes, roi, axes):
    f32 = lambda v: (ctypes.c_float * len(v))(*[float(x) for x in v]) if v is not None else None
    ax = _i64(axes) if axes is not None else None
    return (ax, 0 if axes is None else len(axes), f32(None if scales is None else list(scales)),
            _i64(sizes) if sizes is not None else None, f32(None if roi is None else list(roi)))


def gs_resize_output_shape(x_shape, scales=None, sizes=None, roi=None, axes=None, **attrs):
    """Output extents of Resize (host computation in the library)."""
    at = resize_attrs(**attrs)
    ax, na, sc, sz, ro = _resize_vectors(x_shape, scales, sizes, roi, axes)
    out = (ctypes.c_int64 * len(x_shape))()
    _ok(load_library().gs_resize_output_shape(len(x_shape), _i64(x_shape), ax, na, sc, sz, ro,
                                              ctypes.byref(at), out), "gs_resize_output_shape")
    return tuple(int(v) for v in out)


def gs_resize(X, scales=None, sizes=None, roi=None, axes=None, out=None, **attrs):
    """Resize - 18 of a CUDA tensor; scales / sizes / roi / axes are host sequences and the
    attributes take the operator's names (mode, coordinate_transformation_mode,
    nearest_mode, cubic_coeff_a, exclude_outside, extrapolation_value, antialias,
    keep_aspect_ratio_policy)."""
    torch = _torch()
    _check_tensors(X, out)
    shape = gs_resize_output_shape(tuple(X.shape), scales, sizes, roi, axes, **attrs)
    if out is None:
        out = torch.empty(shape, dtype=X.dtype, device=X.device)
    elif tuple(out.shape) != shape:
        raise ValueError(f"out has shape {tuple(out.shape)}, Resize gives {shape}")
    at = resize_attrs(**attrs)
    ax, na, sc, sz, ro = _resize_vectors(X.shape, scales, sizes, roi, axes)
    _ok(load_library().gs_resize(_ptr(X), X.dim(), _i64(X.shape), ax, na, sc, sz, ro,
                                 ctypes.byref(at), _dtype_code(X), _ptr(out), _stream(X)),
        "gs_resize")
    return out


def gs_device_status(device=None):
    """Synchronise the current stream and report the library's device error word."""
    torch = _torch()
    s = torch.cuda.current_stream(device).cuda_stream
    return load_library().gs_device_status(ctypes.c_void_p(s))


class HostStreamer:
    """Run a batch whose inputs and output live in pinned host memory, chunked over
    the batch axis so the host-to-device copies of chunk i+1, the kernel on chunk
    i and the device-to-host copy of chunk i-1 overlap on three CUDA streams.

    The operators are independent per image, so chunking over N changes nothing
    in the result.  Device buffers are allocated once per shape and reused.
    """

    # With chunks=None the batch is cut into chunks of about this many input
    # bytes (whole images).  The first chunk's upload and the last chunk's
    # download overlap nothing, which favours small chunks; each chunk also
    # costs host time to enqueue, which favours large ones.
    CHUNK_BYTES = 16 << 20
    # Chunk size of the library's own pipeline (gs_affine_sample_from_host).
    # Its chunks cost little host time, yet smaller ones still lose: a chunk of
    # a few images launches too few blocks to fill the GPU.  For 64 x 32 x 128^2
    # fp32 (134 MB of X) 8 chunks measured 0.98 ms per step, 4 chunks 1.00,
    # 16 chunks 1.06, 32 chunks 1.27.
    NATIVE_CHUNK_BYTES = 16 << 20

    def __init__(self, device=None, chunks=None):
        torch = _torch()
        self.device = torch.device(device or "cuda")
        self.chunks = None if chunks is None else int(chunks)
        self.s_in = torch.cuda.Stream(self.device)
        self.s_run = torch.cuda.Stream(self.device)
        self.s_out = torch.cuda.Stream(self.device)
        self._dev = {}

    def _buffers(self, key, shapes, dtype):
        torch = _torch()
        if key not in self._dev:
            self._dev[key] = [torch.empty(s, dtype=dtype, device=self.device) for s in shapes]
        return self._dev[key]

    def run(self, fn, inputs, out_host, batch_axes):
        """fn(*device_chunks, out=device_out_chunk) on chunks along each input's batch axis
        (batch_axes[i] is None for inputs passed whole); out_host is filled in place."""
        torch = _torch()
        N = out_host.shape[0]
        chunks = self.chunks
        if chunks is None:
            in_bytes = sum(t.numel() * t.element_size() for t, ax in zip(inputs, batch_axes)
                           if ax is not None)
            chunks = max(1, min(N, in_bytes // self.CHUNK_BYTES))
        step = max(1, -(-N // chunks))
        key = (tuple((tuple(t.shape), t.dtype) for t in inputs), tuple(out_host.shape),
               out_host.dtype)
        dev = self._buffers(key, [t.shape for t in inputs] + [out_host.shape], out_host.dtype)
        d_in, d_out = dev[:-1], dev[-1]
        cur = torch.cuda.current_stream(self.device)
        for s in (self.s_in, self.s_run, self.s_out):
            s.wait_stream(cur)
        for n0 in range(0, N, step):
            n1 = min(N, n0 + step)
            with torch.cuda.stream(self.s_in):
                parts = []
                for t, d, ax in zip(inputs, d_in, batch_axes):
                    if ax is None:
                        if n0 == 0:
                            d.copy_(t, non_blocking=True)
                        parts.append(d)
                    else:
                        d[n0:n1].copy_(t[n0:n1], non_blocking=True)
                        parts.append(d[n0:n1])
                ev_in = torch.cuda.Event()
                ev_in.record(self.s_in)
            with torch.cuda.stream(self.s_run):
                self.s_run.wait_event(ev_in)
                fn(*parts, out=d_out[n0:n1])
                ev_run = torch.cuda.Event()
                ev_run.record(self.s_run)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(ev_run)
                out_host[n0:n1].copy_(d_out[n0:n1], non_blocking=True)
        for s in (self.s_in, self.s_run, self.s_out):
            cur.wait_stream(s)
        return out_host


def gs_affine_sample_from_host(theta, size, X, mode="linear", padding_mode="zeros",
                               align_corners=0, cubic_coeff_a=-0.75, out=None, streamer=None):
    """gs_affine_sample with theta, X and the output in (pinned) host memory,
    copies overlapped with the kernels; returns the host output, complete once the
    current CUDA stream reaches this point (synchronize before reading it).

    The chunked pipeline runs inside the library (gs_affine_sample_from_host in
    gs.h) on the streamer's three streams and device buffers."""
    torch = _torch()
    size = [int(s) for s in size]
    if out is None:
        out = torch.empty(list(X.shape[:2]) + size[2:], dtype=X.dtype).pin_memory()
    for t in (theta, X, out):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("gs_affine_sample_from_host takes contiguous host tensors")
    if not (theta.dtype == X.dtype == out.dtype):
        raise TypeError("theta, X and out must share one dtype")
    st = streamer or HostStreamer()
    N = X.shape[0]
    chunks = st.chunks
    if chunks is None:
        chunks = max(1, min(N, (X.numel() * X.element_size()) // st.NATIVE_CHUNK_BYTES))
    key = ("affine_from_host", tuple(theta.shape), tuple(X.shape), tuple(out.shape), X.dtype)
    d_th, d_x, d_y = st._buffers(key, [theta.shape, X.shape, out.shape], X.dtype)
    cur = torch.cuda.current_stream(st.device)
    for s in (st.s_in, st.s_run, st.s_out):
        s.wait_stream(cur)
    streams = (ctypes.c_void_p * 3)(st.s_in.cuda_stream, st.s_run.cuda_stream,
                                    st.s_out.cuda_stream)
    _ok(load_library().gs_affine_sample_from_host(
        ctypes.c_void_p(theta.data_ptr()), _i64(size), X.dim() - 2,
        ctypes.c_void_p(X.data_ptr()), _i64(X.shape), _dtype_code(X), MODES[mode],
        PADS[padding_mode], int(align_corners), float(cubic_coeff_a),
        ctypes.c_void_p(out.data_ptr()), _ptr(d_th), _ptr(d_x), _ptr(d_y), int(chunks), streams),
        "gs_affine_sample_from_host")
    for s in (st.s_in, st.s_run, st.s_out):
        cur.wait_stream(s)
    return out


def gs_grid_sample_from_host(X, grid, mode="linear", padding_mode="zeros", align_corners=0,
                             cubic_coeff_a=-0.75, out=None, streamer=None, workspace=None):
    """gs_grid_sample with X, grid and the output in (pinned) host memory, copies
    overlapped with the kernels; returns the host output, complete once the current
    CUDA stream reaches this point (synchronize before reading it).  ``workspace``
    as in gs_grid_sample ("auto" keeps one per streamer and chunk shape)."""
    torch = _torch()
    if out is None:
        out = torch.empty(list(X.shape[:2]) + list(grid.shape[1:-1]), dtype=X.dtype).pin_memory()
    st = streamer or HostStreamer()

    def fn(x, g, out):
        ws = workspace
        if isinstance(ws, str) and ws == "auto":
            nbytes = gs_grid_sample_workspace_size(x.shape, g.shape[1:-1], x.dtype)
            ws = st._buffers(("workspace", nbytes), [(nbytes,)], torch.uint8)[0] if nbytes else None
            if ws is None:
                return gs_grid_sample(x, g, mode, padding_mode, align_corners, cubic_coeff_a,
                                      out=out)
        return gs_grid_sample(x, g, mode, padding_mode, align_corners, cubic_coeff_a, out=out,
                              workspace=ws)
    return st.run(fn, [X, grid], out, [0, 0])
