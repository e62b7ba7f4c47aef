"""DeformConv on the GPU against the oracle, element by element on seeded inputs,
plus the page's worked examples and the full-size workload on sampled outputs."""
import itertools

import numpy as np
import pytest
import torch

from conftest import assert_parity, fixture_array, fixture_names, load_fixture, page_close
from spatial_transformer_sampling_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def exact(t):
    return wl.widened(t)


@pytest.mark.parametrize("name", fixture_names("deformconv__"))
def test_page_examples_deform_conv(gs_cuda, oracle_mod, name):
    fx = load_fixture(name)
    a = fx["attributes"]
    ins = {k: fixture_array(v) for k, v in fx["inputs"].items()}
    kw = dict(kernel_shape=a.get("kernel_shape"), pads=a.get("pads"),
              offset_group=a.get("offset_group", 1))
    cu = {k: wl.as_dtype(v, "float32").cuda() for k, v in ins.items()}
    Y = gs_cuda.gs_deform_conv(cu["X"], cu["W"], cu["offset"], cu.get("B"), cu.get("mask"), **kw)
    ref = oracle_mod.deform_conv(ins["X"], ins["W"], ins["offset"], ins.get("B"), ins.get("mask"),
                                 **kw)
    assert_parity(Y, ref, "float32", fx["citation"])
    assert page_close(exact(Y), fixture_array(fx["outputs"]["Y"])).all(), fx["citation"]


CASES = [
    # N, C, H, W, oC, kernel, pads, strides, dilations, group, og, bias, mask
    (2, 8, 13, 11, 6, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), 1, 1, True, True),
    (1, 6, 9, 14, 4, (3, 2), (0, 1, 2, 0), (2, 1), (1, 2), 2, 1, False, True),
    (2, 8, 10, 10, 8, (2, 2), (1, 0, 0, 1), (1, 2), (2, 1), 1, 2, True, False),
    (1, 12, 11, 9, 6, (3, 3), (2, 2, 2, 2), (2, 2), (2, 2), 3, 4, True, True),
    (1, 40, 9, 17, 70, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), 1, 1, True, True),   # 2 oc blocks, ragged chunks
    (1, 64, 12, 12, 16, (1, 1), (0, 0, 0, 0), (1, 1), (1, 1), 1, 64, False, True),   # 1 channel per offset group
    (3, 4, 5, 31, 3, (5, 3), (2, 1, 2, 1), (1, 3), (1, 1), 1, 1, True, False),
]


@pytest.mark.parametrize("case,dtype", list(itertools.product(range(len(CASES)),
                                                              ["float32", "float16", "bfloat16"])))
def test_deform_conv_cases(gs_cuda, oracle_mod, case, dtype):
    N, C, H, W, oC, k, p, s, d, grp, og, has_b, has_m = CASES[case]
    g = wl.rng(300 + case)
    oH = (H + p[0] + p[2] - d[0] * (k[0] - 1) - 1) // s[0] + 1
    oW = (W + p[1] + p[3] - d[1] * (k[1] - 1) - 1) // s[1] + 1
    K = k[0] * k[1]
    host = {
        "X": wl.as_dtype(g.normal(size=(N, C, H, W)), dtype),
        "W": wl.as_dtype(g.normal(0, 0.3, size=(oC, C // grp) + k), dtype),
        "offset": wl.as_dtype(g.normal(0, 1.5, size=(N, og * K * 2, oH, oW)), dtype),
        "B": wl.as_dtype(g.normal(size=(oC,)), dtype) if has_b else None,
        "mask": wl.as_dtype(g.uniform(0, 1, size=(N, og * K, oH, oW)), dtype) if has_m else None,
    }
    kw = dict(kernel_shape=k, pads=p, strides=s, dilations=d, group=grp, offset_group=og)
    cu = {n: (t.cuda() if t is not None else None) for n, t in host.items()}
    Y = gs_cuda.gs_deform_conv(cu["X"], cu["W"], cu["offset"], cu["B"], cu["mask"], **kw)
    ref = oracle_mod.deform_conv(*[exact(host[n]) if host[n] is not None else None
                                   for n in ("X", "W", "offset", "B", "mask")], **kw)
    assert_parity(Y, ref, dtype, f"deform case {case} {dtype}")


def test_deform_conv_zero_batch_and_channels(gs_cuda):
    X = torch.zeros((0, 4, 8, 8), device="cuda")
    W = torch.zeros((5, 4, 3, 3), device="cuda")
    off = torch.zeros((0, 18, 8, 8), device="cuda")
    assert gs_cuda.gs_deform_conv(X, W, off, pads=(1, 1, 1, 1)).shape == (0, 5, 8, 8)


@pytest.mark.parametrize("dtype", ["float32", "bfloat16"])
def test_full_size_deform2d(gs_cuda, oracle_mod, dtype):
    w = wl.WORKLOADS["deform2d"]
    inp = wl.make_deform_inputs(w)
    host = {k: wl.as_dtype(v, dtype) for k, v in inp.items()}
    cu = {k: v.cuda() for k, v in host.items()}
    kw = dict(kernel_shape=w.kernel, pads=w.pads, strides=w.strides, dilations=w.dilations,
              group=w.group, offset_group=w.offset_group)
    Y = gs_cuda.gs_deform_conv(cu["X"], cu["W"], cu["offset"], cu["B"], cu["mask"], **kw)
    torch.cuda.synchronize()
    g = wl.rng(5)
    idx = np.unique(np.concatenate([g.integers(0, Y.numel(), 20000), [0, Y.numel() - 1]]))
    ref = oracle_mod.deform_conv_at(exact(host["X"]), exact(host["W"]), exact(host["offset"]), idx,
                                    exact(host["B"]), exact(host["mask"]), **kw)
    assert_parity(Y.reshape(-1)[torch.from_numpy(idx).cuda()], ref, dtype, "deform2d sampled")


# shapes the tensor-core kernel takes (group = offset_group = 1, C and oC multiples of 16)
TC_CASES = [
    # N, C, H, W, oC, kernel, pads, strides, dilations, bias, mask
    (2, 32, 13, 11, 16, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), True, True),     # ragged last tile
    (1, 48, 9, 17, 32, (3, 2), (0, 1, 2, 0), (2, 1), (1, 2), False, True),    # 16-channel chunks
    (1, 128, 12, 12, 48, (1, 1), (0, 0, 0, 0), (1, 1), (1, 1), True, False),  # 64-channel chunks
    (1, 64, 16, 16, 128, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), True, True),   # N = 128
    (3, 96, 7, 9, 64, (2, 2), (1, 0, 0, 1), (1, 1), (2, 1), True, True),      # 32-channel chunks
]


@pytest.mark.parametrize("case,dtype", list(itertools.product(range(len(TC_CASES)),
                                                              ["float16", "bfloat16"])))
def test_deform_conv_tensor_core_shapes(gs_cuda, oracle_mod, case, dtype):
    N, C, H, W, oC, k, p, s, d, has_b, has_m = TC_CASES[case]
    g = wl.rng(500 + case)
    oH = (H + p[0] + p[2] - d[0] * (k[0] - 1) - 1) // s[0] + 1
    oW = (W + p[1] + p[3] - d[1] * (k[1] - 1) - 1) // s[1] + 1
    K = k[0] * k[1]
    host = {
        "X": wl.as_dtype(g.normal(size=(N, C, H, W)), dtype),
        "W": wl.as_dtype(g.normal(0, 0.05, size=(oC, C) + k), dtype),
        "offset": wl.as_dtype(g.normal(0, 1.0, size=(N, K * 2, oH, oW)), dtype),
        "B": wl.as_dtype(g.normal(size=(oC,)), dtype) if has_b else None,
        "mask": wl.as_dtype(g.uniform(0, 1, size=(N, K, oH, oW)), dtype) if has_m else None,
    }
    kw = dict(kernel_shape=k, pads=p, strides=s, dilations=d)
    cu = {n: (t.cuda() if t is not None else None) for n, t in host.items()}
    Y = gs_cuda.gs_deform_conv(cu["X"], cu["W"], cu["offset"], cu["B"], cu["mask"], **kw)
    assert gs_cuda.gs_device_status() == 0
    ref = oracle_mod.deform_conv(*[exact(host[n]) if host[n] is not None else None
                                   for n in ("X", "W", "offset", "B", "mask")], **kw)
    assert_parity(Y, ref, dtype, f"deform tc case {case} {dtype}")


# ------------------------------------------------ channel-last workspace path

@pytest.mark.parametrize("case,dtype", list(itertools.product(range(len(TC_CASES)),
                                                              ["float16", "bfloat16"])))
def test_deform_conv_workspace_matches(gs_cuda, oracle_mod, case, dtype):
    """gs_deform_conv_ws: the same values as gs_deform_conv (same weights, same
    order of accumulation), and the oracle's within the tolerance."""
    N, C, H, W, oC, k, p, s, d, has_b, has_m = TC_CASES[case]
    g = wl.rng(700 + case)
    oH = (H + p[0] + p[2] - d[0] * (k[0] - 1) - 1) // s[0] + 1
    oW = (W + p[1] + p[3] - d[1] * (k[1] - 1) - 1) // s[1] + 1
    K = k[0] * k[1]
    host = {
        "X": wl.as_dtype(g.normal(size=(N, C, H, W)), dtype),
        "W": wl.as_dtype(g.normal(0, 0.05, size=(oC, C) + k), dtype),
        "offset": wl.as_dtype(g.normal(0, 2.0, size=(N, K * 2, oH, oW)), dtype),
        "B": wl.as_dtype(g.normal(size=(oC,)), dtype) if has_b else None,
        "mask": wl.as_dtype(g.uniform(0, 1, size=(N, K, oH, oW)), dtype) if has_m else None,
    }
    kw = dict(kernel_shape=k, pads=p, strides=s, dilations=d)
    cu = {n: (t.cuda() if t is not None else None) for n, t in host.items()}
    args = (cu["X"], cu["W"], cu["offset"], cu["B"], cu["mask"])
    assert gs_cuda.gs_deform_conv_workspace_size(
        host["X"].shape, oC, gs_cuda.deform_attrs(k, p, s, d), getattr(torch, dtype)) > 0
    Yw = gs_cuda.gs_deform_conv(*args, workspace="auto", **kw)
    Y0 = gs_cuda.gs_deform_conv(*args, **kw)
    assert gs_cuda.gs_device_status() == 0
    assert torch.equal(Yw, Y0)
    ref = oracle_mod.deform_conv(*[exact(host[n]) if host[n] is not None else None
                                   for n in ("X", "W", "offset", "B", "mask")], **kw)
    assert_parity(Yw, ref, dtype, f"deform ws case {case} {dtype}")


@pytest.mark.parametrize("slots", [1, 2])
def test_deform_conv_workspace_chunks(gs_cuda, slots):
    """A workspace with room for W and fewer image slots than N runs image chunks."""
    g = wl.rng(720 + slots)
    N, C, H, W, oC = 3, 32, 11, 13, 16
    X = wl.as_dtype(g.normal(size=(N, C, H, W)), "bfloat16").cuda()
    Wt = wl.as_dtype(g.normal(0, 0.05, size=(oC, C, 3, 3)), "bfloat16").cuda()
    off = wl.as_dtype(g.normal(0, 1.5, size=(N, 18, H, W)), "bfloat16").cuda()
    a = gs_cuda.deform_attrs((3, 3), (1, 1, 1, 1))
    full = gs_cuda.gs_deform_conv_workspace_size(X.shape, oC, a, torch.bfloat16)
    slot = C * (H * W + 1) * 2
    ws = torch.empty(full - (N - slots) * slot, dtype=torch.uint8, device="cuda")
    Yw = gs_cuda.gs_deform_conv(X, Wt, off, pads=(1, 1, 1, 1), workspace=ws)
    assert torch.equal(Yw, gs_cuda.gs_deform_conv(X, Wt, off, pads=(1, 1, 1, 1)))


def test_deform_conv_workspace_falls_back(gs_cuda):
    """fp32, grouped shapes and a workspace short of W plus one slot run gs_deform_conv."""
    g = wl.rng(730)
    X = torch.from_numpy(g.normal(size=(2, 16, 9, 9)).astype(np.float32)).cuda()
    Wt = torch.from_numpy(g.normal(0, 0.1, size=(16, 16, 3, 3)).astype(np.float32)).cuda()
    off = torch.from_numpy(g.normal(0, 1, size=(2, 18, 9, 9)).astype(np.float32)).cuda()
    a = gs_cuda.deform_attrs((3, 3), (1, 1, 1, 1))
    assert gs_cuda.gs_deform_conv_workspace_size(X.shape, 16, a, torch.float32) == 0
    assert torch.equal(gs_cuda.gs_deform_conv(X, Wt, off, pads=(1, 1, 1, 1), workspace="auto"),
                       gs_cuda.gs_deform_conv(X, Wt, off, pads=(1, 1, 1, 1)))
    Xh, Wh, oh = X.bfloat16(), Wt.bfloat16(), off.bfloat16()
    small = torch.empty(16 * 16 * 9 * 2, dtype=torch.uint8, device="cuda")   # W only
    assert torch.equal(gs_cuda.gs_deform_conv(Xh, Wh, oh, pads=(1, 1, 1, 1), workspace=small),
                       gs_cuda.gs_deform_conv(Xh, Wh, oh, pads=(1, 1, 1, 1)))
    Wg = Wh[:, :8].contiguous()                                             # group = 2
    assert gs_cuda.gs_deform_conv_workspace_size(Xh.shape, 16, gs_cuda.deform_attrs(
        (3, 3), (1, 1, 1, 1), group=2), torch.bfloat16) == 0
    assert torch.equal(gs_cuda.gs_deform_conv(Xh, Wg, oh, pads=(1, 1, 1, 1), group=2,
                                              workspace="auto"),
                       gs_cuda.gs_deform_conv(Xh, Wg, oh, pads=(1, 1, 1, 1), group=2))


def test_full_size_deform2d_workspace(gs_cuda, oracle_mod):
    w = wl.WORKLOADS["deform2d"]
    inp = wl.make_deform_inputs(w)
    host = {k: wl.as_dtype(v, "bfloat16") for k, v in inp.items()}
    cu = {k: v.cuda() for k, v in host.items()}
    kw = dict(kernel_shape=w.kernel, pads=w.pads, strides=w.strides, dilations=w.dilations,
              group=w.group, offset_group=w.offset_group)
    args = (cu["X"], cu["W"], cu["offset"], cu["B"], cu["mask"])
    Y = gs_cuda.gs_deform_conv(*args, workspace="auto", **kw)
    torch.cuda.synchronize()
    assert torch.equal(Y, gs_cuda.gs_deform_conv(*args, **kw))
    g = wl.rng(6)
    idx = np.unique(np.concatenate([g.integers(0, Y.numel(), 20000), [0, Y.numel() - 1]]))
    ref = oracle_mod.deform_conv_at(exact(host["X"]), exact(host["W"]), exact(host["offset"]), idx,
                                    exact(host["B"]), exact(host["mask"]), **kw)
    assert_parity(Y.reshape(-1)[torch.from_numpy(idx).cuda()], ref, "bfloat16",
                  "deform2d with workspace, sampled")


# ---------------------------------- staged persistent tensor-core kernel
#
# Shapes the staged kernel takes (group = offset_group = 1, C % 16 == 0,
# W % 8 == 0, oH*oW % 8 == 0, kH*kW in {1, 2, 3, 4, 6, 9}): one or several
# 16-channel chunks, tiles spanning 1 to 4 output rows and a ragged last tile,
# stride and dilation, no bias / no mask, large offsets whose taps leave the
# staged window (read from global memory), and enough tiles that CTAs take
# more than one.
STAGED_CASES = [
    # N, C, H, W, oC, kernel, pads, strides, dilations, bias, mask, offset sigma
    (2, 64, 24, 32, 64, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), True, True, 1.0),   # 4 rows per tile
    (1, 16, 10, 128, 16, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), True, True, 1.0),  # 1 row per tile
    (1, 48, 20, 40, 48, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), False, True, 1.0),  # ragged last tile
    (2, 32, 16, 16, 32, (1, 1), (0, 0, 0, 0), (1, 1), (1, 1), True, False, 1.0),  # K = 1
    (1, 32, 33, 48, 16, (2, 2), (1, 0, 0, 1), (2, 2), (2, 1), True, True, 1.0),   # K = 4, stride, dil
    (1, 16, 20, 24, 256, (3, 2), (1, 1, 1, 0), (1, 2), (1, 1), True, True, 1.0),  # K = 6, oC = 256
    (2, 32, 32, 32, 32, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), True, True, 6.0),   # taps leave the window
    (10, 16, 64, 64, 16, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), True, True, 1.0),  # 320 tiles
    (1, 16, 8, 8, 32, (1, 3), (0, 1, 0, 1), (1, 1), (1, 1), False, False, 0.7),   # K = 3, one tile
    (1, 32, 12, 16, 16, (2, 1), (0, 0, 1, 0), (1, 1), (1, 1), True, True, 1.0),   # K = 2
]


def _staged_inputs(case, dtype, seed):
    N, C, H, W, oC, k, p, s, d, has_b, has_m, sig = STAGED_CASES[case]
    g = wl.rng(seed)
    oH = (H + p[0] + p[2] - d[0] * (k[0] - 1) - 1) // s[0] + 1
    oW = (W + p[1] + p[3] - d[1] * (k[1] - 1) - 1) // s[1] + 1
    K = k[0] * k[1]
    host = {
        "X": wl.as_dtype(g.normal(size=(N, C, H, W)), dtype),
        "W": wl.as_dtype(g.normal(0, 0.05, size=(oC, C) + k), dtype),
        "offset": wl.as_dtype(g.normal(0, sig, size=(N, K * 2, oH, oW)), dtype),
        "B": wl.as_dtype(g.normal(size=(oC,)), dtype) if has_b else None,
        "mask": wl.as_dtype(1.0 / (1.0 + np.exp(-g.normal(size=(N, K, oH, oW)))), dtype)
        if has_m else None,
    }
    return host, dict(kernel_shape=k, pads=p, strides=s, dilations=d)


@pytest.mark.parametrize("case,dtype", list(itertools.product(range(len(STAGED_CASES)),
                                                              ["float16", "bfloat16"])))
def test_deform_conv_staged_shapes(gs_cuda, oracle_mod, case, dtype):
    host, kw = _staged_inputs(case, dtype, 800 + case)
    cu = {n: (t.cuda() if t is not None else None) for n, t in host.items()}
    args = (cu["X"], cu["W"], cu["offset"], cu["B"], cu["mask"])
    a = gs_cuda.deform_attrs(kw["kernel_shape"], kw["pads"], kw["strides"], kw["dilations"])
    # the staged kernel takes these shapes and needs no workspace
    assert gs_cuda.gs_deform_conv_workspace_size(host["X"].shape, host["W"].shape[0], a,
                                                 getattr(torch, dtype)) == 0
    Y = gs_cuda.gs_deform_conv(*args, **kw)
    assert gs_cuda.gs_device_status() == 0
    ref = oracle_mod.deform_conv(*[exact(host[n]) if host[n] is not None else None
                                   for n in ("X", "W", "offset", "B", "mask")], **kw)
    assert_parity(Y, ref, dtype, f"deform staged case {case} {dtype}")
    # the same call twice gives the same bits, and so does the workspace entry
    assert torch.equal(Y, gs_cuda.gs_deform_conv(*args, **kw))
    assert torch.equal(Y, gs_cuda.gs_deform_conv(*args, workspace="auto", **kw))


def test_deform_conv_staged_matches_unaligned_fallback(gs_cuda, oracle_mod):
    """A tensor off the 16-byte alignment the staged kernel wants runs the
    previous tensor-core kernel; both agree with the oracle."""
    host, kw = _staged_inputs(0, "bfloat16", 850)
    cu = {n: (t.cuda() if t is not None else None) for n, t in host.items()}
    Y = gs_cuda.gs_deform_conv(cu["X"], cu["W"], cu["offset"], cu["B"], cu["mask"], **kw)
    buf = torch.empty(cu["X"].numel() + 1, dtype=torch.bfloat16, device="cuda")
    Xu = buf[1:].view(cu["X"].shape)          # 2 bytes past a 16-byte boundary
    Xu.copy_(cu["X"])
    Yu = gs_cuda.gs_deform_conv(Xu, cu["W"], cu["offset"], cu["B"], cu["mask"], **kw)
    assert gs_cuda.gs_device_status() == 0
    ref = oracle_mod.deform_conv(*[exact(host[n]) for n in ("X", "W", "offset", "B", "mask")],
                                 **kw)
    assert_parity(Y, ref, "bfloat16", "staged")
    assert_parity(Yu, ref, "bfloat16", "unaligned X, previous kernel")


# ------------------------------------------------ fp32 windowed kernel

# shapes the fp32 windowed kernel takes (W % 4 == 0, channels per group and
# per offset group multiples of 8, kH kW <= 9)
F32_CASES = [
    # N, C, H, W, oC, kernel, pads, strides, dilations, group, og, bias, mask, offset sigma
    (2, 16, 24, 32, 64, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), 1, 1, True, True, 1.0),    # 4 rows/tile
    (1, 24, 10, 128, 40, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), 1, 1, True, True, 1.0),   # 1 row/tile
    (1, 16, 20, 40, 130, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), 1, 1, False, True, 1.0),  # ragged, 3 oc blocks
    (2, 32, 16, 16, 32, (1, 1), (0, 0, 0, 0), (1, 1), (1, 1), 1, 1, True, False, 1.0),   # K = 1
    (1, 16, 33, 48, 16, (2, 2), (1, 0, 0, 1), (2, 2), (2, 1), 1, 1, True, True, 1.0),    # stride, dilation
    (1, 32, 20, 24, 24, (3, 2), (1, 1, 1, 0), (1, 2), (1, 1), 2, 1, True, True, 1.0),    # 2 groups
    (2, 32, 16, 16, 32, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), 1, 4, True, True, 1.0),    # 4 offset groups
    (2, 16, 32, 32, 16, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), 1, 1, True, True, 6.0),    # taps leave the window
    (1, 8, 8, 8, 8, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), 1, 1, False, False, 0.7),      # one partial tile
    (1, 16, 7, 4, 8, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), 1, 1, True, True, 1.0),       # 4 columns
    (1, 16, 12, 256, 16, (3, 3), (1, 1, 1, 1), (1, 1), (1, 1), 1, 1, True, True, 1.0),   # wide rows
    (1, 16, 9, 8, 16, (3, 3), (0, 0, 0, 0), (1, 1), (3, 3), 1, 1, True, True, 1.0),      # dilation 3
]


def _f32_inputs(case, seed):
    N, C, H, W, oC, k, p, s, d, grp, og, has_b, has_m, sig = F32_CASES[case]
    g = wl.rng(seed)
    oH = (H + p[0] + p[2] - d[0] * (k[0] - 1) - 1) // s[0] + 1
    oW = (W + p[1] + p[3] - d[1] * (k[1] - 1) - 1) // s[1] + 1
    K = k[0] * k[1]
    host = {
        "X": wl.as_dtype(g.normal(size=(N, C, H, W)), "float32"),
        "W": wl.as_dtype(g.normal(0, 0.05, size=(oC, C // grp) + k), "float32"),
        "offset": wl.as_dtype(g.normal(0, sig, size=(N, og * K * 2, oH, oW)), "float32"),
        "B": wl.as_dtype(g.normal(size=(oC,)), "float32") if has_b else None,
        "mask": wl.as_dtype(1.0 / (1.0 + np.exp(-g.normal(size=(N, og * K, oH, oW)))), "float32")
        if has_m else None,
    }
    return host, dict(kernel_shape=k, pads=p, strides=s, dilations=d, group=grp, offset_group=og)


@pytest.mark.parametrize("case", range(len(F32_CASES)))
def test_deform_conv_f32_window_shapes(gs_cuda, oracle_mod, case):
    host, kw = _f32_inputs(case, 900 + case)
    cu = {n: (t.cuda() if t is not None else None) for n, t in host.items()}
    args = (cu["X"], cu["W"], cu["offset"], cu["B"], cu["mask"])
    Y = gs_cuda.gs_deform_conv(*args, **kw)
    assert gs_cuda.gs_device_status() == 0
    ref = oracle_mod.deform_conv(*[exact(host[n]) if host[n] is not None else None
                                   for n in ("X", "W", "offset", "B", "mask")], **kw)
    assert_parity(Y, ref, "float32", f"deform fp32 window case {case}")
    assert torch.equal(Y, gs_cuda.gs_deform_conv(*args, **kw))


def test_deform_conv_f32_window_matches_unaligned_fallback(gs_cuda, oracle_mod):
    """X off the 16-byte alignment the windowed kernel copies with runs the
    general fp32 kernel; both agree with the oracle and with each other."""
    host, kw = _f32_inputs(0, 950)
    cu = {n: (t.cuda() if t is not None else None) for n, t in host.items()}
    Y = gs_cuda.gs_deform_conv(cu["X"], cu["W"], cu["offset"], cu["B"], cu["mask"], **kw)
    buf = torch.empty(cu["X"].numel() + 1, dtype=torch.float32, device="cuda")
    Xu = buf[1:].view(cu["X"].shape)          # 4 bytes past a 16-byte boundary
    Xu.copy_(cu["X"])
    Yu = gs_cuda.gs_deform_conv(Xu, cu["W"], cu["offset"], cu["B"], cu["mask"], **kw)
    assert gs_cuda.gs_device_status() == 0
    ref = oracle_mod.deform_conv(*[exact(host[n]) for n in ("X", "W", "offset", "B", "mask")],
                                 **kw)
    assert_parity(Y, ref, "float32", "windowed")
    assert_parity(Yu, ref, "float32", "unaligned X, general kernel")
    assert_parity(Y, exact(Yu), "float32", "windowed against general")


def test_deform_conv_f32_nonfinite_offsets(gs_cuda, oracle_mod):
    """Offsets that are NaN, infinite or huge give zero samples, as the general
    kernel and the oracle take them."""
    host, kw = _f32_inputs(0, 960)
    off = host["offset"].clone()
    off.view(-1)[::97] = float("nan")
    off.view(-1)[5::101] = float("inf")
    off.view(-1)[9::89] = -3.0e9
    host["offset"] = off
    cu = {n: (t.cuda() if t is not None else None) for n, t in host.items()}
    Y = gs_cuda.gs_deform_conv(cu["X"], cu["W"], cu["offset"], cu["B"], cu["mask"], **kw)
    assert gs_cuda.gs_device_status() == 0
    ref = oracle_mod.deform_conv(*[exact(host[n]) for n in ("X", "W", "offset", "B", "mask")],
                                 **kw)
    assert_parity(Y, ref, "float32", "non-finite offsets")


def test_deform_conv_f32_window_unaligned_output(gs_cuda, oracle_mod):
    """Y four bytes off a 16-byte boundary takes the windowed kernel's scalar
    stores: the same bits as the vector stores, and the oracle's values."""
    host, kw = _f32_inputs(2, 970)   # 20 x 40 output, 130 output channels
    cu = {n: (t.cuda() if t is not None else None) for n, t in host.items()}
    args = (cu["X"], cu["W"], cu["offset"], cu["B"], cu["mask"])
    Y = gs_cuda.gs_deform_conv(*args, **kw)
    buf = torch.empty(Y.numel() + 1, dtype=torch.float32, device="cuda")
    Yu = buf[1:].view(Y.shape)
    gs_cuda.gs_deform_conv(*args, out=Yu, **kw)
    assert gs_cuda.gs_device_status() == 0
    assert torch.equal(Y, Yu)
    ref = oracle_mod.deform_conv(*[exact(host[n]) if host[n] is not None else None
                                   for n in ("X", "W", "offset", "B", "mask")], **kw)
    assert_parity(Yu, ref, "float32", "unaligned Y")
