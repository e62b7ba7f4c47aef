"""Seeded synthetic inputs for the sampling path (shapes, distributions, seeds).

This module draws random inputs and nothing else: it holds none of the
method's arithmetic, and both the CUDA-path tests and the oracle-side tests
take their inputs from it.  Values are drawn in float64 with numpy's PCG64 and
returned as float64 arrays; callers round them to the I/O dtype (see
``as_dtype``) and hand the rounded values, widened back to float64 exactly,
to the oracle.

Workloads (the operator pages give no benchmark; these are the synthetic
stand-ins, one seed per workload, ``1000 + index``):

  0 gs2d_small   GridSample 2-D, linear, zeros, align_corners=0, fp32:
                 X (1,3,32,32) ~ U(-1,1), grid (1,24,24,2) ~ U(-1.2,1.2).
  1 stn2d        AffineGrid fused into GridSample 2-D (spatial transformer):
                 theta (64,2,3) = [[1,0,0],[0,1,0]] + N(0, 0.1) on every entry,
                 X (64,32,128,128) ~ N(0,1), output 128x128, linear, border,
                 align_corners=1; fp32 and bf16.
  2 gs2d_cubic   GridSample 2-D, cubic (a = -0.75) and nearest, reflection,
                 align_corners=0: X (16,64,256,256) ~ N(0,1), grid
                 (16,256,256,2) ~ U(-1.5,1.5); fp32 and fp16.
  3 stn3d        AffineGrid fused into GridSample 3-D, linear, zeros,
                 align_corners=0: theta (4,3,4) = identity(3x4) + N(0, 0.1),
                 X (4,16,64,64,64) ~ N(0,1), output 64^3; fp32.
  4 deform2d     DeformConv 2-D: X (8,64,64,64) ~ N(0,1), W (64,64,3,3) ~
                 N(0, 0.05), B (64) ~ N(0,1), pads 1, stride 1, group 1,
                 offset_group 1, offset (8,18,64,64) ~ N(0,1),
                 mask (8,9,64,64) = sigmoid(N(0,1)); fp32 and bf16.
  5 resize2d_up  Resize (on the same separable sampler), 2x bilinear upscale,
                 half_pixel: X (16,64,128,128) ~ N(0,1), scales (1,1,2,2);
                 fp32 and bf16.
  6 resize2d_aa  Resize, antialiased bilinear 2x downscale, half_pixel:
                 X (16,64,256,256) ~ N(0,1), scales (1,1,0.5,0.5); fp32.

The second argument of N(., .) is the standard deviation.
"""
from dataclasses import dataclass, field

import numpy as np

WORKLOADS = {}


@dataclass
class Workload:
    index: int
    name: str
    kind: str                      # "grid_sample" | "affine_sample" | "deform_conv" | "resize"
    r: int
    x_shape: tuple
    out_spatial: tuple = ()
    mode: str = "linear"
    padding_mode: str = "zeros"
    align_corners: int = 0
    cubic_coeff_a: float = -0.75
    dtypes: tuple = ("float32",)
    x_dist: tuple = ("normal", 0.0, 1.0)
    grid_dist: tuple = ("uniform", -1.0, 1.0)
    theta_noise: float = 0.1
    # deform conv
    oc: int = 0
    kernel: tuple = (3, 3)
    pads: tuple = (1, 1, 1, 1)
    strides: tuple = (1, 1)
    dilations: tuple = (1, 1)
    group: int = 1
    offset_group: int = 1
    extra: dict = field(default_factory=dict)

    @property
    def seed(self):
        return 1000 + self.index


def _reg(w):
    WORKLOADS[w.name] = w
    return w


_reg(Workload(0, "gs2d_small", "grid_sample", 2, (1, 3, 32, 32), (24, 24),
              x_dist=("uniform", -1.0, 1.0), grid_dist=("uniform", -1.2, 1.2)))
_reg(Workload(1, "stn2d", "affine_sample", 2, (64, 32, 128, 128), (128, 128),
              padding_mode="border", align_corners=1, dtypes=("float32", "bfloat16")))
_reg(Workload(2, "gs2d_cubic", "grid_sample", 2, (16, 64, 256, 256), (256, 256), mode="cubic",
              padding_mode="reflection", dtypes=("float32", "float16"),
              grid_dist=("uniform", -1.5, 1.5), extra={"modes": ("cubic", "nearest")}))
_reg(Workload(3, "stn3d", "affine_sample", 3, (4, 16, 64, 64, 64), (64, 64, 64)))
_reg(Workload(4, "deform2d", "deform_conv", 2, (8, 64, 64, 64), oc=64,
              dtypes=("float32", "bfloat16")))
_reg(Workload(5, "resize2d_up", "resize", 2, (16, 64, 128, 128), (256, 256),
              dtypes=("float32", "bfloat16"), extra={"scales": (1.0, 1.0, 2.0, 2.0), "antialias": 0}))
_reg(Workload(6, "resize2d_aa", "resize", 2, (16, 64, 256, 256), (128, 128),
              extra={"scales": (1.0, 1.0, 0.5, 0.5), "antialias": 1}))


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def draw(g, dist, shape):
    kind = dist[0]
    if kind == "normal":
        return g.normal(dist[1], dist[2], size=shape)
    if kind == "uniform":
        return g.uniform(dist[1], dist[2], size=shape)
    raise ValueError(kind)


def identity_theta(n, r):
    """(n, r, r+1) stack of [I | 0]."""
    t = np.zeros((n, r, r + 1))
    for d in range(r):
        t[:, d, d] = 1.0
    return t


def make_grid_sample_inputs(w, seed=None, x_shape=None, out_spatial=None):
    """X and grid for a GridSample workload (shapes may be overridden for small cases)."""
    g = rng(w.seed if seed is None else seed)
    xs = tuple(x_shape or w.x_shape)
    os_ = tuple(out_spatial or w.out_spatial)
    X = draw(g, w.x_dist, xs)
    grid = draw(g, w.grid_dist, (xs[0],) + os_ + (len(os_),))
    return {"X": X, "grid": grid}


def make_affine_sample_inputs(w, seed=None, x_shape=None, out_spatial=None):
    """theta and X for a fused AffineGrid+GridSample workload; size = (N, C, out...)."""
    g = rng(w.seed if seed is None else seed)
    xs = tuple(x_shape or w.x_shape)
    os_ = tuple(out_spatial or w.out_spatial)
    r = len(os_)
    theta = identity_theta(xs[0], r) + g.normal(0.0, w.theta_noise, size=(xs[0], r, r + 1))
    X = draw(g, w.x_dist, xs)
    size = np.array((xs[0], xs[1]) + os_, dtype=np.int64)
    return {"theta": theta, "X": X, "size": size}


def make_deform_inputs(w, seed=None, x_shape=None, oc=None, kernel=None):
    """X, W, B, offset, mask for a DeformConv workload (stride/pads/dilations from w)."""
    g = rng(w.seed if seed is None else seed)
    xs = tuple(x_shape or w.x_shape)
    oc = oc or w.oc
    kh, kw = kernel or w.kernel
    N, C, H, W_ = xs
    oh = (H + w.pads[0] + w.pads[2] - w.dilations[0] * (kh - 1) - 1) // w.strides[0] + 1
    ow = (W_ + w.pads[1] + w.pads[3] - w.dilations[1] * (kw - 1) - 1) // w.strides[1] + 1
    X = g.normal(0.0, 1.0, size=xs)
    Wt = g.normal(0.0, 0.05, size=(oc, C // w.group, kh, kw))
    B = g.normal(0.0, 1.0, size=(oc,))
    offset = g.normal(0.0, 1.0, size=(N, w.offset_group * kh * kw * 2, oh, ow))
    mask = 1.0 / (1.0 + np.exp(-g.normal(0.0, 1.0, size=(N, w.offset_group * kh * kw, oh, ow))))
    return {"X": X, "W": Wt, "B": B, "offset": offset, "mask": mask}


def make_resize_inputs(w, seed=None, x_shape=None):
    """X for a Resize workload (the scales and attributes are in w)."""
    g = rng(w.seed if seed is None else seed)
    return {"X": draw(g, w.x_dist, tuple(x_shape or w.x_shape))}


def as_dtype(a, dtype):
    """Round a float64 array to a torch CPU tensor of ``dtype`` (round-to-nearest-even)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    return t.to(getattr(torch, dtype) if isinstance(dtype, str) else dtype)


def widened(t):
    """A torch tensor of any float dtype widened exactly to a float64 numpy array."""
    import torch
    return t.detach().to("cpu").to(torch.float64).numpy()
