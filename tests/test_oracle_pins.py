"""The oracle pinned to things other than itself: brute force, closed forms,
invariants and special cases that reduce to library routines.

The brute-force check below uses a different formulation from the oracle's
tap loop: it extends the signal past its border by the padding rule and
convolves the extension with the continuous interpolation kernel (hat for
linear, Keys for cubic, a box at the nearest index for nearest), summing over
every integer position in reach.  Any slip in tap selection, tap order, the
weight pairing or the padding index map shows up as a mismatch.
"""
import itertools

import numpy as np
import pytest
import torch

from spatial_transformer_sampling_gb300 import workloads as wl


# ---------------------------------------------------------------- brute force

def _unnorm(g, n, ac):
    return (g + 1) / 2 * (n - 1) if ac else ((g + 1) * n - 1) / 2


def _fold(x, lo, hi):
    """Reflect x at lo and hi until it lies in [lo, hi] (literal iteration)."""
    if hi <= lo:
        return lo
    for _ in range(10000):
        if x < lo:
            x = 2 * lo - x
        elif x > hi:
            x = 2 * hi - x
        else:
            return x
    raise RuntimeError("fold did not converge")


def _ext_index(m, n, pad, ac):
    """Index of the signal extension at integer m, or None for a zero."""
    if 0 <= m < n:
        return m
    if pad == "zeros":
        return None
    if pad == "border":
        return min(max(m, 0), n - 1)
    lo, hi = (0.0, n - 1.0) if ac else (-0.5, n - 0.5)
    return int(round(min(max(_fold(float(m), lo, hi), 0.0), n - 1.0)))


def _keys(s, a):
    s = abs(s)
    if s <= 1:
        return (a + 2) * s ** 3 - (a + 3) * s ** 2 + 1
    if s < 2:
        return a * s ** 3 - 5 * a * s ** 2 + 8 * a * s - 4 * a
    return 0.0


def _axis_dense(g, n, mode, pad, ac, a):
    """Dense weight over the signal extension: list of (extension index, weight)."""
    x = _unnorm(g, n, ac)
    if mode == "nearest":
        if pad == "border":
            x = min(max(x, 0.0), n - 1.0)
        elif pad == "reflection":
            lo, hi = (0.0, n - 1.0) if ac else (-0.5, n - 0.5)
            x = min(max(_fold(x, lo, hi), 0.0), n - 1.0)
        return [(_ext_index(int(np.rint(x)), n, "zeros", ac), 1.0)]
    out = []
    base = int(np.floor(x))
    for m in range(base - 3, base + 4):
        wgt = max(0.0, 1.0 - abs(x - m)) if mode == "linear" else _keys(x - m, a)
        if wgt != 0.0:
            out.append((_ext_index(m, n, pad, ac), wgt))
    return out


def _brute_grid_sample(X, grid, mode, pad, ac, a=-0.75):
    N, C = X.shape[:2]
    ins = X.shape[2:]
    r = len(ins)
    outs = grid.shape[1:-1]
    Y = np.zeros((N, C) + outs)
    for n in range(N):
        for o in itertools.product(*[range(s) for s in outs]):
            g = grid[(n,) + o]
            per_axis = [_axis_dense(g[r - 1 - d], ins[d], mode, pad, ac, a) for d in range(r)]
            for combo in itertools.product(*per_axis):
                if any(j is None for j, _ in combo):
                    continue
                wgt = np.prod([w for _, w in combo])
                Y[(n, slice(None)) + o] += wgt * X[(n, slice(None)) + tuple(j for j, _ in combo)]
    return Y


CASES = [(r, mode, pad, ac)
         for r in (1, 2, 3)
         for mode in ("linear", "nearest", "cubic")
         for pad in ("zeros", "border", "reflection")
         for ac in (0, 1)]


@pytest.mark.parametrize("r,mode,pad,ac", CASES)
def test_tap_oracle_matches_dense_brute_force(oracle_mod, r, mode, pad, ac):
    g = wl.rng(7 + r)
    ins = {1: (7,), 2: (5, 4), 3: (4, 3, 5)}[r]
    outs = {1: (11,), 2: (4, 5), 3: (3, 2, 4)}[r]
    X = g.normal(size=(2, 2) + ins)
    grid = g.uniform(-2.6, 2.6, size=(2,) + outs + (r,))
    # a few exact landmarks: the extrema, the centre and one far-out point
    flat = grid.reshape(-1, r)
    flat[:4] = np.array([-1.0, 1.0, 0.0, 7.25])[:, None]
    Y = oracle_mod.grid_sample(X, grid, mode, pad, ac)
    Yb = _brute_grid_sample(X, grid, mode, pad, ac)
    np.testing.assert_allclose(Y, Yb, rtol=0, atol=1e-12)


# ranks 4-6 (the operator's rank r+2 X, any r): every mode x padding x
# align_corners at rank 4, a spread of them at ranks 5 and 6
ND_CASES = ([(4, m, p, ac) for m in ("linear", "nearest", "cubic")
             for p in ("zeros", "border", "reflection") for ac in (0, 1)] +
            [(5, "linear", "reflection", 0), (5, "cubic", "border", 1), (5, "nearest", "zeros", 0),
             (6, "linear", "zeros", 1), (6, "cubic", "reflection", 0), (6, "nearest", "border", 1)])


@pytest.mark.parametrize("r,mode,pad,ac", ND_CASES)
def test_tap_oracle_matches_dense_brute_force_rank_nd(oracle_mod, r, mode, pad, ac):
    g = wl.rng(17 + 3 * r)
    ins = {4: (3, 4, 2, 3), 5: (3, 2, 4, 2, 3), 6: (2, 3, 2, 2, 3, 2)}[r]
    outs = {4: (3, 2, 2, 3), 5: (2, 2, 1, 2, 3), 6: (1, 2, 1, 2, 1, 2)}[r]
    X = g.normal(size=(1, 2) + ins)
    grid = g.uniform(-2.6, 2.6, size=(1,) + outs + (r,))
    flat = grid.reshape(-1, r)
    flat[:3] = np.array([-1.0, 1.0, 0.0])[:, None]
    Y = oracle_mod.grid_sample(X, grid, mode, pad, ac)
    Yb = _brute_grid_sample(X, grid, mode, pad, ac)
    np.testing.assert_allclose(Y, Yb, rtol=0, atol=1e-12)


def _positions(grid, ins, ac):
    """Unnormalised positions, outermost axis first (the grid lists innermost first)."""
    r = len(ins)
    return [_unnorm(grid[..., r - 1 - d], ins[d], ac) for d in range(r)]


def test_rank5_linear_reproduces_multilinear_functions(oracle_mod):
    """N-linear interpolation is exact on functions that are affine in each
    coordinate separately (products of ramps, plus ramps)."""
    ins = (4, 3, 5, 3, 4)
    c = np.array([0.3, -0.7, 0.2, 1.1, -0.4])
    e = np.array([1.5, -0.25, 0.75, 0.5, -1.0])
    idx = np.meshgrid(*[np.arange(n, dtype=np.float64) for n in ins], indexing="ij")

    def f(p):
        return np.prod([1.0 + c[d] * p[d] for d in range(5)], axis=0) + \
            sum(e[d] * p[d] for d in range(5))

    X = f(idx)[None, None]
    grid = wl.rng(131).uniform(-1, 1, size=(1, 3, 4, 2, 3, 2, 5))
    Y = oracle_mod.grid_sample(X, grid, "linear", "zeros", 1)
    np.testing.assert_allclose(Y[0, 0], f(_positions(grid[0], ins, 1)), atol=1e-12)


def test_rank4_cubic_reproduces_quadratics_at_a_minus_half(oracle_mod):
    """Keys' kernel with a = -1/2 reproduces polynomials up to degree two on each
    axis (Keys, 1981), so the tensor product reproduces sums of such products."""
    ins = (7, 8, 7, 8)
    idx = np.meshgrid(*[np.arange(n, dtype=np.float64) for n in ins], indexing="ij")

    def f(p):
        return (0.2 * p[0] * p[0] - 0.5 * p[0] * p[3] + 0.1 * p[1] * p[1] + p[2]
                - 0.3 * p[1] * p[2] * p[3] + 0.05 * p[3] * p[3] * p[0] * p[0])

    X = f(idx)[None, None]
    grid = wl.rng(141).uniform(-0.4, 0.4, size=(1, 3, 2, 4, 3, 4))   # every tap inside
    Y = oracle_mod.grid_sample(X, grid, "cubic", "zeros", 1, -0.5)
    np.testing.assert_allclose(Y[0, 0], f(_positions(grid[0], ins, 1)), atol=1e-10)
    Y75 = oracle_mod.grid_sample(X, grid, "cubic", "zeros", 1, -0.75)
    assert np.abs(Y75[0, 0] - f(_positions(grid[0], ins, 1))).max() > 1e-3


def test_rank6_nearest_picks_the_nearest_pixel(oracle_mod):
    """Positions within 0.4 px of a pixel centre read that pixel, on every axis."""
    ins = (3, 4, 2, 3, 4, 2)
    g = wl.rng(151)
    X = g.normal(size=(1, 2) + ins)
    outs = (2, 3, 2, 2, 3, 2)
    pick = np.stack([g.integers(0, ins[d], size=outs) for d in range(6)])     # outermost first
    pos = pick + g.uniform(-0.4, 0.4, size=pick.shape)
    # align_corners=0: x = ((g+1)*n - 1)/2  ->  g = (2x + 1)/n - 1
    grid = np.stack([(2 * pos[d] + 1) / ins[d] - 1 for d in reversed(range(6))], -1)[None]
    Y = oracle_mod.grid_sample(X, grid, "nearest", "zeros", 0)
    for c in range(2):
        np.testing.assert_array_equal(Y[0, c], X[0, c][tuple(pick)])


@pytest.mark.parametrize("a", [-0.5, -0.75, -1.0])
def test_cubic_coefficient_is_a_parameter(oracle_mod, a):
    g = wl.rng(3)
    X = g.normal(size=(1, 1, 6, 5))
    grid = g.uniform(-1.3, 1.3, size=(1, 3, 4, 2))
    Y = oracle_mod.grid_sample(X, grid, "cubic", "border", 0, a)
    Yb = _brute_grid_sample(X, grid, "cubic", "border", 0, a)
    np.testing.assert_allclose(Y, Yb, rtol=0, atol=1e-12)


# -------------------------------------------- library routine: torch CPU fp64

TORCH_CASES = [(r, mode, pad, ac)
               for r in (2, 3)
               for mode in (("bilinear", "nearest", "bicubic") if r == 2 else ("bilinear", "nearest"))
               for pad in ("zeros", "border", "reflection")
               for ac in (0, 1)]


@pytest.mark.parametrize("r,mode,pad,ac", TORCH_CASES)
def test_grid_sample_matches_torch_cpu_fp64(oracle_mod, r, mode, pad, ac):
    """torch.nn.functional.grid_sample, which the GridSample page cites as 'see also'."""
    g = wl.rng(11 + r)
    ins = (9, 7) if r == 2 else (5, 6, 4)
    outs = (6, 8) if r == 2 else (4, 3, 5)
    X = g.normal(size=(2, 3) + ins)
    grid = g.uniform(-1.7, 1.7, size=(2,) + outs + (r,))
    ours = oracle_mod.grid_sample(X, grid, mode, pad, ac)
    ref = torch.nn.functional.grid_sample(torch.from_numpy(X), torch.from_numpy(grid), mode=mode,
                                          padding_mode=pad, align_corners=bool(ac)).numpy()
    np.testing.assert_allclose(ours, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("r,ac", [(2, 0), (2, 1), (3, 0), (3, 1)])
def test_affine_grid_matches_torch_cpu_fp64(oracle_mod, r, ac):
    g = wl.rng(21 + r)
    size = (3, 2, 5, 7) if r == 2 else (3, 2, 4, 5, 6)
    theta = g.normal(size=(3, r, r + 1))
    ours = oracle_mod.affine_grid(theta, size, ac)
    ref = torch.nn.functional.affine_grid(torch.from_numpy(theta), list(size),
                                          align_corners=bool(ac)).numpy()
    np.testing.assert_allclose(ours, ref, rtol=0, atol=1e-13)


# ------------------------------------------------------------- closed forms

@pytest.mark.parametrize("ac", [0, 1])
@pytest.mark.parametrize("mode", ["linear", "nearest", "cubic"])
@pytest.mark.parametrize("r", [2, 3])
def test_identity_theta_reproduces_X(oracle_mod, r, mode, ac):
    g = wl.rng(31)
    xs = (2, 3, 6, 5) if r == 2 else (2, 2, 4, 5, 3)
    X = g.normal(size=xs)
    theta = wl.identity_theta(xs[0], r)
    Y = oracle_mod.affine_sample(theta, xs, X, mode, "zeros", ac)
    np.testing.assert_allclose(Y, X, rtol=0, atol=1e-12)


@pytest.mark.parametrize("ac", [0, 1])
def test_affine_grid_is_exactly_affine_in_the_output_index(oracle_mod, ac):
    g = wl.rng(41)
    theta = g.normal(size=(2, 2, 3))
    H, W = 6, 9
    grid = oracle_mod.affine_grid(theta, (2, 1, H, W), ac)
    step_w = 2.0 / (W - 1) if ac else 2.0 / W
    step_h = 2.0 / (H - 1) if ac else 2.0 / H
    dw = np.diff(grid, axis=2)
    dh = np.diff(grid, axis=1)
    np.testing.assert_allclose(dw, np.broadcast_to(theta[:, None, None, :, 0] * step_w, dw.shape),
                               atol=1e-14)
    np.testing.assert_allclose(dh, np.broadcast_to(theta[:, None, None, :, 1] * step_h, dh.shape),
                               atol=1e-14)
    # the corner positions: centres of the corner pixels (ac=1) or half a pixel in (ac=0)
    first = -1.0 if ac else -1.0 + 1.0 / W
    np.testing.assert_allclose(grid[:, 0, 0, 0], theta[:, 0, 0] * first
                               + theta[:, 0, 1] * (-1.0 if ac else -1.0 + 1.0 / H) + theta[:, 0, 2],
                               atol=1e-14)


def test_extrema_land_on_pixel_centres_or_edges(oracle_mod):
    X = np.arange(5.0).reshape(1, 1, 1, 5) * 3.0 + 1.0
    for ac, exp in ((1, [1.0, 13.0]), (0, [1.0, 13.0])):
        grid = np.array([[[[-1.0, 0.0], [1.0, 0.0]]]])
        Y = oracle_mod.grid_sample(X, grid, "linear", "border", ac)
        np.testing.assert_array_equal(Y[0, 0, 0], exp)
    # ac=0, zeros: the edge is half a pixel out, so the corner value is halved
    Y = oracle_mod.grid_sample(X, np.array([[[[-1.0, 0.0], [1.0, 0.0]]]]), "linear", "zeros", 0)
    np.testing.assert_array_equal(Y[0, 0, 0], [0.5, 6.5])


# --------------------------------------------------------------- invariants

@pytest.mark.parametrize("a", [-0.5, -0.75, -1.0])
@pytest.mark.parametrize("mode", ["linear", "cubic"])
def test_partition_of_unity(oracle_mod, mode, a):
    g = wl.rng(51)
    X = np.full((1, 2, 7, 6), 2.5)
    grid = g.uniform(-3, 3, size=(1, 5, 5, 2))
    Y = oracle_mod.grid_sample(X, grid, mode, "border", 0, a)
    np.testing.assert_allclose(Y, 2.5, atol=1e-13)


def test_linear_reproduces_affine_ramps(oracle_mod):
    H, W = 7, 9
    i, j = np.meshgrid(np.arange(H), np.arange(W), indexing="ij")
    X = (0.3 * i - 1.7 * j + 0.25)[None, None]
    g = wl.rng(61)
    grid = g.uniform(-1, 1, size=(1, 6, 6, 2))
    Y = oracle_mod.grid_sample(X, grid, "linear", "zeros", 1)
    xs = (grid[..., 0] + 1) / 2 * (W - 1)
    ys = (grid[..., 1] + 1) / 2 * (H - 1)
    np.testing.assert_allclose(Y[0, 0], (0.3 * ys - 1.7 * xs + 0.25)[0], atol=1e-12)


def test_cubic_reproduces_quadratics_only_at_a_minus_half(oracle_mod):
    H, W = 12, 12
    i, j = np.meshgrid(np.arange(H), np.arange(W), indexing="ij")
    X = (0.2 * i * i - 0.5 * i * j + 0.1 * j * j + j)[None, None].astype(np.float64)
    g = wl.rng(71)
    grid = g.uniform(-0.6, 0.6, size=(1, 5, 5, 2))   # every tap stays inside
    xs = (grid[..., 0] + 1) / 2 * (W - 1)
    ys = (grid[..., 1] + 1) / 2 * (H - 1)
    exact = (0.2 * ys * ys - 0.5 * ys * xs + 0.1 * xs * xs + xs)[0]
    Y = oracle_mod.grid_sample(X, grid, "cubic", "zeros", 1, -0.5)
    np.testing.assert_allclose(Y[0, 0], exact, atol=1e-11)
    Y75 = oracle_mod.grid_sample(X, grid, "cubic", "zeros", 1, -0.75)
    assert np.abs(Y75[0, 0] - exact).max() > 1e-3


@pytest.mark.parametrize("pad", ["zeros", "border", "reflection"])
def test_nearest_outputs_are_copies_of_X(oracle_mod, pad):
    g = wl.rng(81)
    X = g.normal(size=(2, 3, 6, 7))
    grid = g.uniform(-2.5, 2.5, size=(2, 8, 8, 2))
    Y = oracle_mod.grid_sample(X, grid, "nearest", pad, 0)
    for n in range(2):
        for c in range(3):
            allowed = set(X[n, c].ravel().tolist()) | ({0.0} if pad == "zeros" else set())
            assert set(Y[n, c].ravel().tolist()) <= allowed


def test_linear_border_output_stays_in_the_range_of_X(oracle_mod):
    g = wl.rng(91)
    X = g.normal(size=(1, 4, 6, 6))
    grid = g.uniform(-4, 4, size=(1, 9, 9, 2))
    Y = oracle_mod.grid_sample(X, grid, "linear", "border", 1)
    for c in range(4):
        assert X[0, c].min() - 1e-15 <= Y[0, c].min() and Y[0, c].max() <= X[0, c].max() + 1e-15


@pytest.mark.parametrize("ac", [0, 1])
def test_reflection_matches_literal_folding(oracle_mod, ac):
    """A ramp X = [0, 1, ..., n-1] returns the padded coordinate itself."""
    n = 6
    X = np.arange(float(n)).reshape(1, 1, n)
    g = wl.rng(101)
    gv = np.concatenate([g.uniform(-9, 9, 200), [-1.0, 1.0, 3.0, -3.0]])
    Y = oracle_mod.grid_sample(X, gv.reshape(1, -1, 1), "linear", "reflection", ac)
    lo, hi = (0.0, n - 1.0) if ac else (-0.5, n - 0.5)
    exp = [min(max(_fold(_unnorm(v, n, ac), lo, hi), 0.0), n - 1.0) for v in gv]
    np.testing.assert_allclose(Y[0, 0], exp, atol=1e-12)


def test_reflection_sentence_example(oracle_mod):
    """GridSample padding_mode: x = -3.5 reflects at -1 to 1.5, then at 1 to 0.5.

    With align_corners=1 and three pixels, pixel position p corresponds to
    the page's location p - 1, so the borders -1 and 1 are pixels 0 and 2 and
    a ramp X = [0, 1, 2] returns p = 0.5 + 1.
    """
    assert _fold(-3.5, -1.0, 1.0) == 0.5
    Y = oracle_mod.grid_sample(np.array([[[0.0, 1.0, 2.0]]]), np.array([[[-3.5]]]), "linear",
                               "reflection", 1)
    assert Y[0, 0, 0] == 1.5


@pytest.mark.parametrize("ac", [0, 1])
def test_reflection_is_symmetric_about_the_borders(oracle_mod, ac):
    g = wl.rng(111)
    X = g.normal(size=(1, 2, 5, 6))
    grid = g.uniform(-1, 1, size=(1, 4, 4, 2))
    for mode in ("linear", "cubic"):
        Y = oracle_mod.grid_sample(X, grid, mode, "reflection", ac)
        Y_hi = oracle_mod.grid_sample(X, 2.0 - grid, mode, "reflection", ac)
        Y_lo = oracle_mod.grid_sample(X, -2.0 - grid, mode, "reflection", ac)
        np.testing.assert_allclose(Y_hi, Y, atol=1e-12)
        np.testing.assert_allclose(Y_lo, Y, atol=1e-12)


def test_integer_pixel_shift_of_the_grid_shifts_X(oracle_mod):
    g = wl.rng(121)
    X = g.normal(size=(1, 2, 8, 9))
    W, H = 9, 8
    jj, ii = np.meshgrid(np.arange(2, 6), np.arange(2, 6))
    grid = np.stack([(2 * (jj + 1) + 1) / W - 1, (2 * (ii - 2) + 1) / H - 1], -1)[None]
    Y = oracle_mod.grid_sample(X, grid, "linear", "zeros", 0)
    np.testing.assert_allclose(Y[0], X[0][:, ii - 2, jj + 1], atol=1e-12)


@pytest.mark.parametrize("mode", ["linear", "nearest", "cubic"])
def test_fused_equals_grid_sample_of_affine_grid(oracle_mod, mode):
    g = wl.rng(131)
    X = g.normal(size=(2, 3, 6, 7))
    theta = wl.identity_theta(2, 2) + g.normal(0, 0.2, size=(2, 2, 3))
    size = (2, 3, 5, 4)
    fused = oracle_mod.affine_sample(theta, size, X, mode, "reflection", 0)
    two = oracle_mod.grid_sample(X, oracle_mod.affine_grid(theta, size, 0), mode, "reflection", 0)
    np.testing.assert_array_equal(fused, two)


def test_point_evaluators_match_full_outputs(oracle_mod):
    g = wl.rng(141)
    X = g.normal(size=(2, 3, 6, 7))
    grid = g.uniform(-1.2, 1.2, size=(2, 5, 4, 2))
    Y = oracle_mod.grid_sample(X, grid, "cubic", "reflection", 1)
    idx = g.integers(0, Y.size, 37)
    np.testing.assert_array_equal(
        oracle_mod.grid_sample_at(X, grid, idx, "cubic", "reflection", 1), Y.ravel()[idx])
    theta = wl.identity_theta(2, 2) + g.normal(0, 0.2, size=(2, 2, 3))
    Ya = oracle_mod.affine_sample(theta, (2, 3, 5, 4), X, "linear", "border", 0)
    idx = g.integers(0, Ya.size, 29)
    np.testing.assert_array_equal(
        oracle_mod.affine_sample_at(theta, (2, 3, 5, 4), X, idx, "linear", "border", 0),
        Ya.ravel()[idx])


# ---------------------------------------------------------------- DeformConv

DEFORM_CASES = [
    dict(kernel=(3, 3), pads=(1, 1, 1, 1), strides=(1, 1), dil=(1, 1), group=1, og=1),
    dict(kernel=(3, 2), pads=(0, 1, 2, 0), strides=(2, 1), dil=(1, 2), group=2, og=1),
    dict(kernel=(2, 2), pads=(1, 0, 0, 1), strides=(1, 2), dil=(2, 1), group=1, og=2),
    dict(kernel=(3, 3), pads=(2, 2, 2, 2), strides=(2, 2), dil=(2, 2), group=2, og=4),
]


def _deform_inputs(g, case, N=2, C=4, H=7, W=8, oC=6):
    kh, kw = case["kernel"]
    p, s, d = case["pads"], case["strides"], case["dil"]
    oH = (H + p[0] + p[2] - d[0] * (kh - 1) - 1) // s[0] + 1
    oW = (W + p[1] + p[3] - d[1] * (kw - 1) - 1) // s[1] + 1
    X = g.normal(size=(N, C, H, W))
    Wt = g.normal(size=(oC, C // case["group"], kh, kw))
    B = g.normal(size=(oC,))
    return X, Wt, B, (oH, oW)


def _deform(oracle_mod, X, Wt, off, case, B=None, mask=None):
    return oracle_mod.deform_conv(X, Wt, off, B, mask, kernel_shape=case["kernel"],
                                  pads=case["pads"], strides=case["strides"],
                                  dilations=case["dil"], group=case["group"],
                                  offset_group=case["og"])


@pytest.mark.parametrize("case", DEFORM_CASES)
def test_deform_conv_with_zero_offsets_is_conv2d(oracle_mod, case):
    g = wl.rng(151)
    X, Wt, B, (oH, oW) = _deform_inputs(g, case)
    K = case["kernel"][0] * case["kernel"][1]
    off = np.zeros((X.shape[0], case["og"] * K * 2, oH, oW))
    Y = _deform(oracle_mod, X, Wt, off, case, B)
    p = case["pads"]
    Xp = np.pad(X, ((0, 0), (0, 0), (p[0], p[2]), (p[1], p[3])))
    ref = torch.nn.functional.conv2d(torch.from_numpy(Xp), torch.from_numpy(Wt), torch.from_numpy(B),
                                     stride=case["strides"], dilation=case["dil"],
                                     groups=case["group"]).numpy()
    np.testing.assert_allclose(Y, ref, atol=1e-12)


@pytest.mark.parametrize("case", DEFORM_CASES[:2])
def test_deform_conv_integer_offsets_shift_the_input(oracle_mod, case):
    """Offset (dy, dx) = (1, -2) everywhere equals conv2d of X shifted by (-1, +2)."""
    g = wl.rng(161)
    X, Wt, B, (oH, oW) = _deform_inputs(g, case)
    K = case["kernel"][0] * case["kernel"][1]
    off = np.zeros((X.shape[0], case["og"] * K * 2, oH, oW))
    off[:, 0::2] = 1.0
    off[:, 1::2] = -2.0
    mask = np.full((X.shape[0], case["og"] * K, oH, oW), 0.75)
    Y = _deform(oracle_mod, X, Wt, off, case, None, mask)
    p = case["pads"]
    Xp = np.pad(X, ((0, 0), (0, 0), (p[0], p[2]), (p[1], p[3])))
    Xps = np.zeros_like(Xp)
    Xps[:, :, :-1, 2:] = Xp[:, :, 1:, :-2]
    ref = torch.nn.functional.conv2d(torch.from_numpy(Xps), torch.from_numpy(Wt), None,
                                     stride=case["strides"], dilation=case["dil"],
                                     groups=case["group"]).numpy()
    np.testing.assert_allclose(Y, 0.75 * ref, atol=1e-12)


@pytest.mark.parametrize("case", DEFORM_CASES)
def test_deform_conv_is_a_contraction_of_bilinear_samples(oracle_mod, case):
    """Fractional offsets: each sample is GridSample(linear, zeros, align_corners=0)
    of the unpadded X at the shifted position; the output contracts them with W."""
    g = wl.rng(171)
    X, Wt, B, (oH, oW) = _deform_inputs(g, case)
    N, C, H, W = X.shape
    kh, kw = case["kernel"]
    K = kh * kw
    og = case["og"]
    off = g.normal(0, 1.5, size=(N, og * K * 2, oH, oW))
    mask = g.uniform(0, 1, size=(N, og * K, oH, oW))
    Y = _deform(oracle_mod, X, Wt, off, case, B, mask)
    s, p, d = case["strides"], case["pads"], case["dil"]
    oh, ow = np.meshgrid(np.arange(oH), np.arange(oW), indexing="ij")
    cols = np.zeros((N, C, K, oH, oW))
    for c in range(C):
        o = c // (C // og)
        for k in range(K):
            ki, kj = divmod(k, kw)
            y = oh * s[0] - p[0] + ki * d[0] + off[:, o * 2 * K + 2 * k]
            x = ow * s[1] - p[1] + kj * d[1] + off[:, o * 2 * K + 2 * k + 1]
            grid = np.stack([(2 * x + 1) / W - 1, (2 * y + 1) / H - 1], -1)
            smp = oracle_mod.grid_sample(X[:, c:c + 1], grid, "linear", "zeros", 0)[:, 0]
            cols[:, c, k] = smp * mask[:, o * K + k]
    G = case["group"]
    Cg, oCg = C // G, Wt.shape[0] // G
    ref = np.zeros_like(Y)
    for gi in range(G):
        ref[:, gi * oCg:(gi + 1) * oCg] = np.einsum(
            "ock,nckhw->nohw", Wt[gi * oCg:(gi + 1) * oCg].reshape(oCg, Cg, K),
            cols[:, gi * Cg:(gi + 1) * Cg])
    ref += B[None, :, None, None]
    np.testing.assert_allclose(Y, ref, atol=1e-11)


def test_deform_point_evaluator_matches_full_output(oracle_mod):
    g = wl.rng(181)
    case = DEFORM_CASES[3]
    X, Wt, B, (oH, oW) = _deform_inputs(g, case)
    K = 9
    off = g.normal(size=(X.shape[0], case["og"] * K * 2, oH, oW))
    Y = _deform(oracle_mod, X, Wt, off, case, B)
    idx = g.integers(0, Y.size, 31)
    vals = oracle_mod.deform_conv_at(X, Wt, off, idx, B, None, kernel_shape=case["kernel"],
                                     pads=case["pads"], strides=case["strides"],
                                     dilations=case["dil"], group=case["group"],
                                     offset_group=case["og"])
    np.testing.assert_array_equal(vals, Y.ravel()[idx])


def test_integer_cast_truncates_toward_zero_and_saturates(oracle_mod):
    v = np.array([-129.7, -128.0, -2.9, -0.4, 0.0, 0.99, 3.0, 126.999, 127.5, 300.0])
    np.testing.assert_array_equal(oracle_mod.cast_to_integer(v, "int8"),
                                  [-128, -128, -2, 0, 0, 0, 3, 126, 127, 127])
    np.testing.assert_array_equal(oracle_mod.cast_to_integer(v, "uint8"),
                                  [0, 0, 0, 0, 0, 0, 3, 126, 127, 255])
    np.testing.assert_array_equal(oracle_mod.cast_to_integer([70000.2, -5.0], "uint16"), [65535, 0])
    np.testing.assert_array_equal(oracle_mod.cast_to_integer([-40000.0, 1.5], "int16"), [-32768, 1])
