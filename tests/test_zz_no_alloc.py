"""gs_grid_sample_static (scratch in the library's static device memory, no
allocation in the call) against gs_grid_sample on the GPU.  The entry point
exists for callers that cannot allocate device memory where they call it (a
plugin whose host framework owns all device memory, a loop that must not block
on cudaMalloc/cudaFree, a budget fixed at start-up); it shares one scratch
array per device between all calls.

Collected last on purpose: it must pass alone and after every other test, so
nothing earlier may leave state it depends on.  Each case runs two calls in a
row on different inputs (different shapes, channel counts and padding, so a
stale zero pixel or a stale image in the shared scratch would show) and
compares each result with the existing entry point value for value.
"""
import numpy as np
import pytest
import torch

from conftest import assert_parity
from spatial_transformer_sampling_gb300 import GsError
from spatial_transformer_sampling_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _inputs(seed, xs, out, dtype, lo=-1.3, hi=1.3):
    g = wl.rng(seed)
    Xt = wl.as_dtype(g.normal(size=xs), dtype)
    Gt = wl.as_dtype(g.uniform(lo, hi, size=(xs[0],) + tuple(out) + (len(out),)), dtype)
    return Xt, Gt


CALL_PAIRS = [
    # (x_shape, out, mode, pad, ac, dtype) for the first and the second call
    (((3, 32, 21, 19), (17, 23), "cubic", "reflection", 0, "float32"),
     ((2, 64, 13, 30), (11, 9), "linear", "zeros", 1, "float32")),
    (((2, 16, 40, 33), (29, 31), "linear", "zeros", 0, "float16"),
     ((4, 8, 12, 10), (15, 14), "nearest", "border", 1, "float16")),
    (((2, 128, 9, 11), (7, 13), "cubic", "zeros", 1, "bfloat16"),
     ((3, 72, 17, 16), (19, 18), "cubic", "border", 0, "bfloat16")),
]


@pytest.mark.parametrize("pair", range(len(CALL_PAIRS)))
def test_static_matches_grid_sample_on_two_calls_in_a_row(gs_cuda, oracle_mod, pair):
    outs, refs = [], []
    for k, (xs, out, mode, pad, ac, dtype) in enumerate(CALL_PAIRS[pair]):
        Xt, Gt = _inputs(900 + 10 * pair + k, xs, out, dtype)
        Xd, Gd = Xt.cuda(), Gt.cuda()
        outs.append((gs_cuda.gs_grid_sample_static(Xd, Gd, mode, pad, ac),
                     gs_cuda.gs_grid_sample(Xd, Gd, mode, pad, ac)))
        refs.append((oracle_mod.grid_sample(wl.widened(Xt), wl.widened(Gt), mode, pad, ac),
                     dtype, mode))
    torch.cuda.synchronize()
    assert gs_cuda.gs_device_status() == 0
    for (Ys, Y0), (ref, dtype, mode) in zip(outs, refs):
        assert torch.equal(Ys, Y0)
        if mode == "nearest":
            np.testing.assert_array_equal(wl.widened(Ys), ref)
        else:
            assert_parity(Ys, ref, dtype, f"static scratch, {mode}")


def test_static_chunks_a_batch_larger_than_the_scratch(gs_cuda):
    # 16.8 MB slots: three to a chunk in 64 MiB, four chunks for ten images
    Xt, Gt = _inputs(951, (10, 256, 128, 128), (40, 36), "float32")
    Xd, Gd = Xt.cuda(), Gt.cuda()
    for mode in ("cubic", "linear"):
        Ys = gs_cuda.gs_grid_sample_static(Xd, Gd, mode, "reflection", 0)
        assert torch.equal(Ys, gs_cuda.gs_grid_sample(Xd, Gd, mode, "reflection", 0))


# The edges of the chunking over the 64 MiB scratch: one image per chunk with a
# slot just under the limit, and a batch whose last chunk is exactly full.
CHUNK_EDGES = [
    # x_shape, slot bytes / images per chunk
    ((2, 64, 511, 511), "(511*511 + 1) * 64 * 4 B = 63.75 MiB: one image per chunk, two chunks"),
    ((6, 256, 128, 128), "16.8 MB slots, three per chunk: two full chunks"),
]


@pytest.mark.parametrize("case", range(len(CHUNK_EDGES)))
def test_static_chunk_edges_match_grid_sample_and_the_oracle(gs_cuda, oracle_mod, case):
    xs, why = CHUNK_EDGES[case]
    Xt, Gt = _inputs(970 + case, xs, (24, 20), "float32")
    Xd, Gd = Xt.cuda(), Gt.cuda()
    Ys = gs_cuda.gs_grid_sample_static(Xd, Gd, "cubic", "border", 0)
    assert torch.equal(Ys, gs_cuda.gs_grid_sample(Xd, Gd, "cubic", "border", 0)), why
    assert gs_cuda.gs_device_status() == 0
    # a few outputs of every image (first and last channel included) from the oracle
    g = wl.rng(980 + case)
    per_img = Ys[0].numel()
    idx = np.concatenate([n * per_img + np.concatenate([[0, per_img - 1],
                                                        g.integers(0, per_img, 30)])
                          for n in range(xs[0])])
    ref = oracle_mod.grid_sample_at(wl.widened(Xt), wl.widened(Gt), idx, "cubic", "border", 0)
    got = Ys.reshape(-1)[torch.from_numpy(idx).cuda()]
    assert_parity(got, ref, "float32", f"static scratch chunk edge: {why}")


def test_static_rejects_an_image_larger_than_the_scratch(gs_cuda):
    # (512*513 + 1) * 64 fp32 elements: 67.2 MB > GS_STATIC_WORKSPACE_BYTES
    X = torch.zeros((1, 64, 512, 513), device="cuda")
    grid = torch.zeros((1, 4, 4, 2), device="cuda")
    with pytest.raises(GsError, match="bad shape"):
        gs_cuda.gs_grid_sample_static(X, grid, "linear", "zeros", 0)
    # the same image in half precision fits (33.6 MB)
    Xh, gh = X.half(), grid.half()
    assert torch.equal(gs_cuda.gs_grid_sample_static(Xh, gh, "linear", "zeros", 0),
                       gs_cuda.gs_grid_sample(Xh, gh, "linear", "zeros", 0))


def test_static_shapes_outside_the_channel_last_path_use_no_scratch(gs_cuda):
    for xs, out in (((2, 6, 9, 10), (7, 8)),          # 24 bytes per pixel: no 16-byte vectors
                    ((2, 8, 37), (45,)),              # rank 1
                    ((1, 8, 5, 6, 7), (4, 5, 6))):    # rank 3
        Xt, Gt = _inputs(960 + len(out), xs, out, "float32")
        Xd, Gd = Xt.cuda(), Gt.cuda()
        assert torch.equal(gs_cuda.gs_grid_sample_static(Xd, Gd, "linear", "border", 0),
                           gs_cuda.gs_grid_sample(Xd, Gd, "linear", "border", 0))
