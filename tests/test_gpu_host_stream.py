"""The host-streaming calls (pinned host buffers, chunked, copies overlapped with the
kernels) give exactly the device call's results."""
import pytest
import torch

from spatial_transformer_sampling_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("chunks", [1, 3, 8])
def test_affine_sample_from_host_matches_device_call(gs_cuda, chunks):
    w = wl.WORKLOADS["stn2d"]
    inp = wl.make_affine_sample_inputs(w, x_shape=(7, 5, 64, 48), out_spatial=(40, 56))
    T, X = wl.as_dtype(inp["theta"], "float32"), wl.as_dtype(inp["X"], "float32")
    ref = gs_cuda.gs_affine_sample(T.cuda(), inp["size"], X.cuda(), "linear", "border", 1).cpu()
    st = gs_cuda.HostStreamer("cuda", chunks=chunks)
    got = gs_cuda.gs_affine_sample_from_host(T.pin_memory(), inp["size"], X.pin_memory(),
                                             "linear", "border", 1, streamer=st)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    got2 = gs_cuda.gs_affine_sample_from_host(T.pin_memory(), inp["size"], X.pin_memory(),
                                              "linear", "border", 1, streamer=st)
    torch.cuda.synchronize()
    assert torch.equal(got2, ref)


def test_grid_sample_from_host_matches_device_call(gs_cuda):
    g = wl.rng(3)
    X = wl.as_dtype(g.normal(size=(5, 3, 20, 30)), "float16")
    G = wl.as_dtype(g.uniform(-1.2, 1.2, size=(5, 11, 13, 2)), "float16")
    ref = gs_cuda.gs_grid_sample(X.cuda(), G.cuda(), "cubic", "reflection", 0).cpu()
    got = gs_cuda.gs_grid_sample_from_host(X.pin_memory(), G.pin_memory(), "cubic", "reflection",
                                           0, streamer=gs_cuda.HostStreamer("cuda", chunks=2))
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
