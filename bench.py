"""Benchmark of the spatial-transformer sampling path on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME] [--dtype DT] [--no-extra]

A step is one pass of the hot path over one batch: by default the fused
AffineGrid+GridSample 2-D workload "stn2d" -- theta (64,2,3) = identity +
N(0,0.1), X (64,32,128,128) ~ N(0,1) fp32, output 128x128, linear, border,
align_corners=1 -- one gs_affine_sample call.  Inputs are seeded synthetic
data resident in HBM before the timed region; L2 is flushed before every timed
step, outside the step's CUDA-event interval: a 512 MiB buffer is written and
then read, so L2 holds only clean, unrelated lines when the step starts (no
write-back of the flush is charged to the step).  Time is
taken with CUDA events on the stream the kernel runs on; the timed region is
bracketed by barrier + synchronize, and the max over ranks is reported.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the images are independent; there is no exchange step; rank r draws its
images at the workload's seed + r) and `value` is the whole job's output
elements per second over the slowest rank's time.

Beside the cold-L2 headline the line carries the median step time and a
warm-L2 figure (the same steps back to back, no flush).

--impl reference times the CPU oracle (plain C, fp64, OpenMP over output
elements) on a bounded sample of the same workload and prints the same JSON
line with "impl": "reference".
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from spatial_transformer_sampling_gb300 import workloads as wl  # noqa: E402

DT_SHORT = {"float32": "f32", "float16": "f16", "bfloat16": "bf16"}
DT_BYTES = {"float32": 4, "float16": 2, "bfloat16": 2}
METRIC = "GridSample output elems/s (achieved HBM GB/s in roofline)"
UNIT = "elems/s"


# ------------------------------------------------------------------ helpers

def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="stn2d")
    p.add_argument("--dtype", default="float32")
    p.add_argument("--mode", default=None, help="override the workload's mode")
    p.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    p.add_argument("--workspace", action="store_true",
                   help="GridSample workloads: gs_grid_sample_ws with the workspace it asks for")
    p.add_argument("--extra-steps", type=int, default=100)
    p.add_argument("--sample-seconds", type=float, default=20.0,
                   help="--impl reference: oracle time per step (a bounded sample of the batch)")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# CUDA sources each kernel is built from (most specific tag prefix first).
KERNEL_SOURCES = {
    "band_kernel": ["gs_band.cuh", "gs_sample.cuh", "gs_common.cuh", "gs_ptx.cuh", "gs_internal.h"],
    "nhwc_sample_kernel": ["gs_nhwc.cuh", "gs_sample.cuh", "gs_common.cuh", "gs_internal.h"],
    "sample_kernel": ["gs_sample.cuh", "gs_common.cuh", "gs_ptx.cuh", "gs_internal.h"],
    "deform_tc_nhwc": ["gs_deform_tc.cuh", "gs_copy.cuh", "gs_common.cuh", "gs_ptx.cuh",
                       "gs_internal.h"],
    "deform_st_kernel": ["gs_deform_st.cuh", "gs_tma.cuh", "gs_common.cuh", "gs_ptx.cuh",
                         "gs_internal.h"],
    "deform_f32_kernel": ["gs_deform_f32.cu", "gs_common.cuh", "gs_ptx.cuh", "gs_internal.h"],
    "deform": ["gs_deform.cuh", "gs_deform_tc.cuh", "gs_common.cuh", "gs_ptx.cuh", "gs_internal.h"],
    "vol_tma_kernel": ["gs_vol_tma.cuh", "gs_vol.cuh", "gs_tma.cuh", "gs_sample.cuh",
                       "gs_common.cuh", "gs_ptx.cuh", "gs_internal.h"],
    "vol_kernel": ["gs_vol.cuh", "gs_sample.cuh", "gs_common.cuh", "gs_ptx.cuh", "gs_internal.h"],
    "resize_": ["gs_resize.cuh", "gs_common.cuh", "gs_ptx.cuh", "gs_internal.h"],
}


def kernel_source_sha(kernel_tag=None):
    """Hash of the CUDA sources a kernel is built from: recorded ncu traffic is
    reported only while those sources are unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "spatial_transformer_sampling_gb300", "csrc")
    names = sorted(os.listdir(csrc))
    if kernel_tag is not None:
        names = next((v for k, v in KERNEL_SOURCES.items() if kernel_tag.startswith(k)), names)
    for name in sorted(names):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_tag, workload, dtype):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha(kernel_tag)
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kv = dict(item.split("=", 1) for item in line.split())
        if (kv.get("kernel") == kernel_tag and kv.get("workload") == workload
                and kv.get("dtype") == dtype and kv.get("src_sha") == sha):
            return float(kv["dram_bytes_per_launch"])
    return None


def host_inputs(w, dtype, seed):
    """One replica's seeded inputs on the host, rounded to dtype (torch CPU tensors)."""
    if w.kind == "affine_sample":
        inp = wl.make_affine_sample_inputs(w, seed=seed)
        return {"theta": wl.as_dtype(inp["theta"], dtype), "X": wl.as_dtype(inp["X"], dtype)}
    if w.kind == "grid_sample":
        inp = wl.make_grid_sample_inputs(w, seed=seed)
        return {"X": wl.as_dtype(inp["X"], dtype), "grid": wl.as_dtype(inp["grid"], dtype)}
    if w.kind == "resize":
        return {"X": wl.as_dtype(wl.make_resize_inputs(w, seed=seed)["X"], dtype)}
    return {k: wl.as_dtype(v, dtype) for k, v in wl.make_deform_inputs(w, seed=seed).items()}


def replica_seed(w, rank):
    """Rank r of a replicated run draws its own images: the workload's seed + r."""
    return w.seed + rank


def max_over_ranks(x, world, device=None):
    """The largest per-rank value over all ranks (the slowest replica sets the job's
    time); x itself on one rank.  device is where the collective's tensor lives
    (a CUDA device under NCCL, None for the CPU under gloo)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(outputs_per_rank, world, ms):
    """Whole-job throughput: every replica's outputs over the slowest replica's time."""
    return outputs_per_rank * world / (ms * 1e-3)


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples for one GPU, with timestamps."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        window = "timed region"
        if len(inside) < 2:   # a short region: keep the samples around it
            inside = [p for t, p in self.samples if t0 - 1.0 <= t <= t1 + 1.0]
            window = "timed region +- 1 s"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "no samples"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(inside[0][1]), "reasons": reasons, "samples": len(inside),
                "window": window}


# --------------------------------------------------------------- workloads

class Case:
    """One workload on one device: inputs in HBM, a launch closure, byte/flop counts."""

    def __init__(self, name, dtype, device, mode=None, rank=0, workspace=False):
        import torch
        self.w = wl.WORKLOADS[name]
        self.name, self.dtype, self.device = name, dtype, device
        self.mode = mode or self.w.mode
        self.ws = None
        self.launches = 1   # kernels per step
        w = self.w
        eb = DT_BYTES[dtype]
        import spatial_transformer_sampling_gb300 as gs
        self.gs = gs
        self.host = host_inputs(w, dtype, replica_seed(w, rank))
        if w.kind == "affine_sample":
            self.size = [w.x_shape[0], w.x_shape[1], *w.out_spatial]
            self.outputs = int(np.prod(self.size))
            if w.r == 2:
                self.kernel_tag = f"band_kernel<{DT_SHORT[dtype]},{self.mode}>"
            elif self.mode != "cubic":
                # the TMA-staged kernel (inputs 16-byte aligned, rows in whole 16-byte runs)
                self.kernel_tag = f"vol_tma_kernel<{DT_SHORT[dtype]},{self.mode}>"
            else:
                self.kernel_tag = f"sample_kernel<{DT_SHORT[dtype]},{w.r},{self.mode},affine>"
        elif w.kind == "grid_sample":
            self.outputs = w.x_shape[0] * w.x_shape[1] * int(np.prod(w.out_spatial))
            self.kernel_tag = f"sample_kernel<{DT_SHORT[dtype]},{w.r},{self.mode},grid>"
            if workspace:
                nbytes = gs.gs_grid_sample_workspace_size(w.x_shape, w.out_spatial,
                                                          getattr(torch, dtype))
                if nbytes:
                    self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
                    slot = w.x_shape[1] * (int(np.prod(w.x_shape[2:])) + 1) * eb
                    per = nbytes // slot
                    self.launches = 2 * (-(-w.x_shape[0] // per))   # copy + sample per chunk
                    self.kernel_tag = f"nhwc_sample_kernel<{DT_SHORT[dtype]},{w.r},{self.mode}>"
        elif w.kind == "resize":
            self.outputs = w.x_shape[0] * w.x_shape[1] * int(np.prod(w.out_spatial))
            self.resize_kw = dict(scales=list(w.extra["scales"]), mode=self.mode,
                                  antialias=w.extra["antialias"])
            # the kernel gs_resize takes for these shapes: 16-bit types with an even
            # output width up to 512 pair outputs; fp32 with at most four taps per
            # output stays on the row kernel; the rest (antialias) is staged
            if eb == 2 and w.out_spatial[-1] % 2 == 0 and w.out_spatial[-1] <= 512:
                kname = "resize_pair_kernel"
            elif eb == 4 and not w.extra["antialias"]:
                kname = "resize_rows_kernel"
            else:
                kname = "resize_stage_kernel"
            self.kernel_tag = f"{kname}<{DT_SHORT[dtype]},{w.r},{self.mode}>"
        else:
            N, C, H, W_ = w.x_shape
            oH = (H + w.pads[0] + w.pads[2] - (w.kernel[0] - 1) - 1) // w.strides[0] + 1
            oW = (W_ + w.pads[1] + w.pads[3] - (w.kernel[1] - 1) - 1) // w.strides[1] + 1
            self.outputs = N * w.oc * oH * oW
            self.flops = 2.0 * N * oH * oW * w.oc * (C // w.group) * w.kernel[0] * w.kernel[1]
            # the kernels the plain call takes for this shape (3x3, C and oC multiples
            # of 16, group 1): windowed FFMA for fp32, staged tcgen05 for 16-bit types
            self.kernel_tag = (f"deform_f32_kernel<{DT_SHORT[dtype]}>" if dtype == "float32"
                               else f"deform_st_kernel<{DT_SHORT[dtype]}>")
            if workspace:
                a = gs.deform_attrs(w.kernel, w.pads, w.strides, w.dilations, w.group,
                                    w.offset_group)
                nbytes = gs.gs_deform_conv_workspace_size(w.x_shape, w.oc, a, getattr(torch, dtype))
                if nbytes:
                    self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
                    self.launches = 2   # pack W with copy X, then sample + contract
                    self.kernel_tag = f"deform_tc_nhwc<{DT_SHORT[dtype]}>"
        self.dev = {k: v.to(device) for k, v in self.host.items()}
        self.out = torch.empty(self._out_shape(), dtype=self.dev["X"].dtype, device=device)
        # algorithmic bytes: every input read once, the output written once
        self.bytes = sum(t.numel() for t in self.host.values()) * eb + self.outputs * eb

    def _out_shape(self):
        w = self.w
        if w.kind == "affine_sample":
            return self.size
        if w.kind in ("grid_sample", "resize"):
            return list(w.x_shape[:2]) + list(w.out_spatial)
        N, C, H, W_ = w.x_shape
        return [N, w.oc, H, W_]

    def run(self, dev=None, out=None):
        d = dev or self.dev
        out = self.out if out is None else out
        w = self.w
        if w.kind == "affine_sample":
            return self.gs.gs_affine_sample(d["theta"], self.size, d["X"], self.mode,
                                            w.padding_mode, w.align_corners, w.cubic_coeff_a,
                                            out=out)
        if w.kind == "grid_sample":
            return self.gs.gs_grid_sample(d["X"], d["grid"], self.mode, w.padding_mode,
                                          w.align_corners, w.cubic_coeff_a, out=out,
                                          workspace=self.ws)
        if w.kind == "resize":
            return self.gs.gs_resize(d["X"], out=out, **self.resize_kw)
        return self.gs.gs_deform_conv(d["X"], d["W"], d["offset"], d["B"], d["mask"],
                                      kernel_shape=w.kernel, pads=w.pads, strides=w.strides,
                                      dilations=w.dilations, group=w.group,
                                      offset_group=w.offset_group, out=out, workspace=self.ws)


def flush_l2(buf):
    """Write then read a buffer larger than L2 (leaves L2 clean and cold for the step)."""
    buf.zero_()
    return buf.amax()


def time_steps(case, steps, warmup, flush, barrier=None):
    """Per-step CUDA-event durations (ms) of the hot path, L2 flushed before each step
    (flush None: steps back to back, warm L2)."""
    import torch
    stream = torch.cuda.current_stream(case.device)
    for _ in range(warmup):
        if flush is not None:
            flush_l2(flush)
        case.run()
    torch.cuda.synchronize(case.device)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if barrier:
        barrier()
    torch.cuda.synchronize(case.device)
    t0 = time.time()
    for i in range(steps):
        if flush is not None:
            flush_l2(flush)
        starts[i].record(stream)
        case.run()
        ends[i].record(stream)
    torch.cuda.synchronize(case.device)
    if barrier:
        barrier()
    t1 = time.time()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], t0, t1


def time_e2e(case, steps, warmup):
    """Host buffers in, host buffer out, through the library's host-streaming call:
    pinned H2D copies, the kernels and the D2H copy of Y, chunked over the batch so
    copies in both directions overlap the kernels.  Per step."""
    import torch
    gs = case.gs
    w = case.w
    stream = torch.cuda.current_stream(case.device)
    pinned = {k: v.pin_memory() for k, v in case.host.items()}
    out_host = torch.empty(case.out.shape, dtype=case.out.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pinned.values())
    d2h = out_host.numel() * out_host.element_size()
    streamer = gs.HostStreamer(case.device)

    if w.kind == "affine_sample":
        def step():
            gs.gs_affine_sample_from_host(pinned["theta"], case.size, pinned["X"], case.mode,
                                          w.padding_mode, w.align_corners, w.cubic_coeff_a,
                                          out=out_host, streamer=streamer)
    elif w.kind == "grid_sample":
        def step():
            gs.gs_grid_sample_from_host(pinned["X"], pinned["grid"], case.mode, w.padding_mode,
                                        w.align_corners, w.cubic_coeff_a, out=out_host,
                                        streamer=streamer,
                                        workspace="auto" if case.ws is not None else None)
    elif w.kind == "resize":
        def fn(x, out):
            return gs.gs_resize(x, out=out, **case.resize_kw)

        def step():
            streamer.run(fn, [pinned["X"]], out_host, [0])
    else:
        d = {k: torch.empty_like(v, device=case.device) for k, v in case.host.items()}

        def step():
            for k in d:
                d[k].copy_(pinned[k], non_blocking=True)
            case.run(dev=d)
            out_host.copy_(case.out, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(case.device)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        step()
    e.record(stream)
    e.synchronize()
    ms = s.elapsed_time(e) / steps
    return ms, h2d, d2h


# fp32 FMA peak of the CUDA cores: 152 SMs x 128 fp32 lanes x 2 flops x 2.07 GHz
# (the GB300's SM count and maximum SM clock); the bound of the fp32 DeformConv
# kernel, whose contraction runs on FFMA.
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def roofline_for(case, ms, pk):
    if case.w.kind == "deform_conv" and case.dtype == "float32":
        achieved = case.flops / (ms * 1e-3) / 1e12
        return {"bound": "alu", "achieved": round(achieved, 3), "peak": round(FP32_ALU_TFLOPS, 1),
                "unit": "TFLOP/s", "frac": round(achieved / FP32_ALU_TFLOPS, 4),
                "traffic": recorded_traffic(case.kernel_tag, case.name, case.dtype),
                "peak_source": "derived: 152 SMs x 128 fp32 FMA/clk x 2 x 2.07 GHz"}
    if case.w.kind == "deform_conv":
        achieved = case.flops / (ms * 1e-3) / 1e12
        peak = pk["bf16_tflops"]
        return {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "traffic": recorded_traffic(case.kernel_tag, case.name, case.dtype),
                "peak_source": pk["source"]}
    achieved = case.bytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / pk["hbm_gbs"], 4),
            "traffic": recorded_traffic(case.kernel_tag, case.name, case.dtype),
            "algorithmic_bytes": case.bytes, "peak_source": pk["source"]}


# ------------------------------------------------------------- CPU oracle

def oracle_sample(case, budget_s=12.0, threads=None):
    """Time the oracle on a bounded slice of the workload: whole images, doubling the
    count (and cycling through the batch) until about budget_s of CPU time is spent.
    threads: OpenMP threads (default every host core, whatever OMP_NUM_THREADS says)."""
    import oracle
    w = case.w
    threads = threads or oracle.num_procs()
    oracle.set_num_threads(threads)
    if not hasattr(case, "host64"):   # widen once; each step reuses it
        case.host64 = {k: wl.widened(v) for k, v in case.host.items()}
    h = case.host64
    N = w.x_shape[0]
    total_t, total_out, images = 0.0, 0, 0
    n_img = 1
    while total_t < budget_s:
        start = images % N
        n = min(n_img, N - start)
        sl = slice(start, start + n)
        t = time.perf_counter()
        if w.kind == "affine_sample":
            size = [n] + case.size[1:]
            Y = oracle.affine_sample(h["theta"][sl], size, h["X"][sl], case.mode, w.padding_mode,
                                     w.align_corners, w.cubic_coeff_a)
        elif w.kind == "grid_sample":
            Y = oracle.grid_sample(h["X"][sl], h["grid"][sl], case.mode, w.padding_mode,
                                   w.align_corners, w.cubic_coeff_a)
        elif w.kind == "resize":
            Y = oracle.resize(h["X"][sl], **case.resize_kw)
        else:
            Y = oracle.deform_conv(h["X"][sl], h["W"], h["offset"][sl], h["B"], h["mask"][sl],
                                   kernel_shape=w.kernel, pads=w.pads, strides=w.strides,
                                   dilations=w.dilations, group=w.group,
                                   offset_group=w.offset_group)
        total_t += time.perf_counter() - t
        total_out += Y.size
        images += n
        n_img = min(2 * n_img, N)
    return {"value": total_out / total_t, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{images} images of {case.name} ({total_out} outputs, first images of the "
                      f"batch, cycling; {total_t:.1f} s of fp64 C on {threads} OpenMP threads)"}


# ------------------------------------------------------------------- main

def workload_desc(case):
    w = case.w
    if w.kind == "affine_sample":
        return (f"{case.name}: fused AffineGrid+GridSample {w.r}-D, theta ({w.x_shape[0]},{w.r},"
                f"{w.r + 1}) = identity + N(0,{w.theta_noise}), X {tuple(w.x_shape)} ~ N(0,1) "
                f"{case.dtype}, out {tuple(w.out_spatial)}, {case.mode}, {w.padding_mode}, "
                f"align_corners={w.align_corners}")
    if w.kind == "grid_sample":
        ws = getattr(case, "ws", None)
        via = (f"; gs_grid_sample_ws, channel-last workspace {ws.numel() / 2**20:.0f} MiB"
               if ws is not None else "")
        return (f"{case.name}: GridSample {w.r}-D, X {tuple(w.x_shape)} {w.x_dist}, grid "
                f"({w.x_shape[0]},{','.join(map(str, w.out_spatial))},{w.r}) {w.grid_dist}, "
                f"{case.dtype}, {case.mode}, {w.padding_mode}, align_corners={w.align_corners}"
                f"{via}")
    if w.kind == "resize":
        return (f"{case.name}: Resize {w.r}-D, X {tuple(w.x_shape)} ~ N(0,1) {case.dtype}, scales "
                f"{tuple(w.extra['scales'])}, {case.mode}, half_pixel, "
                f"antialias={w.extra['antialias']}, out {tuple(w.out_spatial)}")
    ws = getattr(case, "ws", None)
    via = (f"; gs_deform_conv_ws, channel-last workspace {ws.numel() / 2**20:.1f} MiB"
           if ws is not None else "")
    return (f"{case.name}: DeformConv 2-D, X {tuple(w.x_shape)}, W ({w.oc},{w.x_shape[1]},3,3), "
            f"pads 1, stride 1, offset/mask from N(0,1), {case.dtype}{via}")


def main():
    args = parse()
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        return reference_arm(args, rank, world)

    import torch
    import torch.distributed as dist
    import __graft_entry__
    __graft_entry__.build()

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    barrier = None
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
        barrier = dist.barrier
    pk = peaks()
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=device)

    case = Case(args.workload, args.dtype, device, args.mode, rank=rank,
                workspace=args.workspace)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        time.sleep(0.6)   # let nvidia-smi start reporting before the timed region
    per_step, t0, t1 = time_steps(case, args.steps, args.warmup, flush, barrier)
    clocks = sampler.summary(t0, t1) if sampler else None
    if sampler:
        sampler.stop()
    ms = sum(per_step) / len(per_step)
    ms_max = max_over_ranks(ms, world, device)
    value = job_value(case.outputs, world, ms_max)
    ms_median = max_over_ranks(statistics.median(per_step), world, device)

    # warm L2: the same steps back to back with no flush in between
    warm_steps, _, _ = time_steps(case, min(args.steps, 500), 5, None, barrier)
    warm_ms = max_over_ranks(sum(warm_steps) / len(warm_steps), world, device)

    e2e_ms, h2d, d2h = time_e2e(case, max(5, min(50, args.steps // 10)), 3)
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    e2e_value = job_value(case.outputs, world, e2e_ms)

    extra = []
    if rank == 0 and not args.no_extra:
        for name, dt, mode, ws in (
                ("stn2d", "bfloat16", None, False), ("stn3d", "float32", None, False),
                ("gs2d_cubic", "float32", "cubic", False), ("gs2d_cubic", "float16", "cubic", False),
                ("gs2d_cubic", "float32", "nearest", False),
                ("gs2d_cubic", "float16", "nearest", False),
                ("gs2d_cubic", "float32", "cubic", True), ("gs2d_cubic", "float16", "cubic", True),
                ("gs2d_cubic", "float32", "nearest", True),
                ("gs2d_cubic", "float16", "nearest", True),
                ("gs2d_small", "float32", None, False),
                ("deform2d", "float32", None, False), ("deform2d", "bfloat16", None, False),
                ("deform2d", "bfloat16", None, True),
                ("resize2d_up", "float32", None, False), ("resize2d_up", "bfloat16", None, False),
                ("resize2d_aa", "float32", None, False)):
            if (name, dt, mode, ws) == (args.workload, args.dtype, args.mode, args.workspace):
                continue
            c2 = Case(name, dt, device, mode, workspace=ws)
            st, _, _ = time_steps(c2, args.extra_steps, 5, flush)
            m2 = sum(st) / len(st)
            extra.append({"workload": workload_desc(c2), "dtype": DT_SHORT[dt],
                          "ms_per_step": round(m2, 5), "value": round(c2.outputs / (m2 * 1e-3), 1),
                          "unit": UNIT, "kernel": c2.kernel_tag, "launches_per_step": c2.launches,
                          "roofline": roofline_for(c2, m2, pk)})
            del c2
            torch.cuda.empty_cache()

    cpu = oracle_sample(case) if rank == 0 and world == 1 else None   # N=1 only
    if cpu is not None:
        # the same oracle on one core (a shorter sample), beside the all-core figure
        one = oracle_sample(case, budget_s=min(args.sample_seconds, 12.0) / 4, threads=1)
        cpu["single_thread"] = {"value": one["value"], "unit": one["unit"], "cores": 1,
                                "sample": one["sample"]}
    if world > 1:
        dist.barrier()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 5),
            "ms_median": round(ms_median, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DT_SHORT[args.dtype], "data": "synthetic (seeded PCG64; no dataset)",
            "config": {"workload": workload_desc(case),
                       "l2": "flushed before every step: 512 MiB written then read (outside the timed interval)",
                       "parallelism": f"replicas x{world} (independent images, no collective)"},
            "roofline": roofline_for(case, ms, pk),
            "warm_l2": {"value": round(job_value(case.outputs, world, warm_ms), 1), "unit": UNIT,
                        "ms_per_step": round(warm_ms, 5), "steps": len(warm_steps),
                        "note": "no flush between steps (inputs may stay in L2)"},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4)},
            "gpu_launches": args.steps * case.launches,
            "clocks": clocks,
            "kernel": case.kernel_tag,
            "src_sha": kernel_source_sha(case.kernel_tag),
            "workloads": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def reference_arm(args, rank, world):
    """The CPU oracle as the reference implementation (rank 0 only)."""
    if rank != 0:
        return
    w = wl.WORKLOADS[args.workload]

    class HostCase:
        pass

    case = HostCase()
    case.w, case.name, case.dtype = w, args.workload, args.dtype
    case.mode = args.mode or w.mode
    case.host = host_inputs(w, args.dtype, replica_seed(w, 0))
    if w.kind == "affine_sample":
        case.size = [w.x_shape[0], w.x_shape[1], *w.out_spatial]
    elif w.kind == "resize":
        case.resize_kw = dict(scales=list(w.extra["scales"]), mode=case.mode,
                              antialias=w.extra["antialias"])
    # the whole run stays within a few minutes: ~150 s of oracle time in all
    per_step_budget = min(args.sample_seconds, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(case, budget_s=per_step_budget / 4)
    vals = []
    last = None
    for _ in range(args.steps):
        last = oracle_sample(case, budget_s=per_step_budget)
        vals.append(last["value"])
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": DT_SHORT[args.dtype], "data": "synthetic (seeded PCG64; no dataset)",
        "config": {"workload": workload_desc(case),
                   "note": "each step times the oracle on a bounded slice of whole images"},
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": last["cores"],
                         "kind": "oracle", "sample": last["sample"]},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
