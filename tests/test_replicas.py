"""The replicated (N > 1) path of the benchmark, on the CPU with two gloo ranks.

Sampling shards by image with no exchange step, so a run on N GPUs is N
independent replicas.  Each rank draws its own images (the workload's seed +
rank) and times its own replica; the job's time is the slowest rank's, and the
job's throughput counts every rank's outputs.  The one collective is the
max over ranks of the timings.  With GPUs that collective runs on NCCL;
here the same helpers run on gloo, and the launcher path (torchrun, rank 0
prints the line, the other ranks print nothing) runs end to end through the
reference arm, which needs no GPU.
"""
import dataclasses
import hashlib
import json
import multiprocessing
import os
import socket
import subprocess
import sys
import time

import numpy as np
import pytest

import bench
from spatial_transformer_sampling_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _digest(host):
    h = hashlib.sha256()
    for k in sorted(host):
        h.update(k.encode() + host[k].contiguous().numpy().tobytes())
    return h.hexdigest()


def _small(name):
    """A workload with its batch cut to two images (the draw order is unchanged)."""
    w = wl.WORKLOADS[name]
    return dataclasses.replace(w, x_shape=(2,) + tuple(w.x_shape[1:]))


def _rank_main(rank, port, q):
    """One gloo rank: the reductions bench.py applies to its per-rank timings, and
    the inputs this rank's replica would draw."""
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    try:
        dist.init_process_group("gloo", rank=rank, world_size=WORLD)
        out = {"rank": rank}
        # per-rank step times: the slowest replica sets the job's time
        out["ms_max"] = bench.max_over_ranks([3.0, 5.0][rank], WORLD)
        out["ms_max_swapped"] = bench.max_over_ranks([7.5, 2.0][rank], WORLD)
        # a barrier-bracketed interval in which rank 1 does twice the work
        dist.barrier()
        t0 = time.perf_counter()
        time.sleep(0.05 * (rank + 1))
        dist.barrier()
        out["wall_ms"] = bench.max_over_ranks((time.perf_counter() - t0) * 1e3, WORLD)
        out["value"] = bench.job_value(1000, WORLD, out["ms_max"])
        # each replica's inputs
        out["digests"] = {}
        for name in ("gs2d_small", "stn2d", "deform2d", "resize2d_up"):
            w = _small(name)
            out["digests"][name] = _digest(bench.host_inputs(w, "float32",
                                                             bench.replica_seed(w, rank)))
        gathered = [None] * WORLD
        dist.all_gather_object(gathered, out["digests"])
        out["all_digests"] = gathered
        dist.barrier()
        dist.destroy_process_group()
        q.put(out)
    except BaseException as e:   # report, do not hang the parent
        q.put({"rank": rank, "error": repr(e)})


@pytest.fixture(scope="module")
def rank_results():
    ctx = multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in range(WORLD):
            r = q.get(timeout=180)
            res[r["rank"]] = r
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
                p.join()
    for r in res.values():
        assert "error" not in r, r
    return res


def test_job_time_is_the_slowest_rank(rank_results):
    for r in range(WORLD):
        assert rank_results[r]["ms_max"] == 5.0
        assert rank_results[r]["ms_max_swapped"] == 7.5


def test_barrier_interval_covers_the_longest_rank(rank_results):
    # rank 1 slept 100 ms inside the barriers; every rank reports at least that
    for r in range(WORLD):
        assert rank_results[r]["wall_ms"] >= 100.0
    assert rank_results[0]["wall_ms"] == rank_results[1]["wall_ms"]


def test_job_value_counts_every_replica(rank_results):
    # 1000 outputs on each of 2 ranks in 5 ms (the slower rank) = 400,000 per second
    for r in range(WORLD):
        assert rank_results[r]["value"] == pytest.approx(2 * 1000 / 5e-3)


def test_replicas_draw_their_own_inputs(rank_results):
    all_d = rank_results[0]["all_digests"]
    assert all_d == rank_results[1]["all_digests"]
    for name in all_d[0]:
        assert all_d[0][name] != all_d[1][name], name
        # rank r's inputs are exactly the workload's draw at seed + r
        for r in range(WORLD):
            w = _small(name)
            assert all_d[r][name] == _digest(bench.host_inputs(w, "float32", w.seed + r))


def test_rank0_inputs_are_the_single_gpu_inputs():
    w = wl.WORKLOADS["gs2d_small"]
    inp = wl.make_grid_sample_inputs(w)
    host = bench.host_inputs(w, "float32", bench.replica_seed(w, 0))
    np.testing.assert_array_equal(host["X"].numpy(), inp["X"].astype(np.float32))
    np.testing.assert_array_equal(host["grid"].numpy(), inp["grid"].astype(np.float32))


def test_one_rank_needs_no_process_group():
    assert bench.max_over_ranks(4.25, 1) == 4.25
    assert bench.job_value(10, 1, 2.0) == pytest.approx(5000.0)


def test_reference_arm_under_torchrun_prints_one_line(oracle_mod):
    """bench.py --impl reference launched like the N=2 job: rank 0 alone times
    the oracle and prints one JSON line; rank 1 exits 0 without work."""
    port = _free_port()
    env = dict(os.environ)
    env.pop("OMP_NUM_THREADS", None)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           str(WORLD), "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", str(WORLD),
           "--steps", "2", "--warmup", "0", "--workload", "gs2d_small", "--sample-seconds", "0.2"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == WORLD and d["steps"] == 2
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    # the oracle ran on every host core, not the one thread torchrun gives each rank
    assert d["cpu_baseline"]["cores"] == oracle_mod.num_procs()
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_do_no_work():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "gs2d_small", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
