"""Host logic of the multi-rank bench on CPU: two gloo ranks (no GPU).

Each rank runs its own batch (the path shards by sequence with no exchange), so the only cross-rank
steps are the barrier and the max-reduction of the step time; the ranks draw different inputs; the
reference arm runs on rank 0 only.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    from spec_decode_verify_gb300 import workloads as wl

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(dist, torch.device("cpu"))
        step_us = 10.0 * (rank + 1)
        got = bench.reduce_max(dist, step_us, torch.device("cpu"))
        w = wl.WORKLOADS[wl.WORKLOAD_ORDER[1]]
        x = wl.make_inputs(w, seed=w.seed + 1009 * rank)["x"]
        xs = [torch.zeros_like(x.float()) for _ in range(world)]
        dist.all_gather(xs, x.float().contiguous())
        out[rank] = (got, bool(torch.equal(xs[0], xs[1])))
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_and_distinct_batches():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        if p.is_alive():
            p.kill()
            pytest.fail("rank did not finish")
        assert p.exitcode == 0
    assert out[0][0] == pytest.approx(20.0) and out[1][0] == pytest.approx(20.0)
    assert out[0][1] is False  # each rank draws its own batch


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    import bench
    from spec_decode_verify_gb300 import workloads as wl

    class Args:
        steps, warmup = 1, 3

    # rank 1 of 2 returns 0 immediately and prints nothing
    assert bench.run_reference(Args, wl.WORKLOADS[bench.wl.BENCH_WORKLOAD], 2, 1) == 0


def _bench_env():
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    env["CUDA_VISIBLE_DEVICES"] = ""  # the CPU path of the launcher (gloo), even on a GPU host
    return env


def test_bench_gpus_n_launches_n_ranks():
    """`bench.py --gpus 2` without a launcher starts two ranks itself (torch.distributed.run, gloo
    on CPU): the one JSON line comes from rank 0 and reports n_gpus 2 (the reference arm, which
    runs on the CPU)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3", "--workload", "n1_t2_dim512_w4_f32_dense"],
                       capture_output=True, text=True, env=_bench_env(), timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    assert lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"


def test_bench_gpus_must_match_world_size():
    """Under a launcher, --gpus must equal WORLD_SIZE (an N-GPU line never comes from fewer ranks)."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = _bench_env()
    env.update(WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3", "--workload", "n1_t2_dim512_w4_f32_dense"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode != 0 and "does not match WORLD_SIZE" in r.stderr
