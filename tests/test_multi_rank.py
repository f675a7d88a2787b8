"""The multi-GPU path of the benchmark is "replicas only": every rank runs the
layer on its own tokens, and the only cross-rank steps are a barrier and the
max of the step times.  These tests run that host logic with two gloo ranks
on the CPU (no GPU): the rank environment, the max over ranks, the
whole-job weak-scaling throughput, and the reference arm printing from
rank 0 only."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    ws, r, local = bench.dist_env()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, ws, torch.device("cpu"))
    value = bench.job_tokens_per_s(ws, 8192, ms)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, ws, r, local, ms, value))


def test_max_over_ranks_and_job_throughput_with_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ws, r, local, ms, value in out:
        assert (ws, r, local) == (world, rank, rank)
        assert ms == 15.0                       # the slowest rank's step time, on every rank
        assert value == pytest.approx(world * 8192 / 0.015)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.job_tokens_per_s(1, 1000, 2.0) == pytest.approx(500000.0)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_from_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload",
                        "tiny_fp32_T256_h128_E8_K2_F512_gelu", "--sample-tokens", "16"],
                       capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if rank == 0:
        assert len(lines) == 1
        d = json.loads(lines[0])
        assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
        assert d["cpu_baseline"]["kind"] == "oracle"
    else:
        assert lines == []
