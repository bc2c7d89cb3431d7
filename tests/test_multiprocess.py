"""The N > 1 benchmark path on the CPU: two gloo ranks (no GPU).

The forward pass shards by (batch, KV head) with no exchange step, so N GPUs
run N independent replicas; the only cross-rank operations are the bench's
barrier and the max over ranks of the timed durations. Both are checked here
with world size 2, and `bench.py --impl reference` is launched under torchrun
(rank 0 alone runs and prints one JSON line, the other rank exits 0).
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), GQA_BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    m = bench.max_over_ranks(1.5 + rank, w, torch.device("cpu"))
    out[rank] = m
    torch.distributed.destroy_process_group()


def test_max_over_ranks_and_barrier_two_gloo_ranks():
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ, GQA_BENCH_BACKEND="gloo", CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "prompt_f32_b1_s16"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
