"""The multi-process (N > 1) path of bench.py, on CPU with the gloo backend.

The method shards by request with no exchange step: every rank runs its own
replica of the step on independent requests, the ranks meet only at a barrier
and in a max-reduction of their elapsed times, and rank 0 alone prints the
result line.  These tests run world_size-2 process groups on the CPU.
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


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from compressed_kv_attention_gated_gb300 import synth

    dist.init_process_group("gloo", rank=rank, world_size=ws)
    mine = 10.0 + 5.0 * rank  # elapsed ms of this rank
    m = bench._max_over_ranks(mine, ws, torch.device("cpu"))
    bench._barrier(ws)
    d = synth.pooled_decode("cpu", seed=bench.replica_seed(rank), B=8)
    q.put((rank, m, d["key"].float().sum().item()))
    dist.destroy_process_group()


def test_two_ranks_max_and_independent_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]  # both ranks see the slowest rank's time
    assert res[0][2] != res[1][2]  # replicas draw different requests


def test_whole_job_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.whole_job_value(1000, 1, 10, 1000.0) == 10000.0
    assert bench.whole_job_value(1000, 4, 10, 1000.0) == 40000.0


def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["value"] > 0
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["cpu_baseline"]["kind"] == "oracle"
