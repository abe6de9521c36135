"""The N > 1 host logic of bench.py, run as two gloo ranks on the CPU.

With N GPUs the bench runs one process per GPU, each on its own shard of the
workload (weak scaling, no data-path collective); the only collectives are the
barrier and the max over ranks of the step time, and rank 0 alone prints.
These tests exercise exactly that logic with the gloo backend, no GPU.
"""
from __future__ import annotations

import argparse
import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import numpy as np
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, str(ROOT))
    import torch
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (world, rank, rank)
    slowest = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
    e2e = bench.max_over_ranks(10.0 - rank, world, torch.device("cpu"))
    args = argparse.Namespace(workload="kv_cache", layers=1)
    shard = bench.workload_arrays(args, rank)
    dist.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"slowest": slowest, "e2e": e2e, "tensors": len(shard),
                   "head": shard[0][:64].tolist(), "head_v": shard[1][:64].tolist()}, f)
    dist.destroy_process_group()


def test_two_ranks_take_the_max_and_hold_disjoint_shards(tmp_path):
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    r = [json.loads((tmp_path / f"rank{k}.json").read_text()) for k in range(2)]
    # every rank sees the slowest rank's time
    assert r[0]["slowest"] == r[1]["slowest"] == 2.5
    assert r[0]["e2e"] == r[1]["e2e"] == 10.0
    # weak scaling: each rank its own cache (layers offset by rank), same shape
    from weight_compression_codec_gb300 import inputs

    assert r[0]["tensors"] == r[1]["tensors"] == 2
    for k in range(2):
        assert r[k]["head"] == inputs.kv_cache_tensor(k, 0)[:64].tolist()
        assert r[k]["head_v"] == inputs.kv_cache_tensor(k, 1)[:64].tolist()
    assert not np.array_equal(np.array(r[0]["head"]), np.array(r[1]["head"]))


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), str(ROOT / "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "paged_kv"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
