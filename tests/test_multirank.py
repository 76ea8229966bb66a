"""The multi-GPU path's host logic with two ranks on the CPU (gloo).

Decode and prefill shard by sequence or query chunk: every rank runs its own
batch from its own seed with no collective on the data path, and the job's time
is the slowest rank's (a max over ranks). These tests run that logic in two
processes, the way torchrun starts one process per GPU.
"""
from __future__ import annotations

import json
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    import synth

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        env = bench.dist_env()
        # per-rank step times: the job's time is the slowest rank's
        mx = bench.reduce_max([1.0 + rank, 10.0 - 3.0 * rank], "cpu")
        # each rank's own batch: same shapes, different data
        seed = bench.shard_seed(7, rank)
        inp = synth.decode_inputs([64, 33], 1, "bf16", seed)
        digest = int(np.asarray(inp.q, np.uint64).sum() % (1 << 61))
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"env": list(env), "max": mx, "seed": seed, "digest": digest,
                       "q_shape": list(inp.q.shape)}, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_shard_and_take_the_slowest(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(world)]
    for i in range(world):
        assert r[i]["env"] == [i, world, i]
        assert r[i]["max"] == [2.0, 10.0]  # max over ranks of (1 + rank, 10 - 3 rank)
    assert r[0]["seed"] != r[1]["seed"]
    assert r[0]["q_shape"] == r[1]["q_shape"]
    assert r[0]["digest"] != r[1]["digest"]


def test_single_process_values_pass_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max([3.5, 1.0], "cpu") == [3.5, 1.0]
    assert bench.dist_env()[1] >= 1


def test_job_rate_is_the_whole_job():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 64 queries in 0.5 ms (the slower rank) = 256000 queries/s
    assert bench.job_rate(64, 2, 0.5) == pytest.approx(256000.0)
    assert bench.shard_seed(7, 0) == 7 and bench.shard_seed(7, 3) == 3007
