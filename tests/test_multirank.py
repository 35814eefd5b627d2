"""World-size-2 gloo checks of the multi-rank path on CPU: each rank draws its own batch of
sequences (no data-path exchange), the oracle's per-rank results are independent of the
other rank, and the benchmark's whole-job aggregation sums bytes and takes the slowest
rank's time."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    import workloads

    wl = workloads.shard("tiny", rank, world)
    r = oracle.decode_workload(wl)
    np.save(os.path.join(out_dir, f"out{rank}.npy"), r["out"])
    np.save(os.path.join(out_dir, f"q{rank}.npy"), wl.query.float().numpy())
    step_bytes = float(wl.algorithmic_bytes())
    ms = 1.0 + rank  # rank 1 is the slow one
    tot, slowest = bench.combine_ranks(step_bytes, ms, torch.device("cpu"), world)
    allb = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(allb, torch.tensor([step_bytes], dtype=torch.float64))
    assert tot == sum(float(x) for x in allb)
    assert slowest == float(world)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_shards_and_aggregation(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    q0, q1 = np.load(tmp_path / "q0.npy"), np.load(tmp_path / "q1.npy")
    assert not np.array_equal(q0, q1), "ranks must draw different batches"
    # a rank's result depends only on its own shard: recompute rank 1's shard alone
    import oracle
    import workloads

    r1 = oracle.decode_workload(workloads.shard("tiny", 1, 2))
    assert np.array_equal(r1["out"], np.load(tmp_path / "out1.npy"))
