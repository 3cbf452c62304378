"""The multi-rank path on CPU: two gloo ranks each run their share of a
batch (through the oracle, standing in for the GPU kernels) and the gathered
result equals the unsharded batch; timings reduce to the slowest rank."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from chunk_wise_weight_gb300.shard import max_over_ranks, shard_range


@pytest.mark.parametrize("total,world", [(4, 2), (5, 2), (1, 3), (8, 8), (7, 3)])
def test_shard_range_partitions(total, world):
    seen = []
    sizes = []
    for r in range(world):
        a, b = shard_range(total, world, r)
        seen.extend(range(a, b))
        sizes.append(b - a)
    assert seen == list(range(total))
    assert max(sizes) - min(sizes) <= 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from chunk_wise_weight_gb300 import make_inputs
        inp = make_inputs(4, 8, 3, 5, seed=77)
        a, b = shard_range(4, world, rank)
        mine = dict(inp)
        mine["H"], mine["X0"] = inp["H"][a:b], inp["X0"][a:b]
        O = torch.from_numpy(oracle.forward(mine, 0.4, 4)["O"])
        parts = [torch.zeros(2, 8, 3, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(parts, O)
        slowest = max_over_ranks(float(rank + 1))
        if rank == 0:
            full = oracle.forward(inp, 0.4, 4)["O"]
            np.save(os.path.join(result_dir, "gathered.npy"), torch.cat(parts).numpy())
            np.save(os.path.join(result_dir, "full.npy"), full)
            np.save(os.path.join(result_dir, "slowest.npy"), np.array([slowest]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_the_batch(tmp_path):
    mp.spawn(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    np.testing.assert_array_equal(np.load(tmp_path / "gathered.npy"), np.load(tmp_path / "full.npy"))
    assert float(np.load(tmp_path / "slowest.npy")[0]) == 2.0


def test_max_over_ranks_without_group():
    assert max_over_ranks(3.5) == 3.5
