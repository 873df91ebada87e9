"""Two-rank data-parallel host logic on CPU (gloo): no GPU.

Each rank takes a block of whole response groups, counts its valid rows and
all-reduces the count; both ranks must derive the same global token-mean
scale, and the shards must cover every group exactly once.
"""

import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from precision_off_policy_gb300 import dp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, lengths, group_size, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        n_groups = len(lengths) // group_size
        groups = dp.shard_groups(n_groups, world, rank)
        local = sum(int(lengths[g * group_size + i]) for g in groups for i in range(group_size))
        total = dp.global_valid_tokens(local)
        out[rank] = (list(groups), local, total, dp.token_mean_scale(total))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_ranks_agree_on_the_global_token_scale(world):
    rng = np.random.default_rng(0)
    group_size = 4
    lengths = rng.integers(64, 513, size=7 * group_size)  # 7 groups: uneven split
    mgr = mp.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_worker, args=(world, port, lengths, group_size, out), nprocs=world, join=True,
                       start_method="spawn")
    res = [out[r] for r in range(world)]
    covered = sorted(g for r in res for g in r[0])
    assert covered == list(range(7))
    assert res[0][2] == res[1][2] == int(lengths.sum())
    assert res[0][1] + res[1][1] == int(lengths.sum())
    assert res[0][3] == res[1][3] == float(np.float32(1.0 / int(lengths.sum())))


def test_shard_groups_edge_cases():
    assert list(dp.shard_groups(0, 2, 1)) == []
    assert [len(dp.shard_groups(5, 3, r)) for r in range(3)] == [2, 2, 1]
    with pytest.raises(ValueError):
        dp.shard_groups(4, 2, 2)
    assert dp.global_valid_tokens(17) == 17  # not distributed: the local count
    assert dp.token_mean_scale(0) == 0.0
    # a count beyond 2^24 keeps its value until the final division
    assert dp.token_mean_scale(2**24 + 1) == float(np.float32(1.0 / (2**24 + 1)))
