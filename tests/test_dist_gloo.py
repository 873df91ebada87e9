"""Two-rank data-parallel host logic on CPU (gloo): no GPU.

Each rank takes a block of whole response groups, counts its valid rows and
all-reduces the count; both ranks must derive the same global token-mean
scale, and the shards must cover every group exactly once.  With the FP64
oracle standing in for each rank's kernel, the ranks' rows (advantages from
their own groups, local response indices, the global scale) must reproduce
the single-process gradients, log-probabilities and losses exactly.
"""

import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import synth
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
    mgr = mp.get_context("spawn").Manager()
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


def _shard_worker(rank, world, port, b, out):
    import oracle

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        G, L = b["group_size"], b["L_pad"]
        groups = dp.shard_groups(b["n_groups"], world, rank)
        r0, r1 = groups.start * G, groups.stop * G  # this rank's responses
        rows = slice(r0 * L, r1 * L)                # and their rows
        resp = b["row_response"][rows].copy()
        resp[resp >= 0] -= r0
        scale = dp.token_mean_scale(dp.global_valid_tokens(int((resp >= 0).sum())))
        adv = oracle.group_advantages(b["rewards"][r0:r1], len(groups), G, True, 1e-6).astype(np.float32)
        shard = dict(logits=b["logits"][rows], V=b["V"], rec_ids=b["rec_ids"][rows],
                     rec_logprobs=b["rec_logprobs"][rows], rec_count=None, sampled=b["sampled"][rows],
                     rollout_logprob=b["rollout_logprob"][rows], row_response=resp, adv=adv)
        prm = oracle.make_params(inv_temperature=b["inv_temperature"], grad_scale=scale)
        g, la, o, _ = oracle.rows(shard, prm, nthreads=1)
        out[rank] = (g, la, o["loss"].copy(), scale)
    finally:
        dist.destroy_process_group()


def test_two_ranks_reproduce_the_single_process_rows():
    import oracle

    world = 2
    cfg = synth.config("C1", n_prompts=3, V=512, K=16, L_pad=6)  # 3 groups of 4: an uneven split
    b = synth.to_numpy(synth.make_batch(cfg))
    b["L_pad"] = cfg["L_pad"]
    adv = oracle.group_advantages(b["rewards"], b["n_groups"], b["group_size"], True, 1e-6).astype(np.float32)
    scale = dp.token_mean_scale(int((b["row_response"] >= 0).sum()))
    prm = oracle.make_params(inv_temperature=b["inv_temperature"], grad_scale=scale)
    g_ref, la_ref, o_ref, _ = oracle.rows(dict(b, adv=adv, rec_count=None), prm, nthreads=1)
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_shard_worker, args=(world, _free_port(), b, out), nprocs=world, join=True,
                       start_method="spawn")
    res = [out[r] for r in range(world)]
    assert res[0][3] == res[1][3] == scale
    assert np.array_equal(np.concatenate([r[0] for r in res]), g_ref)
    assert np.array_equal(np.concatenate([r[1] for r in res]), la_ref)
    assert np.array_equal(np.concatenate([r[2] for r in res]), o_ref["loss"])
    assert len(dp.shard_groups(b["n_groups"], world, 0)) == 2  # the split really is uneven
