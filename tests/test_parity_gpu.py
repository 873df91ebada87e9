"""GPU parity: the CUDA library against the FP64 oracle, element by element.

Inputs come from the seeded generator (``synth``); advantages for the fused
kernel come from the oracle's own group statistics.  Tolerances are those of
``sc_parity``.  Sizes: the tiny configuration in full, reduced copies of the
large ones (full vocabulary, fewer rows, several clusters' worth of rows and
a ragged tail), and the full-size configurations with sampled rows plus
invariants on every row.
"""

import zlib

import numpy as np
import pytest
import torch

import oracle
import precision_off_policy_gb300 as sc
import synth
from sc_parity import (check_rows, diag_rows, grad_bits, host_batch, oracle_adv, oracle_params, run_gpu,
                       sc_params)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sc.build()
    sc.lib()


def _full_check(batch, p, what, inplace=False, with_rollout=True, nthreads=0, rows=None):
    adv = oracle_adv(batch)
    g, lp, d, status = run_gpu(batch, p, adv, inplace=inplace, with_rollout=with_rollout)
    T = batch["logits"].shape[0]
    rows = np.arange(T) if rows is None else np.asarray(rows)
    bn = host_batch(batch, adv, with_rollout)
    out = []
    for r0 in range(0, rows.size, 256):
        rr = rows[r0:r0 + 256]
        out.append(check_rows(bn, p, rr, grad_bits(g, rr), lp.cpu().numpy()[rr], diag_rows(d, rr),
                              nthreads=nthreads, what=what))
    st = int(status.item())
    assert st & (sc.SC_STATUS_TIMEOUT_LOAD | sc.SC_STATUS_TIMEOUT_EXCHANGE) == 0, f"{what}: status {st:#x}"
    return g, lp, d, st


# -------------------------------------------------------------------------
# Group advantages


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4", "C5"])
def test_group_advantages_match_oracle(name):
    cfg = synth.config(name)
    _, rewards = synth.responses(cfg)
    n = cfg["n_per_prompt"]
    a_gpu = sc.sc_group_advantages(rewards.cuda(), rewards.numel() // n, n).cpu().numpy()
    a_or = oracle.group_advantages(rewards.numpy(), rewards.numel() // n, n, True, 1e-6)
    np.testing.assert_allclose(a_gpu, a_or, rtol=1e-6, atol=1e-7)


def test_group_advantages_fractional_large_and_mean_only():
    rng = np.random.default_rng(5)
    r = np.concatenate([rng.random(64), [1.0, 1.001, 1.0, 1.0], [3e30, -3e30, 1e30, -1e30],
                        [0.25] * 4, rng.standard_normal(37 * 4) * 1e3]).astype(np.float32)
    ng = r.size // 4
    for norm in (True, False):
        a_gpu = sc.sc_group_advantages(torch.from_numpy(r).cuda(), ng, 4, norm).cpu().numpy()
        a_or = oracle.group_advantages(r, ng, 4, norm, 1e-6)
        np.testing.assert_allclose(a_gpu, a_or, rtol=1e-6, atol=1e-30)
    assert np.all(a_gpu[r.size - 37 * 4 - 4:r.size - 37 * 4] == 0)  # the all-equal group
    # large groups and in-place
    big = torch.rand(3 * 1000, device="cuda")
    ref = oracle.group_advantages(big.cpu().numpy(), 3, 1000, True, 1e-6)
    sc.sc_group_advantages(big, 3, 1000, out=big)
    np.testing.assert_allclose(big.cpu().numpy(), ref, rtol=1e-6, atol=1e-7)


# -------------------------------------------------------------------------
# The fused kernel


def test_c1_tiny_full_parity():
    batch = synth.make_batch("C1")
    p = sc_params(batch)
    _, _, _, st = _full_check(batch, p, "C1")
    assert st == 0


def test_c1_without_rollout_logprob():
    batch = synth.make_batch("C1")
    _, _, d, _ = _full_check(batch, sc_params(batch), "C1 no rollout", with_rollout=False)
    assert np.all(sc.diag_to_numpy(d)["k3"] == 0)


@pytest.mark.parametrize("name", ["C2", "C4", "C5"])
def test_reduced_configs_full_parity(name):
    # full vocabulary, a few responses: several rows per cluster, padding,
    # ragged counts and the peaked large-vocabulary rows.
    over = dict(n_prompts=1, n_per_prompt=4 if name != "C5" else 8, L_pad=24)
    if name == "C2":
        over.update(len_lo=5, len_hi=24)
    batch = synth.make_batch(synth.config(name, **over))
    _full_check(batch, sc_params(batch), f"{name} reduced")


def test_c3_chunk_reduced_full_parity():
    cfg = synth.config("C3", n_prompts=2, L_pad=40, len_lo=10, len_hi=40, chunk_rows=40 * 4)
    batch = synth.make_batch(cfg, chunk=1)
    _full_check(batch, sc_params(batch), "C3 reduced chunk 1")


@pytest.mark.parametrize("flags", [0, sc.SC_FLAGS_VECTOR])
@pytest.mark.parametrize("V", [1, 3, 8, 13, 1000, 4097, 33333])
def test_ragged_vocabulary_sizes(V, flags):
    K = min(128, V)
    cfg = synth.config("C1", V=V, K=K, L_pad=5, sigma=2.5)
    batch = synth.make_batch(cfg)
    _full_check(batch, sc_params(batch, flag_layout=flags), f"V={V} flags={flags}")


@pytest.mark.parametrize("flags", [sc.SC_FLAGS_ENTRY, sc.SC_FLAGS_VECTOR])
@pytest.mark.parametrize("cluster,threads,stages", [(1, 128, 1), (2, 256, 2), (3, 384, 3), (4, 512, 4),
                                                    (8, 256, 1), (16, 128, 2), (16, 256, 3), (5, 256, 2)])
def test_explicit_launch_shapes(cluster, threads, stages, flags):
    cfg = synth.config("C2", n_prompts=1, n_per_prompt=2, L_pad=16, len_lo=10, len_hi=16, V=30011)
    batch = synth.make_batch(cfg)
    _full_check(batch, sc_params(batch, cluster_size=cluster, threads=threads, stages=stages, flag_layout=flags),
                f"C={cluster} NT={threads} stages={stages} flags={flags}")


@pytest.mark.parametrize("flags", [0, sc.SC_FLAGS_VECTOR])
def test_largest_vocabulary_and_head(flags):
    # the largest sizes the call accepts: V = 2^20 (clusters of 16 CTAs) and
    # K_max = 1024 recorded ids per row
    cfg = synth.config("C1", V=1 << 20, K=1024, L_pad=3, sigma=2.5)
    batch = synth.make_batch(cfg)
    _full_check(batch, sc_params(batch, flag_layout=flags), f"V=2^20 K=1024 flags={flags}")


def test_automatic_flag_layout_follows_residency():
    # per-entry flags at 151936 entries (4 CTAs x 74 clusters beat 3 x 97);
    # per-vector flags at 248320 (5 x 58 beat 6 x 46): the plan with more CTAs
    p = sc.params(K_max=128)
    q1, q2 = sc.sc_plan_query(151936, p), sc.sc_plan_query(248320, p)
    assert q1["flag_layout"] == sc.SC_FLAGS_ENTRY and q1["cluster_size"] == 4, q1
    assert q2["flag_layout"] == sc.SC_FLAGS_VECTOR and q2["cluster_size"] == 5, q2
    assert q2["cluster_size"] * q2["max_clusters"] > 6 * sc.sc_plan_query(248320, sc.params(
        K_max=128, cluster_size=6))["max_clusters"]


@pytest.mark.parametrize("mode", [sc.SC_IS_TIS, sc.SC_IS_MIS])
@pytest.mark.parametrize("centering", [True, False])
def test_importance_weighting_modes(mode, centering):
    # a wider sampler mismatch so that weights leave [0.5, 5] and exceed 2
    cfg = synth.config("C1", sigma_s=1.5, L_pad=16)
    batch = synth.make_batch(cfg)
    p = sc_params(batch, is_mode=mode, centering=centering)
    adv = oracle_adv(batch)
    g, lp, d, _ = run_gpu(batch, p, adv)
    bn = host_batch(batch, adv)
    # rows whose weight sits at a bound within float rounding decide differently: skip them
    G, LA, OUT, _ = oracle.rows(bn, oracle.make_params(is_mode=mode, centering=centering), np.arange(len(lp)))
    w = np.exp(LA - bn["rollout_logprob"].astype(np.float64))
    bounds = [p.tis_max] if mode == sc.SC_IS_TIS else [p.mis_min, p.mis_max]
    ok = np.all([np.abs(w - b) > 1e-3 * b for b in bounds], axis=0)
    rows = np.nonzero(ok)[0]
    assert rows.size >= len(lp) // 2
    check_rows(bn, p, rows, grad_bits(g, rows), lp.cpu().numpy()[rows], diag_rows(d, rows),
               what=f"is_mode={mode} centering={centering}")
    flags = sc.diag_to_numpy(d)["flags"]
    bit = sc.FLAG_IS_TRUNC if mode == sc.SC_IS_TIS else sc.FLAG_IS_REJECT
    assert np.any(flags & bit), "the test inputs should exercise the weight bound"


@pytest.mark.parametrize("sign", [1.0, -1.0])
def test_clipped_grpo_mode(sign):
    """The clipped GRPO baseline: a wide sampler mismatch spreads the ratio
    across both clip bounds; the advantages are the per-rollout means."""
    cfg = synth.config("C1", sigma_s=1.5, L_pad=16)
    batch = synth.make_batch(cfg)
    p = sc_params(batch, is_mode=sc.SC_IS_CLIP, centering=False, grad_scale=1.0 / 8)
    adv = (sign * np.abs(oracle_adv(batch)) + 0.25 * sign).astype(np.float32)  # one sign per run
    g, lp, d, _ = run_gpu(batch, p, adv)
    bn = host_batch(batch, adv)
    G, LA, OUT, _ = oracle.rows(bn, oracle_params(p), np.arange(len(lp)))
    w = np.exp(LA - bn["rollout_logprob"].astype(np.float64))
    ok = np.all([np.abs(w - b) > 1e-3 * b for b in [1.0 - 0.2, 1.0 + 0.3]], axis=0)
    rows = np.nonzero(ok)[0]
    assert rows.size >= len(lp) // 2
    check_rows(bn, p, rows, grad_bits(g, rows), lp.cpu().numpy()[rows], diag_rows(d, rows), what=f"clip A{sign:+}")
    flags = sc.diag_to_numpy(d)["flags"][rows]
    np.testing.assert_array_equal(flags & sc.FLAG_CLIPPED, OUT["flags"][rows] & oracle.FLAG_CLIPPED)
    assert np.any(flags & sc.FLAG_CLIPPED), "some rows should have the clipped term as the minimum"
    assert np.any((flags & sc.FLAG_CLIPPED) == 0) and np.any(~((w > 0.8) & (w < 1.3))[rows] & ((flags & sc.FLAG_CLIPPED) == 0)), \
        "some rows outside the clip range should keep their gradient"
    gr = g.float().cpu().numpy()[rows]
    assert np.all(gr[(flags & sc.FLAG_CLIPPED) != 0] == 0)


def test_rollout_mean_advantages_match_oracle():
    for name in ["C1", "C2", "C5"]:
        cfg = synth.config(name)
        lengths, rewards = synth.responses(cfg)
        L = cfg["L_pad"]
        n_resp = rewards.numel()
        rows = torch.arange(n_resp * L)
        rr = torch.where((rows % L) < lengths[rows // L], rows // L, torch.full_like(rows, -1)).to(torch.int32)
        rr[5] = n_resp + 3  # an out-of-range index counts for nobody
        adv = oracle.group_advantages(rewards.numpy(), n_resp // cfg["n_per_prompt"], cfg["n_per_prompt"])
        adv32 = adv.astype(np.float32)
        out, counts = sc.sc_rollout_mean_advantages(torch.from_numpy(adv32).cuda(), rr.cuda())
        ref, rc = oracle.rollout_mean_advantages(adv32.astype(np.float64), rr.numpy(), n_resp)
        assert counts.cpu().numpy().tolist() == rc.tolist(), name
        np.testing.assert_array_equal(out.cpu().numpy(), ref.astype(np.float32), err_msg=name)
    # in place, and an empty batch of rows
    a = torch.tensor([2.0, -1.0], device="cuda")
    out, counts = sc.sc_rollout_mean_advantages(a, torch.tensor([0, 0, 1, 0], dtype=torch.int32, device="cuda"), out=a)
    assert a.cpu().tolist() == [float(np.float32(2.0) / np.float32(3.0)), -1.0]
    out, counts = sc.sc_rollout_mean_advantages(a, torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert out.cpu().tolist() == [0.0, 0.0] and counts.cpu().tolist() == [0, 0]


def test_temperature_and_grad_scale():
    cfg = synth.config("C1", temperature=0.7, L_pad=12)
    batch = synth.make_batch(cfg)
    _full_check(batch, sc_params(batch, grad_scale=1.0 / 96.0), "T=0.7 scale=1/96")


def test_in_place_equals_out_of_place_bitwise():
    cfg = synth.config("C2", n_prompts=1, n_per_prompt=2, L_pad=16, len_lo=8, len_hi=16)
    batch = synth.make_batch(cfg)
    p = sc_params(batch)
    adv = oracle_adv(batch)
    g1, lp1, d1, _ = run_gpu(batch, p, adv)
    g2, lp2, d2, _ = run_gpu(batch, p, adv, inplace=True)
    assert torch.equal(g1.view(torch.int16), g2.view(torch.int16))
    assert torch.equal(lp1, lp2) and torch.equal(d1, d2)


def test_deterministic_across_calls():
    batch = synth.make_batch(synth.config("C1", L_pad=16))
    p = sc_params(batch)
    adv = oracle_adv(batch)
    r1 = run_gpu(batch, p, adv)
    r2 = run_gpu(batch, p, adv)
    for a, b in zip(r1[:3], r2[:3]):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)


def test_run_time_row_hand_out_is_deterministic_and_leaves_the_workspace_zero():
    # 1024 rows over the persistent grid: the first rows are dealt round robin,
    # the last rows handed out at run time, so which cluster takes which
    # row changes from call to call; every output must not.
    cfg = synth.config("C2", n_prompts=1, n_per_prompt=2, L_pad=512, len_lo=64, len_hi=512)
    batch = synth.make_batch(cfg)
    p = sc_params(batch)
    adv = oracle_adv(batch)
    runs = [run_gpu(batch, p, adv) for _ in range(3)]
    for r in runs[1:]:
        assert torch.equal(runs[0][0].view(torch.int16), r[0].view(torch.int16))
        assert torch.equal(runs[0][1], r[1]) and torch.equal(runs[0][2], r[2])
        assert int(r[3].item()) == 0
    ws = sc.workspace(torch.device("cuda"))
    assert int(ws.abs().sum().item()) == 0


def test_concurrent_streams_with_their_own_workspaces():
    # Two launches at once on two streams (the binding gives each stream its
    # own workspace, so their run-time row counters do not meet): each result
    # equals the same call run alone.
    dev = torch.device("cuda")
    cfg_a = synth.config("C2", n_prompts=1, n_per_prompt=2, L_pad=512, len_lo=64, len_hi=512)
    cfg_b = synth.config("C4", n_prompts=1, n_per_prompt=2, L_pad=256)
    outs = {}
    for name, cfg in (("a", cfg_a), ("b", cfg_b)):
        b = synth.make_batch(cfg)
        adv = torch.as_tensor(oracle_adv(b), device=dev)
        x = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in b.items()}
        outs[name] = (x, adv, sc_params(b))
    alone = {}
    for name, (x, adv, p) in outs.items():
        g, lp, _ = sc.sc_center_forward_backward(x["logits"], x["rec_ids"], x["rec_logprobs"], x["rec_count"],
                                                 x["sampled"], x["rollout_logprob"], x["row_response"], adv, p)
        torch.cuda.synchronize()
        alone[name] = (g.clone(), lp.clone())
    streams = {"a": torch.cuda.Stream(), "b": torch.cuda.Stream()}
    res = {}
    for _ in range(3):
        for name, (x, adv, p) in outs.items():
            s = streams[name]
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                res[name] = sc.sc_center_forward_backward(
                    x["logits"], x["rec_ids"], x["rec_logprobs"], x["rec_count"], x["sampled"], x["rollout_logprob"],
                    x["row_response"], adv, p, stream=s)
        torch.cuda.synchronize()
        for name in outs:
            assert torch.equal(res[name][0].view(torch.int16), alone[name][0].view(torch.int16)), name
            assert torch.equal(res[name][1], alone[name][1]), name
    for s in streams.values():
        assert int(sc.workspace(dev, s).abs().sum().item()) == 0


# -------------------------------------------------------------------------
# Edge cases


def _edit(batch, **kw):
    b = dict(batch)
    for k, v in kw.items():
        b[k] = v
    return b


def test_head_hygiene_duplicates_out_of_range_counts():
    batch = synth.make_batch(synth.config("C1", L_pad=6))
    T, K = batch["rec_ids"].shape
    ids = batch["rec_ids"].clone()
    ids[0, 5] = ids[0, 2]            # a repeat
    ids[1, 0] = 5000                 # out of range (V = 1024)
    ids[2, 7] = -1                   # out of range
    ids[3, 10:20] = ids[3, 0]        # many repeats
    ids[4, 1] = batch["sampled"][4]  # the sampled token inside the head
    count = torch.full((T,), K, dtype=torch.int32)
    count[5] = 0                     # empty head
    count[6] = 300                   # out of range: clamped to K
    count[7] = -4                    # out of range: clamped to 0
    count[8] = 1
    b = _edit(batch, rec_ids=ids, rec_count=count)
    _, _, d, st = _full_check(b, sc_params(b), "head hygiene")
    f = sc.diag_to_numpy(d)["flags"]
    assert f[0] & sc.FLAG_DUP_ID and f[1] & sc.FLAG_BAD_ID and f[2] & sc.FLAG_BAD_ID
    assert f[6] & sc.FLAG_BAD_COUNT and f[7] & sc.FLAG_BAD_COUNT
    assert st & sc.SC_STATUS_DATA


def test_bad_rows_and_all_masked():
    batch = synth.make_batch(synth.config("C1", L_pad=6))
    resp = batch["row_response"].clone()
    samp = batch["sampled"].clone()
    resp[3] = 99                     # response index beyond n_resp
    samp[4] = 1024                   # sampled id beyond V
    samp[5] = -2
    resp[6:9] = -1                   # padding
    b = _edit(batch, row_response=resp, sampled=samp)
    g, lp, d, st = _full_check(b, sc_params(b), "bad rows")
    assert torch.all(g[3:9] == 0)
    assert st & sc.SC_STATUS_DATA
    b2 = _edit(batch, row_response=torch.full_like(resp, -1))
    g2, lp2, d2, st2 = _full_check(b2, sc_params(b2), "all masked")
    assert torch.all(g2 == 0) and torch.all(lp2 == 0) and st2 == 0


def test_empty_batch_and_empty_head_parameter():
    batch = synth.make_batch(synth.config("C1", L_pad=4))
    p = sc_params(batch)
    z = lambda t: t[:0]
    g, lp, d = sc.sc_center_forward_backward(
        z(batch["logits"]).cuda(), z(batch["rec_ids"]).cuda(), z(batch["rec_logprobs"]).cuda(), None,
        z(batch["sampled"]).cuda(), None, z(batch["row_response"]).cuda(),
        torch.zeros(8, device="cuda"), p)
    assert g.shape == (0, 1024)
    # K_max = 0: no recorded head at all -> plain policy gradient
    b = _edit(batch, rec_ids=batch["rec_ids"][:, :0].contiguous(), rec_logprobs=batch["rec_logprobs"][:, :0].contiguous())
    _full_check(b, sc_params(b, K_max=0), "K_max=0")


def test_autograd_wrapper_matches_direct_call():
    batch = synth.make_batch(synth.config("C1", L_pad=8))
    p = sc_params(batch, grad_scale=1.0 / 64.0)
    adv = torch.from_numpy(oracle_adv(batch)).cuda()
    b = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in batch.items()}
    logits = b["logits"].clone().requires_grad_(True)
    loss, logp, diag = sc.score_centered_loss(logits, b["rec_ids"], b["rec_logprobs"], b["rec_count"], b["sampled"],
                                              b["rollout_logprob"], b["row_response"], adv, p)
    (2.0 * loss).backward()
    g, lp, d = sc.sc_center_forward_backward(b["logits"], b["rec_ids"], b["rec_logprobs"], b["rec_count"],
                                             b["sampled"], b["rollout_logprob"], b["row_response"], adv, p,
                                             diag_out=torch.empty((64, 16), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(logits.grad, g * 2.0)
    assert torch.equal(logp, lp) and torch.equal(diag, d)
    rows = sc.diag_to_numpy(d)["loss"].astype(np.float64)
    assert abs(float(loss.detach()) - rows.sum() / 64.0) <= 1e-5 * max(1.0, abs(rows.sum() / 64.0))


def _unprotected(batch):
    """Mask of the entries that are neither recorded ids nor the sampled token."""
    T, V = batch["logits"].shape
    keep = torch.ones(T, V, dtype=torch.bool)
    ids = batch["rec_ids"].long()
    ok = (ids >= 0) & (ids < V)
    keep.scatter_(1, torch.where(ok, ids, torch.zeros_like(ids)), False)
    keep[torch.arange(T), batch["sampled"].long()] = False
    return keep


@pytest.mark.parametrize("cluster,threads,flags", [(0, 0, 0), (2, 128, 0), (0, 0, 2), (2, 128, 2)])
def test_wide_dynamic_range_and_infinite_logits(cluster, threads, flags):
    """Entries far above the exponent offset a warp takes from its first vectors
    (2^y would overflow), -inf entries (0 * -inf), and warps whose first vectors
    are all -inf: each takes the exact per-thread path and must still match."""
    batch = synth.make_batch(synth.config("C1", V=8192, L_pad=8))
    z = batch["logits"].float().clone()
    free = _unprotected(batch)
    row0 = torch.zeros_like(free[0])
    row0[6000:6003] = True                     # row 0: three entries at +120
    z[0, row0 & free[0]] = 120.0
    row3 = torch.zeros_like(free[3])
    row3[4000:4100] = True                     # row 3: a block at +90
    z[3, row3 & free[3]] = 90.0
    neg = torch.zeros_like(free)
    neg[1, 100:200] = True                     # row 1: scattered -inf
    neg[2, :2048] = True                       # row 2: the first 2048 entries -inf
    z[neg & free] = float("-inf")
    b = _edit(batch, logits=z.to(torch.bfloat16))
    _full_check(b, sc_params(b, cluster_size=cluster, threads=threads, flag_layout=flags),
                f"dynamic range {cluster},{threads} flags={flags}")


def test_row_stride_larger_than_vocab():
    batch = synth.make_batch(synth.config("C1", V=1000, L_pad=8))
    T = batch["logits"].shape[0]
    wide = torch.zeros((T, 1024), dtype=torch.bfloat16)
    wide[:, :1000] = batch["logits"]
    wide = wide.cuda()
    adv = oracle_adv(batch)
    p = sc_params(batch)
    out = torch.full((T, 1016), 7.0, dtype=torch.bfloat16, device="cuda")
    b = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in batch.items()}
    sc.sc_center_forward_backward(wide, b["rec_ids"], b["rec_logprobs"], None, b["sampled"],
                                  b["rollout_logprob"], b["row_response"], torch.as_tensor(adv).cuda(), p,
                                  V=1000, grad_out=out)
    ref = run_gpu(batch, p, adv)[0]
    assert torch.equal(out[:, :1000].view(torch.int16), ref.view(torch.int16))
    assert torch.all(out[:, 1000:] == 7.0)


# -------------------------------------------------------------------------
# Full-size configurations


@pytest.mark.slow
def test_c2_full_size_every_row():
    batch = synth.make_batch("C2", device="cuda")
    _full_check(batch, sc_params(batch), "C2 full")


def _invariants(batch, g, d, p):
    """Properties that hold at any size, checked on every row on the device.
    Returns the fraction of rows with a nonzero advantage whose bf16 output
    meets the bare row-sum bound 1e-3 |a| with no rounding allowance."""
    diag = sc.diag_to_numpy(d)
    valid = batch["row_response"].cpu().numpy() >= 0
    assert np.all(diag["flags"][~valid] == sc.FLAG_MASKED)
    a = np.abs(diag["adv"] * diag["is_weight"]) * p.inv_temperature * abs(p.grad_scale)
    # the kernel's FP32 row sums: the derived FP32 rounding bound (sc_parity.fp32_row_sum_bound)
    assert np.all(np.abs(diag["row_sum"]) <= 1e-3 * a * np.maximum(1, diag["rho"]) + 1e-7), "FP32 row sums"
    # bf16 output row sums, with half an ulp per element of rounding allowance
    gs = g.double().sum(dim=1).cpu().numpy()
    gabs = g.float().abs()
    e = torch.floor(torch.log2(gabs.clamp_min(2.0**-126)))
    half_ulp = (0.5 * torch.exp2(e - 7) * (gabs > 0)).double().sum(dim=1).cpu().numpy()
    assert np.all(np.abs(gs) <= 1e-3 * a + half_ulp + 1e-7), "bf16 row sums"
    assert np.all(np.isfinite(diag["loss"])) and np.all(diag["P_H"][valid] <= 1.0 + 1e-6)
    assert np.all(np.abs(diag["P_H"] + diag["tail_pi"] - valid) <= 1e-5)
    live = a > 0
    return float(np.mean(np.abs(gs)[live] <= 1e-3 * a[live])) if live.any() else 1.0


@pytest.mark.slow
@pytest.mark.parametrize("name,chunk", [("C4", 0), ("C5", 0), ("C3", 0), ("C3", 17)])
def test_full_size_sampled_rows_and_invariants(name, chunk):
    cfg = synth.config(name)
    batch = synth.make_batch(cfg, chunk=chunk, device="cuda")
    T = batch["logits"].shape[0]
    p = sc_params(batch)
    adv = oracle_adv(batch)
    g, lp, d, status = run_gpu(batch, p, adv)
    assert int(status.item()) & 0x6 == 0
    rng = np.random.default_rng(zlib.crc32(f"{name}/{chunk}".encode()))
    rows = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 192, replace=False)]))
    bn = {k: v for k, v in batch.items()}
    # only the sampled rows travel to the host for the oracle
    sub = {k: (v[torch.as_tensor(rows, device=v.device)] if isinstance(v, torch.Tensor) and v.dim() >= 1
               and v.shape[0] == T else v) for k, v in bn.items()}
    bh = host_batch(sub, adv)
    check_rows(bh, p, np.arange(rows.size), grad_bits(g, rows), lp.cpu().numpy()[rows], diag_rows(d, rows),
               what=f"{name} chunk {chunk} sampled")
    bare = _invariants(batch, g, d, p)
    print(f"{name} chunk {chunk}: {bare:.3f} of the rows meet the bare bf16 row-sum bound")


# -------------------------------------------------------------------------
# The clamped-denominator regime: the trainer's mass sits on the recorded ids
# (1 - P_H below 1e-6, clamped) while the sampler's tail 1 - Q_H stays large,
# so rho = max(1 - Q_H, 1e-6) / 1e-6 reaches 1e4 .. 1e6 and the unrecorded
# entries get mu_hat = s p with s of the same order.


def _clamp_regime_asserts(diag, valid):
    f = diag["flags"][valid]
    rho = diag["rho"][valid]
    clamped = (f & sc.FLAG_CLAMP_PI) != 0
    assert clamped.mean() >= 0.5, f"only {clamped.mean():.2f} of the rows clamp 1 - P_H"
    assert not np.any(f & sc.FLAG_CLAMP_MU), "the sampler's tail should stay above 1e-6"
    # rho = max(1 - Q_H, 1e-6) / 1e-6 on a clamped row: 1e3 and more wherever the
    # sampler leaves more than 1e-3 of its mass outside the recorded ids
    big = rho[clamped] >= 1e3
    assert big.mean() >= 0.9, f"only {big.mean():.2f} of the clamped rows reach rho >= 1e3"
    assert np.median(rho[clamped]) >= 1e4, f"median rho of clamped rows {np.median(rho[clamped])}"
    return clamped.mean(), float(np.median(rho))


def test_clamped_denominator_reduced_full_parity():
    cfg = synth.config("C2R", n_prompts=1, n_per_prompt=4, L_pad=24, len_lo=5, len_hi=24)
    batch = synth.make_batch(cfg)
    _, _, d, _ = _full_check(batch, sc_params(batch), "rho >> 1 reduced")
    frac, med = _clamp_regime_asserts(sc.diag_to_numpy(d), batch["row_response"].numpy() >= 0)
    print(f"rho >> 1 reduced: {frac:.2f} of the rows clamped, median rho {med:.3g}")


@pytest.mark.slow
def test_clamped_denominator_full_size_sampled_rows_and_invariants():
    batch = synth.make_batch("C2R", device="cuda")
    T = batch["logits"].shape[0]
    p = sc_params(batch)
    adv = oracle_adv(batch)
    g, lp, d, status = run_gpu(batch, p, adv)
    assert int(status.item()) & 0x6 == 0
    valid = batch["row_response"].cpu().numpy() >= 0
    frac, med = _clamp_regime_asserts(sc.diag_to_numpy(d), valid)
    rng = np.random.default_rng(zlib.crc32(b"C2R"))
    vrows = np.nonzero(valid)[0]
    rows = np.unique(np.concatenate([[0, T - 1], rng.choice(vrows, 192, replace=False)]))
    sub = {k: (v[torch.as_tensor(rows, device=v.device)] if isinstance(v, torch.Tensor) and v.dim() >= 1
               and v.shape[0] == T else v) for k, v in batch.items()}
    check_rows(host_batch(sub, adv), p, np.arange(rows.size), grad_bits(g, rows), lp.cpu().numpy()[rows],
               diag_rows(d, rows), what="rho >> 1 full size sampled")
    bare = _invariants(batch, g, d, p)
    print(f"rho >> 1 full size: {frac:.2f} of the rows clamped, median rho {med:.3g}, "
          f"{bare:.3f} meet the bare bf16 row-sum bound")


# -------------------------------------------------------------------------
# Failure path: a wait that runs out.  The test hook (`test_stall`) makes every
# CTA leave out the bulk copy of its first row's first chunk, so the waits for
# it can never complete: the launch must give up after `wait_limit_us`, set
# SC_STATUS_TIMEOUT_LOAD, let its other copies land, leave the workspace zero
# and return with the context usable.  Nothing faults, traps or spins forever.


@pytest.mark.parametrize("cluster,threads,stages", [(0, 0, 0), (8, 128, 2)])
def test_a_wait_that_runs_out_sets_the_status_and_the_next_call_is_clean(cluster, threads, stages):
    dev = torch.device("cuda")
    cfg = synth.config("C2", n_prompts=1, n_per_prompt=2, L_pad=512, len_lo=64, len_hi=512)
    batch = synth.make_batch(cfg)
    adv = oracle_adv(batch)
    shape = dict(cluster_size=cluster, threads=threads, stages=stages)
    g_ok, lp_ok, d_ok, st_ok = run_gpu(batch, sc_params(batch, **shape), adv)
    assert int(st_ok.item()) == 0
    p_stall = sc_params(batch, wait_limit_us=2000, test_stall=1, **shape)
    _, _, _, st = run_gpu(batch, p_stall, adv)  # synchronises: a CUDA error would raise here
    assert int(st.item()) & sc.SC_STATUS_TIMEOUT_LOAD, f"status {int(st.item()):#x}"
    ws = sc.workspace(dev)
    assert int(ws.abs().sum().item()) == 0, "the workspace is left zero after a launch that gave up"
    # the same context runs a normal call cleanly afterwards
    g2, lp2, d2, st2 = run_gpu(batch, sc_params(batch, **shape), adv)
    assert int(st2.item()) == 0
    assert torch.equal(g2.view(torch.int16), g_ok.view(torch.int16))
    assert torch.equal(lp2, lp_ok) and torch.equal(d2, d_ok)
    assert int(ws.abs().sum().item()) == 0


def test_binding_on_a_stream_that_is_not_current():
    # The binding's workspace for a stream is zero-filled on that stream, so the
    # first launch on a fresh, non-current stream sees it zeroed.
    dev = torch.device("cuda")
    cfg = synth.config("C2", n_prompts=1, n_per_prompt=2, L_pad=512, len_lo=64, len_hi=512)
    batch = synth.make_batch(cfg)
    adv = oracle_adv(batch)
    p = sc_params(batch)
    g_ref, lp_ref, d_ref, _ = run_gpu(batch, p, adv)
    for _ in range(2):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        x = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in batch.items()}
        advd = torch.as_tensor(adv, device=dev)
        diag = torch.zeros((x["logits"].shape[0], 16), dtype=torch.int32, device=dev)
        torch.cuda.synchronize()
        g, lp, d = sc.sc_center_forward_backward(x["logits"], x["rec_ids"], x["rec_logprobs"], x["rec_count"],
                                                 x["sampled"], x["rollout_logprob"], x["row_response"], advd, p,
                                                 diag_out=diag, stream=s)
        s.synchronize()
        assert torch.equal(g.view(torch.int16), g_ref.view(torch.int16))
        assert torch.equal(lp, lp_ref) and torch.equal(d, d_ref)
        assert int(sc.workspace(dev, s).abs().sum().item()) == 0


def test_batch_loss_is_the_scaled_sum_of_the_row_losses():
    """sc_batch_loss: grad_scale * sum of the rows' losses in a fixed order,
    one FP32 rounding; the same bits on every call; 0 for no rows."""
    batch = synth.make_batch(synth.config("C2", n_prompts=1, n_per_prompt=2, L_pad=512, len_lo=64, len_hi=512))
    p = sc_params(batch, grad_scale=1.0 / 997.0)
    adv = oracle_adv(batch)
    _, _, d, _ = run_gpu(batch, p, adv)
    rows = sc.diag_to_numpy(d)["loss"].astype(np.float64)
    want = float(np.float32(p.grad_scale)) * rows.sum()
    got = [float(sc.sc_batch_loss(d, p.grad_scale).item()) for _ in range(3)]
    assert got[0] == got[1] == got[2]
    # FP64 partial sums: the only rounding that matters is the final one to FP32
    assert abs(got[0] - want) <= 2.0 ** -23 * abs(want) + 1e-30
    empty = sc.sc_batch_loss(torch.zeros((0, 16), dtype=torch.int32, device="cuda"), 1.0)
    assert float(empty.item()) == 0.0
