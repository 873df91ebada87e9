"""GPU parity of the sampler-side top-K capture against the FP64 oracle.

Sampler logits follow the workloads' recipe (FP32 trainer logits plus the
sampler's Gaussian perturbation); edge cases force every path of the
selection: exact ties beyond the candidate buffer, crowded bins, -inf
entries, short and ragged rows, and top-p crossings both inside the selected
entries and far below them.
"""

import numpy as np
import pytest
import torch

import oracle
import precision_off_policy_gb300 as sc
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sc.build()
    sc.lib()


def sampler_logits(name, rows, sigma_s=None, seed=0):
    """FP32 sampler logits: a config's trainer logits plus its sampler noise."""
    cfg = synth.config(name)
    b = synth.make_batch(cfg, device="cuda")
    z = b["logits"][:rows].float()
    g = torch.Generator(device="cuda").manual_seed(1234 + seed)
    s = cfg["sigma_s"] if sigma_s is None else sigma_s
    return (z + torch.randn(z.shape, generator=g, device="cuda") * s).contiguous()


def run(z, K, inv_t, top_p, stride=None):
    T, V = z.shape
    if stride is not None and stride != V:
        buf = torch.full((T, stride), float("nan"), dtype=torch.float32, device="cuda")
        buf[:, :V] = z
        ids, lp, cnt = sc.sc_topk_capture(buf, K, inv_t, top_p, V=V)
    else:
        ids, lp, cnt = sc.sc_topk_capture(z, K, inv_t, top_p)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), lp.cpu().numpy(), cnt.cpu().numpy()


def boundary_is_clear(z_row, inv_t, top_p, K, rel=1e-6):
    """(clear, extra) for one row's nucleus boundary, from FP64.

    An entry whose preceding mass lies within `rel` of top_p may fall on
    either side of the boundary under rounding.  When such an entry could
    change the count (its position is within the first K), the row is not
    clear.  Otherwise the ids and the count are fixed, and only the nucleus
    mass, and with it every recorded log-probability, can move by the mass of
    one such entry: `extra` is the largest of those masses over the nucleus
    mass (0 when no entry is that close)."""
    if top_p >= 1.0:
        return True, 0.0
    x = z_row.astype(np.float64) * inv_t
    order = np.lexsort((np.arange(x.size), -x))
    p = np.exp(x[order] - x.max())
    p /= p.sum()
    before = np.concatenate([[0.0], np.cumsum(p)[:-1]])
    near = np.nonzero(np.abs(before - top_p) <= rel)[0]
    if near.size == 0:
        return True, 0.0
    if near.min() <= K:
        return False, 0.0
    nucleus = p[before < top_p].sum()
    return True, float(p[np.clip(np.concatenate([near - 1, near]), 0, p.size - 1)].max() / nucleus)


def check(z, K, inv_t, top_p, what, stride=None, lp_tol=2e-6, rows=None):
    """GPU capture of every row of z, compared with the oracle on `rows` (all by default)."""
    ids, lp, cnt = run(z, K, inv_t, top_p, stride)
    if rows is not None:
        sel = torch.as_tensor(np.asarray(rows), device=z.device)
        z = z.index_select(0, sel)
        ids, lp, cnt = ids[rows], lp[rows], cnt[rows]
    zc = z.cpu().numpy()
    oids, olp, ocnt = oracle.topk_capture(zc, K, inv_t, top_p)
    verdicts = [boundary_is_clear(zc[t], inv_t, top_p, K) for t in range(zc.shape[0])]
    clear = np.array([v[0] for v in verdicts])
    assert clear.sum() >= max(1, zc.shape[0] // 2), f"{what}: too few unambiguous rows"
    for t in np.nonzero(clear)[0]:
        row_tol = lp_tol + verdicts[t][1]
        assert cnt[t] == ocnt[t], f"{what} row {t}: count {cnt[t]} vs {ocnt[t]}"
        np.testing.assert_array_equal(ids[t], oids[t], err_msg=f"{what} row {t}: ids")
        c = ocnt[t]
        fin = np.isfinite(olp[t, :c])
        assert np.array_equal(lp[t, :c][~fin], olp[t, :c][~fin]), f"{what} row {t}: infinite logprobs"
        a, o = lp[t, :c][fin].astype(np.float64), olp[t, :c][fin].astype(np.float64)
        err = np.abs(a - o) / (1 + np.abs(o))
        assert np.all(err <= row_tol), f"{what} row {t}: logprob error {err.max():.3g} at {int(err.argmax())}"
        assert np.all(lp[t, c:] == 0)
    return ids, lp, cnt


@pytest.mark.parametrize("inv_t,top_p", [(1.0, 1.0), (1 / 0.7, 0.95), (1.0, 0.5), (2.0, 0.99)])
def test_small_vocabulary(inv_t, top_p):
    z = sampler_logits("C1", 64)
    check(z, 128, inv_t, top_p, f"C1 inv_t={inv_t} top_p={top_p}")


@pytest.mark.parametrize("name,inv_t,top_p", [("C2", 1.0, 1.0), ("C2", 1 / 0.7, 0.95), ("C4", 1.0, 1.0),
                                               ("C4", 1.0, 0.9)])
def test_full_vocabulary_rows(name, inv_t, top_p):
    z = sampler_logits(name, 48)
    check(z, 128, inv_t, top_p, f"{name} inv_t={inv_t} top_p={top_p}")


def test_ties_beyond_the_candidate_buffer_and_crowded_bins():
    V = 20000
    rows = []
    rows.append(np.full(V, 0.75, np.float32))                              # one value everywhere
    r = np.full(V, -3.0, np.float32); r[17] = 4.0; r[9000:9005] = 2.0; rows.append(r)
    rows.append((1.0 + np.arange(V, dtype=np.float32) * 1e-7).astype(np.float32))  # one crowded top bin
    rng = np.random.default_rng(3)
    r = rng.choice(np.array([0.5, 0.25, -1.0], np.float32), V); rows.append(r)      # a few values, many ties
    z = torch.from_numpy(np.stack(rows)).cuda()
    for K, top_p in [(128, 1.0), (1000, 1.0), (64, 0.5), (128, 0.3)]:
        check(z, K, 1.0, top_p, f"ties K={K} top_p={top_p}")


def test_infinite_entries_short_rows_and_padded_strides():
    rng = np.random.default_rng(4)
    for V, stride in [(5, 8), (13, 16), (1001, 1004), (4099, 4100)]:
        z = (rng.standard_normal((6, V)) * 2).astype(np.float32)
        z[0, ::3] = -np.inf
        z[1, 1:] = -np.inf  # a single finite entry
        # a single finite entry outside the 1/16 threshold sample (at V = 4099 the
        # sample reads entries 0-127 and 2048-2175): the one-pass path leaves at its
        # sample, after its first copies have started, and the exact path takes the row
        z[2, :] = -np.inf
        z[2, 200 if V > 2048 else V // 2] = 1.5
        check(torch.from_numpy(z).cuda(), 8, 1.0, 1.0, f"V={V}", stride=stride)
        check(torch.from_numpy(z).cuda(), 8, 1.3, 0.8, f"V={V} top_p", stride=stride)


def test_deterministic_across_calls():
    z = sampler_logits("C2", 16)
    a = run(z, 128, 1 / 0.7, 0.95)
    b = run(z, 128, 1 / 0.7, 0.95)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("inv_t,top_p", [(1.0, 0.95), (1.0, 0.99), (1 / 0.7, 0.99)])
def test_nucleus_far_below_the_candidates(inv_t, top_p):
    # flat rows: nuclei of thousands of entries, beyond the one-pass
    # candidates, so their mass comes from the histogram and crossing-bin passes
    z = sampler_logits("C2", 48)
    _, _, cnt = check(z, 128, inv_t, top_p, f"wide nucleus inv_t={inv_t} top_p={top_p}")
    assert np.mean(cnt == 128) > 0.5


@pytest.mark.slow
@pytest.mark.parametrize("inv_t,top_p", [(1 / 0.7, 0.95), (1.0, 0.95)])
def test_full_batch_sampled_rows(inv_t, top_p):
    # all 4096 rows of the quick-check batch's sampler logits through the
    # persistent grid (rounds of rows per thread group, rows left to the exact
    # path between rounds); 192 sampled rows and the first and last compared
    z = sampler_logits("C2", 4096, seed=7)
    rng = np.random.default_rng(4096)
    rows = np.unique(np.concatenate([[0, 4095], rng.choice(4096, 192, replace=False)]))
    check(z, 128, inv_t, top_p, f"4096 rows inv_t={inv_t} top_p={top_p}", rows=rows)


@pytest.mark.slow
def test_run_time_hand_out_matches_the_launch_deal_and_leaves_the_workspace_zero():
    # the same rows with the last eighth handed out at run time and with every
    # row dealt at launch: the same bits (every sum has a fixed order)
    z = sampler_logits("C2", 2048, seed=9)
    outs = []
    for dynamic in (True, False, True):
        ids, lp, cnt = sc.sc_topk_capture(z, 128, 1 / 0.7, 0.95, dynamic=dynamic)
        torch.cuda.synchronize()
        outs.append((ids.cpu(), lp.cpu(), cnt.cpu()))
    for o in outs[1:]:
        for x, y in zip(outs[0], o):
            assert torch.equal(x, y)
    assert int(sc.workspace(torch.device("cuda")).abs().sum().item()) == 0
