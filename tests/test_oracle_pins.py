"""Pins of the FP64 oracle against what the pages and the mathematics fix.

Nothing here runs the CUDA library.  Each test checks the oracle against
something other than itself: numbers printed on the pages (``tests/golden``),
hand-derived closed forms on designed inputs, library routines the method
reduces to (scipy's softmax / log-softmax / entropy, torch's bf16 cast),
finite differences of the loss, and brute-force expectations on tiny
vocabularies.

The method is the one of the "Score Centering" section of the Agent
Lightning docs page "Score Centering":
rho = max(1-Q_H,1e-6)/max(1-P_H,1e-6),
loss = -sg(A) [log p_a - sum_H sg(q_v - rho p_v) log p_v].
"""

import math
import os

import numpy as np
import pytest
import torch
from scipy.special import log_softmax, softmax
from scipy.stats import entropy as scipy_entropy

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
LN2 = math.log(2.0)


def bf16_bits(values):
    """bf16 bit patterns of float values, cast by torch (round to nearest even)."""
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().astype(np.uint16)


def bf16_values(bits):
    return oracle.bf16_to_double(bits)


def mu_hat_from_grad(g, a, coef):
    """Invert g = coef * (e_a - mu_hat) for mu_hat."""
    e = np.zeros_like(g)
    e[a] = 1.0
    return e - g / coef


# --------------------------------------------------------------------------
# bf16 rounding: the lecture's printed numbers and torch's cast.


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def test_bf16_rounding_golden():
    seen = set()
    for parts in _golden_lines("bf16_rounding.txt"):
        kind = parts[0]
        seen.add(kind)
        if kind == "round":
            assert oracle.bf16_round(float(parts[1])) == float(parts[2])
        elif kind == "steps":
            start, inc, n = float(parts[1]), float(parts[2]), int(parts[3])
            copy = oracle.bf16_round(start)
            master, steps = start, 0
            while oracle.bf16_round(master) == copy:
                master += inc
                steps += 1
                assert steps < 10_000
            assert steps == n
        elif kind == "grid":
            x, k, e = float(parts[1]), int(parts[2]), int(parts[3])
            assert oracle.bf16_round(x) == k * 2.0**e
        elif kind == "spacing":
            x, e = float(parts[1]), int(parts[2])
            v = oracle.bf16_round(x)
            up = oracle.bf16_round(v + 0.75 * 2.0**e)
            assert up - v == 2.0**e
    assert seen == {"round", "steps", "grid", "spacing"}


def test_bf16_rne_matches_torch_cast_on_random_floats():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 10.0,
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),  # subnormal range
        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.3895313e38], dtype=np.float32),
    ])
    ours = np.array([oracle.bf16_bits(float(v)) for v in x], dtype=np.uint16)
    np.testing.assert_array_equal(ours, bf16_bits(x))


def test_bf16_decode_round_trip_all_finite_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bf16_values(bits)
    finite = np.isfinite(vals)
    back = np.array([oracle.bf16_bits(float(v)) for v in vals[finite]], dtype=np.uint16)
    # -0.0 and +0.0 keep their sign bits; every finite pattern maps back to itself.
    np.testing.assert_array_equal(back, bits[finite])
    assert bf16_values(np.array([0x3F80]))[0] == 1.0
    assert bf16_values(np.array([0xC000]))[0] == -2.0


# --------------------------------------------------------------------------
# Group advantages (docs "Training": group std normalisation; release note
# section 4: mean-only variant, fractional rewards kept).


def test_advantages_closed_form_one_success_in_four():
    # mean 0.25, unbiased std 0.5 -> (1 - 0.25) / 0.5 = 1.5 and -0.5.
    A = oracle.group_advantages([1, 0, 0, 0], 1, 4, True, 0.0)
    np.testing.assert_allclose(A, [1.5, -0.5, -0.5, -0.5], rtol=0, atol=1e-15)
    A = oracle.group_advantages([1, 0, 0, 0], 1, 4, True, 1e-6)
    np.testing.assert_allclose(A, np.array([0.75, -0.25, -0.25, -0.25]) / (0.5 + 1e-6), rtol=1e-15)


def test_advantages_all_equal_group_is_exactly_zero():
    for r in ([0, 0, 0, 0], [1, 1, 1, 1], [0.3, 0.3, 0.3, 0.3], [7.0]):
        A = oracle.group_advantages(r, 1, len(r), True, 1e-6)
        assert np.all(A == 0.0)


def test_advantages_keep_fractional_rewards_distinct():
    # Release note section 4: 1.0 and 1.001 collapsed once rewards were cast to
    # bf16 first; in the advantage computation they must stay distinct.
    assert oracle.bf16_round(1.001) == oracle.bf16_round(1.0)
    A = oracle.group_advantages([1.0, 1.001], 1, 2, True, 0.0)
    assert A[0] < 0 < A[1]
    np.testing.assert_allclose(A, [-1 / math.sqrt(2), 1 / math.sqrt(2)], rtol=1e-6)


def test_advantages_mean_only_and_no_overflow():
    A = oracle.group_advantages([3.0, 1.0, 2.0], 1, 3, False, 1e-6)
    np.testing.assert_allclose(A, [1.0, -1.0, 0.0], atol=1e-15)
    # Squares of these rewards overflow binary32; the std must not.
    big = np.array([3e30, -3e30, 1e30, -1e30], dtype=np.float32).astype(np.float64)
    A = oracle.group_advantages(big, 1, 4, True, 1e-6)
    std = np.std(big, ddof=1)
    np.testing.assert_allclose(A, big / std, rtol=1e-12)


def test_advantages_several_groups_match_numpy_per_group():
    rng = np.random.default_rng(3)
    r = rng.random((8, 8)).astype(np.float32)
    A = oracle.group_advantages(r.ravel(), 8, 8, True, 1e-6).reshape(8, 8)
    rd = r.astype(np.float64)
    ref = (rd - rd.mean(1, keepdims=True)) / (rd.std(1, ddof=1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(A, ref, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# A hand-worked row (closed form) and a clamped row.


def test_hand_worked_dyadic_row():
    # z = [2,1,0,0] at inverse temperature ln 2 gives p = [1/2, 1/4, 1/8, 1/8].
    # H = {0, 1} with q = [0.6, 0.3]:  P_H = 3/4, Q_H = 0.9, rho = 0.1/0.25 = 0.4,
    # c = [0.6-0.2, 0.3-0.1] = [0.4, 0.2], s = 1 - 0.9 + 0.4*0.75 = 0.4,
    # mu_hat = [0.6, 0.3, 0.05, 0.05].  With a = 2, A = 1:
    # loss = -(log 1/8 - 0.4 log 1/2 - 0.2 log 1/4) = 2.2 ln 2,
    # grad = ln2 * (-1) * (e_2 - mu_hat) = ln2 * [0.6, 0.3, -0.95, 0.05],
    # entropy = 1.75 ln 2.
    z = bf16_bits([2, 1, 0, 0])
    p = oracle.make_params(inv_temperature=LN2)
    g, o = oracle.row(z, [0, 1], np.log([0.6, 0.3]).astype(np.float32), a=2, A=1.0, params=p)
    tol = dict(rtol=0, atol=2e-7)
    np.testing.assert_allclose(o["P_H"], 0.75, **tol)
    np.testing.assert_allclose(o["Q_H"], 0.9, **tol)
    np.testing.assert_allclose(o["rho"], 0.4, **tol)
    np.testing.assert_allclose(o["s"], 0.4, **tol)
    np.testing.assert_allclose(o["loss"], 2.2 * LN2, **tol)
    np.testing.assert_allclose(o["logp_a"], -3 * LN2, **tol)
    np.testing.assert_allclose(o["entropy"], 1.75 * LN2, **tol)
    np.testing.assert_allclose(g, LN2 * np.array([0.6, 0.3, -0.95, 0.05]), **tol)
    assert o["flags"] == 0 and o["n_valid_k"] == 2


def test_sampled_token_inside_head():
    # Same row, a = 0 (inside H):  grad = ln2 * (-1) * (e_0 - mu_hat)
    # = ln2 * [-0.4, 0.3, 0.05, 0.05];  loss = -(log 1/2 - (-0.8 ln2)) = 0.2 ln 2... with
    # log p_0 = -ln2:  -( -ln2 + 0.8 ln2 ) = 0.2 ln2.
    z = bf16_bits([2, 1, 0, 0])
    p = oracle.make_params(inv_temperature=LN2)
    g, o = oracle.row(z, [0, 1], np.log([0.6, 0.3]).astype(np.float32), a=0, A=1.0, params=p)
    np.testing.assert_allclose(g, LN2 * np.array([-0.4, 0.3, 0.05, 0.05]), atol=2e-7)
    np.testing.assert_allclose(o["loss"], 0.2 * LN2, atol=2e-7)


def test_clamped_denominator_row():
    # z = [1,0,0] at inverse temperature 20: 1 - P_H = 2e^-20/(1+2e^-20) ~ 4.1e-9 < 1e-6,
    # so the denominator clamps and rho = max(0.01, 1e-6)/1e-6 = 1e4 (q_0 = 0.99).
    # Off H the reconstructed mu_hat is s * p_v with s = 1 - Q_H + rho P_H, which
    # under the clamp is no longer rho (s = rho + 0.01 - rho (1 - P_H)).
    z = bf16_bits([1, 0, 0])
    p = oracle.make_params(inv_temperature=20.0)
    lp0 = np.float32(np.log(0.99))
    q0 = math.exp(float(lp0))
    g, o = oracle.row(z, [0], [lp0], a=1, A=1.0, params=p)
    eps = 2 * math.exp(-20) / (1 + 2 * math.exp(-20))
    # 1 - P_H in double precision carries ~1e-15 absolute error: ~1e-6 relative here.
    np.testing.assert_allclose(o["tail_pi"], eps, rtol=1e-5)
    np.testing.assert_allclose(o["rho"], (1 - q0) / 1e-6, rtol=1e-12)
    assert o["flags"] & oracle.FLAG_CLAMP_PI and not o["flags"] & oracle.FLAG_CLAMP_MU
    mu_hat = mu_hat_from_grad(g, 1, -20.0)
    pv = math.exp(-20) / (1 + 2 * math.exp(-20))
    rho = (1 - q0) / 1e-6
    np.testing.assert_allclose(o["s"], (1 - q0) + rho * (1 - eps), rtol=1e-12)
    np.testing.assert_allclose(mu_hat[1:], ((1 - q0) + rho * (1 - eps)) * pv, rtol=1e-9)
    np.testing.assert_allclose(mu_hat.sum(), 1.0, atol=1e-12)


def test_both_clamps_give_rho_one():
    # H = everything with sum q = 1 - 1e-9: both tails below 1e-6, rho = 1e-6/1e-6 = 1.
    z = bf16_bits([0.5, -0.25, 1.0])
    q = softmax(bf16_values(z))
    lp = np.log(q).astype(np.float32)
    g, o = oracle.row(z, [0, 1, 2], lp, a=2, A=2.0)
    assert o["rho"] == 1.0
    assert o["flags"] & oracle.FLAG_CLAMP_PI and o["flags"] & oracle.FLAG_CLAMP_MU


# --------------------------------------------------------------------------
# Reductions to library routines.


def _random_row(rng, V, scale=2.0):
    return bf16_bits(rng.standard_normal(V) * scale)


@pytest.mark.parametrize("inv_t", [1.0, 1 / 0.7])
def test_empty_head_reduces_to_plain_policy_gradient(inv_t):
    # K = 0: P_H = Q_H = 0, rho = 1, s = 1, no centering term: the loss is
    # -A log p_a and the gradient is (1/T)(-A)(e_a - softmax(z/T)).
    rng = np.random.default_rng(11)
    z = _random_row(rng, 300)
    x = bf16_values(z) * inv_t
    a, A = 17, -0.8
    g, o = oracle.row(z, [], [], a=a, A=A, params=oracle.make_params(inv_temperature=inv_t))
    ref = inv_t * (-A) * (np.eye(300)[a] - softmax(x))
    np.testing.assert_allclose(g, ref, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(o["loss"], -A * log_softmax(x)[a], rtol=1e-12)
    assert o["rho"] == 1.0 and o["s"] == 1.0


def test_logp_and_entropy_match_scipy():
    rng = np.random.default_rng(12)
    z = _random_row(rng, 1000, 3.0)
    ids = rng.choice(1000, 40, replace=False).astype(np.int32)
    lp = np.log(rng.random(40) / 80).astype(np.float32)
    x = bf16_values(z) / 0.7
    g, o = oracle.row(z, ids, lp, a=5, A=1.0, params=oracle.make_params(inv_temperature=1 / 0.7))
    np.testing.assert_allclose(o["logp_a"], log_softmax(x)[5], rtol=1e-12)
    np.testing.assert_allclose(o["entropy"], scipy_entropy(softmax(x)), rtol=1e-10)
    np.testing.assert_allclose(o["P_H"], softmax(x)[ids].sum(), rtol=1e-12)
    np.testing.assert_allclose(o["Q_H"], np.exp(lp.astype(np.float64)).sum(), rtol=1e-12)


def test_matching_recorded_head_gives_uncentered_gradient():
    # q = p on p's own top-K: every c_v = q_v - rho p_v vanishes up to the
    # binary32 rounding of the recorded logprobs, and mu_hat = p.
    rng = np.random.default_rng(13)
    V, K = 2000, 128
    z = _random_row(rng, V, 3.0)
    x = bf16_values(z)
    pi = softmax(x)
    ids = np.argsort(-pi)[:K].astype(np.int32)
    lp = log_softmax(x)[ids].astype(np.float32)
    a, A = int(ids[3]), 1.3
    g, o = oracle.row(z, ids, lp, a=a, A=A)
    ref = (-A) * (np.eye(V)[a] - pi)
    np.testing.assert_allclose(g, ref, rtol=0, atol=1e-6 * abs(A))
    np.testing.assert_allclose(o["rho"], 1.0, rtol=1e-5)


def test_full_head_with_unit_mass_gives_mu_hat_equal_q():
    # K >= V and sum q = 1: mu_hat = q + (1 - Q_H) p = q.
    rng = np.random.default_rng(14)
    V = 64
    z = _random_row(rng, V)
    q = rng.dirichlet(np.ones(V))
    lp = np.log(q).astype(np.float32)
    ids = rng.permutation(V).astype(np.int32)
    a, A = 9, 0.7
    g, o = oracle.row(z, ids, lp[ids], a=a, A=A)
    mu_hat = mu_hat_from_grad(g, a, -A)
    np.testing.assert_allclose(mu_hat, np.exp(lp.astype(np.float64)), atol=1e-6)


# --------------------------------------------------------------------------
# Finite differences of the loss with the stop-gradient constants held fixed.


@pytest.mark.parametrize("inv_t,seed,clamp", [(1.0, 21, False), (1 / 0.7, 22, False), (6.0, 23, True)])
def test_gradient_matches_central_differences(inv_t, seed, clamp):
    rng = np.random.default_rng(seed)
    V, K = 24, 7
    z = _random_row(rng, V, 2.0)
    ids = rng.choice(V, K, replace=False).astype(np.int32)
    if clamp:
        z = bf16_bits(np.where(np.arange(V) == ids[0], 8.0, bf16_values(z)))
    lp = np.log(rng.dirichlet(np.ones(K)) * 0.9).astype(np.float32)
    a, A = int(rng.integers(V)), -1.7
    g, o = oracle.row(z, ids, lp, a=a, A=A, params=oracle.make_params(inv_temperature=inv_t))
    assert bool(o["flags"] & oracle.FLAG_CLAMP_PI) == clamp
    zf = bf16_values(z)
    pi0 = softmax(zf * inv_t)
    c = np.exp(lp.astype(np.float64)) - o["rho"] * pi0[ids]  # held constant (sg)

    def loss(zz):
        l = log_softmax(zz * inv_t)
        return -A * (l[a] - np.dot(c, l[ids]))

    np.testing.assert_allclose(loss(zf), o["loss"], rtol=1e-10, atol=1e-13)
    h = 1e-5
    fd = np.empty(V)
    for v in range(V):
        e = np.zeros(V)
        e[v] = h
        fd[v] = (loss(zf + e) - loss(zf - e)) / (2 * h)
    # truncation error ~ h^2 |f'''| and cancellation error ~ eps |loss| / h
    atol = 1e-8 * max(1.0, inv_t) ** 3 + 1e-15 * abs(o["loss"]) / h
    np.testing.assert_allclose(g, fd, rtol=1e-6, atol=atol)


# --------------------------------------------------------------------------
# Structure: row sums, the proportional-tail reading, brute force.


def test_row_sums_vanish_with_and_without_clamps():
    rng = np.random.default_rng(31)
    for trial in range(20):
        V = int(rng.integers(2, 400))
        K = int(rng.integers(0, min(V, 128) + 1))
        z = _random_row(rng, V, float(rng.choice([1.0, 3.0, 12.0])))
        ids = rng.choice(V, K, replace=False).astype(np.int32)
        lp = np.log(rng.dirichlet(np.ones(max(K, 1)))[:K] * rng.random()).astype(np.float32)
        A = float(rng.standard_normal())
        g, o = oracle.row(z, ids, lp, a=int(rng.integers(V)), A=A)
        assert abs(g.sum()) <= 1e-12 * max(abs(A), 1e-300) * max(1.0, o["rho"])
        assert abs(o["row_sum"]) <= 1e-12 * max(abs(A), 1e-300) * max(1.0, o["rho"])


def test_unclamped_mu_hat_is_q_on_head_and_proportional_to_p_elsewhere():
    # The docs page models the behaviour mass outside the recorded ids as the
    # current policy scaled to that mass: mu_hat = q on H and rho * p off H,
    # total mass 1.
    rng = np.random.default_rng(32)
    V, K = 500, 50
    z = _random_row(rng, V, 2.0)
    ids = rng.choice(V, K, replace=False).astype(np.int32)
    lp = np.log(rng.dirichlet(np.ones(K)) * 0.8).astype(np.float32)
    a, A = 77, 0.9
    g, o = oracle.row(z, ids, lp, a=a, A=A)
    assert o["flags"] == 0
    mu_hat = mu_hat_from_grad(g, a, -A)
    np.testing.assert_allclose(mu_hat[ids], np.exp(lp.astype(np.float64)), rtol=1e-10, atol=1e-15)
    off = np.setdiff1d(np.arange(V), ids)
    pi = softmax(bf16_values(z))
    ratio = mu_hat[off] / pi[off]
    np.testing.assert_allclose(ratio, ratio[0], rtol=1e-9)
    np.testing.assert_allclose(ratio[0], (1 - np.exp(lp.astype(np.float64)).sum()) / (1 - pi[ids].sum()),
                               rtol=1e-10)
    np.testing.assert_allclose(mu_hat.sum(), 1.0, atol=1e-12)


@pytest.mark.parametrize("V", [2, 5, 9, 16])
def test_brute_force_expected_centered_score(V):
    # Enumerate every sampled token a ~ mu and every head size K = 0..V:
    #  (1) mu_hat does not depend on a;
    #  (2) E_{a~mu}[g] = coef * (mu - mu_hat);
    #  (3) when mu's unrecorded tail is proportional to p, E_{a~mu}[g] = 0.
    rng = np.random.default_rng(100 + V)
    z = _random_row(rng, V, 1.5)
    pi = softmax(bf16_values(z))
    A = 1.25
    for K in range(V + 1):
        order = rng.permutation(V)
        ids = order[:K].astype(np.int32)
        mu = rng.dirichlet(np.ones(V))
        lp = np.log(mu[ids]).astype(np.float32)
        qH = np.exp(lp.astype(np.float64))
        # (1) and (2) with an arbitrary behaviour distribution
        mu_eff = mu.copy()
        mu_eff[ids] = qH
        mu_eff /= mu_eff.sum()
        grads = np.stack([oracle.row(z, ids, lp, a=a, A=A)[0] for a in range(V)])
        mh = [mu_hat_from_grad(grads[a], a, -A) for a in range(V)]
        for a in range(1, V):
            np.testing.assert_allclose(mh[a], mh[0], atol=1e-14)
        np.testing.assert_allclose(mu_eff @ grads, -A * (mu_eff - mh[0]), atol=1e-14)
        # (3) behaviour distribution whose tail is proportional to p
        tail_mu = 1.0 - qH.sum()
        off = order[K:]
        mu_prop = np.zeros(V)
        mu_prop[ids] = qH
        if K < V:
            mu_prop[off] = tail_mu * pi[off] / pi[off].sum()
            if tail_mu < 1e-6 or pi[off].sum() < 1e-6:
                continue  # a clamp is active: the proportional tail is not reproduced
        np.testing.assert_allclose(mu_prop @ grads, 0.0, atol=1e-12 if K < V else 2e-6)


# --------------------------------------------------------------------------
# Head hygiene readings: out-of-range ids are dropped, repeats after the first.


def test_duplicate_and_out_of_range_ids_are_dropped():
    rng = np.random.default_rng(41)
    V = 100
    z = _random_row(rng, V)
    ids = np.array([4, 9, 4, 150, -3, 22], dtype=np.int32)
    lp = np.log(np.array([0.2, 0.1, 0.3, 0.05, 0.05, 0.1])).astype(np.float32)
    g, o = oracle.row(z, ids, lp, a=5, A=1.0)
    keep = [0, 1, 5]
    g2, o2 = oracle.row(z, ids[keep], lp[keep], a=5, A=1.0)
    np.testing.assert_array_equal(g, g2)
    assert o["n_valid_k"] == 3
    assert o["flags"] & oracle.FLAG_DUP_ID and o["flags"] & oracle.FLAG_BAD_ID
    assert o2["flags"] == 0


def test_bad_sampled_id_is_an_error_row():
    z = bf16_bits([0.1, 0.2, 0.3])
    g, o = oracle.row(z, [0], np.log([0.5]).astype(np.float32), a=3, A=1.0)
    assert np.all(g == 0) and o["flags"] == oracle.FLAG_BAD_SAMPLED


# --------------------------------------------------------------------------
# Importance weighting (settings table: is_mode none / tis / mis, tis_max,
# mis_min, mis_max, centering) and the lecture's TIS worked numbers.


def _two_token_row(p0):
    """z and inverse temperature giving p = (p0, 1 - p0) exactly (up to fp64)."""
    return bf16_bits([0.0, -1.0]), math.log(p0 / (1 - p0))


def test_tis_worked_numbers():
    for parts in _golden_lines("tis_worked_example.txt"):
        pi_a, mu_a, wmax, w, wt, bias = map(float, parts)
        z, inv_t = _two_token_row(pi_a)
        rl = float(np.float32(math.log(mu_a)))
        mu_seen = math.exp(rl)
        prm = oracle.make_params(is_mode=oracle.IS_TIS, tis_max=wmax, inv_temperature=inv_t)
        g, o = oracle.row(z, [], [], a=0, A=1.0, params=prm, rollout_logprob=rl)
        np.testing.assert_allclose(math.exp(o["logp_a"]), pi_a, rtol=1e-12)
        np.testing.assert_allclose(pi_a / mu_seen, w, rtol=1e-6)
        np.testing.assert_allclose(o["is_weight"], wt, rtol=1e-6)
        assert bool(o["flags"] & oracle.FLAG_IS_TRUNC) == (w > wmax)
        # the weight scales the plain score: g = (1/T)(-A wt)(e_a - p)
        np.testing.assert_allclose(g, inv_t * (-o["is_weight"]) * (np.array([1, 0]) - [pi_a, 1 - pi_a]),
                                   rtol=1e-10)
        np.testing.assert_allclose(max(0.0, pi_a - wmax * mu_a), bias, atol=1e-12)


def test_tis_bias_closed_form_by_enumeration():
    # E_pi[f] - E_mu[min(w, wmax) f] = sum_{w > wmax} (pi - wmax mu) f, with the
    # truncated weights read from the oracle for each sampled token.
    z, inv_t = _two_token_row(0.20)
    pi = np.array([0.20, 0.80])
    mu = np.array([0.01, 0.99])
    f = np.array([1.7, -0.4])
    prm = oracle.make_params(is_mode=oracle.IS_TIS, tis_max=2.0, inv_temperature=inv_t,
                             centering=False)
    wt = np.array([oracle.row(z, [], [], a=a, A=1.0, params=prm,
                              rollout_logprob=math.log(mu[a]))[1]["is_weight"] for a in range(2)])
    lhs = pi @ f - (mu * wt) @ f
    w = pi / mu
    rhs = np.sum(np.where(w > 2.0, pi - 2.0 * mu, 0.0) * f)
    np.testing.assert_allclose(lhs, rhs, atol=1e-6)
    np.testing.assert_allclose(rhs, 0.18 * f[0], atol=1e-12)


def test_mis_rejects_outside_interval_and_keeps_inside():
    for pi_a, mu_a, keep in [(0.55, 0.50, True), (0.20, 0.01, False), (0.2, 0.5, False)]:
        z, inv_t = _two_token_row(pi_a)
        prm = oracle.make_params(is_mode=oracle.IS_MIS, inv_temperature=inv_t)
        g, o = oracle.row(z, [], [], a=0, A=1.0, params=prm, rollout_logprob=math.log(mu_a))
        if keep:
            np.testing.assert_allclose(o["is_weight"], pi_a / mu_a, rtol=1e-6)
            assert not o["flags"] & oracle.FLAG_IS_REJECT
        else:
            assert o["is_weight"] == 0.0 and np.all(g == 0.0)
            assert o["flags"] & oracle.FLAG_IS_REJECT


def test_centering_off_is_plain_weighted_score():
    rng = np.random.default_rng(51)
    V = 200
    z = _random_row(rng, V)
    ids = rng.choice(V, 30, replace=False).astype(np.int32)
    lp = np.log(rng.dirichlet(np.ones(30)) * 0.7).astype(np.float32)
    prm = oracle.make_params(centering=False)
    g, o = oracle.row(z, ids, lp, a=3, A=-2.0, params=prm)
    np.testing.assert_allclose(g, 2.0 * (np.eye(V)[3] - softmax(bf16_values(z))), rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(o["loss"], 2.0 * log_softmax(bf16_values(z))[3], rtol=1e-12)


# --------------------------------------------------------------------------
# K3 diagnostic (docs "Score Centering", last paragraph).


def test_k3_zero_when_rollout_logprob_matches():
    rng = np.random.default_rng(61)
    z = _random_row(rng, 50)
    _, o = oracle.row(z, [], [], a=4, A=1.0)
    _, o2 = oracle.row(z, [], [], a=4, A=1.0, rollout_logprob=o["logp_a"])
    assert abs(o2["k3"]) < 1e-15


def test_k3_is_nonnegative_and_second_order():
    rng = np.random.default_rng(62)
    z = _random_row(rng, 50)
    _, o = oracle.row(z, [], [], a=4, A=1.0)
    for d in [1e-3, -1e-3, 0.5, -2.0]:
        _, o2 = oracle.row(z, [], [], a=4, A=1.0, rollout_logprob=o["logp_a"] - d)
        assert o2["k3"] >= 0
        if abs(d) <= 1e-3:
            np.testing.assert_allclose(o2["k3"], d * d / 2, rtol=2e-3)


# --------------------------------------------------------------------------
# Batch entry: masked rows, error rows, ragged counts.


def test_batch_masks_padding_and_flags_bad_rows():
    rng = np.random.default_rng(71)
    T, V, Kmax = 6, 40, 5
    logits = bf16_bits(rng.standard_normal((T, V)))
    ids = np.stack([rng.choice(V, Kmax, replace=False) for _ in range(T)]).astype(np.int32)
    lp = np.log(np.full((T, Kmax), 0.1)).astype(np.float32)
    batch = dict(logits=logits, V=V, rec_ids=ids, rec_logprobs=lp,
                 rec_count=np.array([5, 0, 3, 9, 2, 1], np.int32),
                 sampled=np.array([1, 2, 3, 4, 5, 6], np.int32), rollout_logprob=None,
                 row_response=np.array([0, 1, -1, 0, 2, 1], np.int32),
                 adv=np.array([0.5, -1.0], np.float32))
    g, la, out, _ = oracle.rows(batch, oracle.make_params(), nthreads=3)
    assert out["flags"][2] == oracle.FLAG_MASKED and np.all(g[2] == 0) and la[2] == 0
    assert out["flags"][4] == oracle.FLAG_BAD_RESPONSE and np.all(g[4] == 0)
    assert out["flags"][3] & oracle.FLAG_BAD_COUNT and out["n_valid_k"][3] == 5
    assert out["n_valid_k"][1] == 0
    for t in (0, 1, 5):
        k = batch["rec_count"][t]
        g1, o1 = oracle.row(logits[t], ids[t, :k], lp[t, :k], a=batch["sampled"][t],
                            A=float(batch["adv"][batch["row_response"][t]]))
        np.testing.assert_array_equal(g[t], g1)
        assert out["loss"][t] == o1["loss"]


# --------------------------------------------------------------------------
# Clipped GRPO baseline (the `grpo` preset of the docs page's "Training"
# section: clipped objective, clip widths 0.2 / 0.3, per-rollout mean loss).


def _clip_case(rng, V, w_target, A, inv_t=1.0, lo=0.2, hi=0.3):
    z = _random_row(rng, V, 2.0)
    a = int(rng.integers(V))
    zf = bf16_values(z)
    lpa = log_softmax(zf * inv_t)[a]
    old = float(np.float32(lpa - np.log(w_target)))
    prm = oracle.make_params(is_mode=oracle.IS_CLIP, centering=False, inv_temperature=inv_t,
                             clip_low=lo, clip_high=hi)
    g, o = oracle.row(z, [], [], a=a, A=A, params=prm, rollout_logprob=old)
    return z, zf, a, old, g, o


@pytest.mark.parametrize("w_target,A,active", [
    (1.0, 1.3, True), (1.1, -0.8, True),        # inside the clip range: the ratio's gradient
    (1.6, 1.3, False), (0.5, -0.8, False),      # clipped term is the minimum: no gradient
    (0.5, 1.3, True), (1.6, -0.8, True),        # unclipped term is the minimum: gradient flows
    # between the widths (1 - 0.3 < w < 1 - 0.2, 1 + 0.2 < w < 1 + 0.3): the
    # lower width 0.2 clips 0.75, the upper width 0.3 keeps 1.25 inside
    (0.75, -0.8, False), (1.25, 1.3, True),
])
def test_clipped_grpo_gradient_matches_central_differences(w_target, A, active):
    rng = np.random.default_rng(int(w_target * 100) + (7 if A > 0 else 11))
    V, inv_t, lo, hi = 20, 1.25, 0.2, 0.3
    z, zf, a, old, g, o = _clip_case(rng, V, w_target, A, inv_t, lo, hi)

    def loss(zz):
        w = np.exp(log_softmax(zz * inv_t)[a] - old)
        return -min(w * A, min(max(w, 1 - lo), 1 + hi) * A)

    np.testing.assert_allclose(loss(zf), o["loss"], rtol=1e-12)
    assert bool(o["flags"] & oracle.FLAG_CLIPPED) == (not active)
    h = 1e-6
    fd = np.array([(loss(zf + h * np.eye(V)[v]) - loss(zf - h * np.eye(V)[v])) / (2 * h) for v in range(V)])
    np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-8)
    if not active:
        assert np.all(g == 0.0) and o["is_weight"] == 0.0


def test_clipped_grpo_at_unit_ratio_is_the_plain_policy_gradient():
    rng = np.random.default_rng(5)
    V, A, inv_t = 37, -1.1, 1 / 0.7
    z, zf, a, old, g, o = _clip_case(rng, V, 1.0, A, inv_t)
    # ratio 1 (up to the FP32 rounding of the old log-probability)
    w = np.exp(log_softmax(zf * inv_t)[a] - old)
    p = softmax(zf * inv_t)
    ref = inv_t * (-A * w) * (np.eye(V)[a] - p)
    np.testing.assert_allclose(g, ref, rtol=1e-12, atol=1e-15)
    assert abs(o["loss"] + A * w) <= 1e-12
    assert abs(g.sum()) <= 1e-12


def test_clipped_grpo_rejects_centering():
    rng = np.random.default_rng(6)
    z = _random_row(rng, 8, 1.0)
    prm = oracle.make_params(is_mode=oracle.IS_CLIP, centering=True)
    with pytest.raises(ValueError):
        oracle.row(z, [], [], a=0, A=1.0, params=prm, rollout_logprob=-1.0)


def test_rollout_mean_advantages_hand_counts():
    adv = np.array([1.5, -0.5, -0.5, -0.5, 2.0])
    rr = np.array([0, 0, 0, 1, -1, 3, 3, 3, 3, 1, 7, -1], dtype=np.int32)  # 7 is out of range
    out, counts = oracle.rollout_mean_advantages(adv, rr, 5)
    assert counts.tolist() == [3, 2, 0, 4, 0]
    np.testing.assert_array_equal(out, [0.5, -0.25, 0.0, -0.125, 0.0])
    # agrees with a bincount over the valid response indices
    ok = (rr >= 0) & (rr < 5)
    assert counts.tolist() == np.bincount(rr[ok], minlength=5).tolist()


# --------------------------------------------------------------------------
# Sampler-side top-K capture (the top K behaviour probabilities recorded per
# generated position, docs page "Score Centering").


def test_topk_capture_hand_worked_nucleus():
    # p = [1/2, 1/4, 1/8, 1/8]; top_p 0.7: the mass before entry 1 is 1/2 < 0.7 and
    # before entry 2 it is 3/4 >= 0.7, so the nucleus is {0, 1} with mass 3/4.
    z = np.log(np.array([[4.0, 2.0, 1.0, 1.0]])).astype(np.float32)
    ids, lp, cnt = oracle.topk_capture(z, 3, 1.0, 0.7)
    assert ids.tolist() == [[0, 1, -1]] and cnt.tolist() == [2]
    np.testing.assert_allclose(lp[0, :2], np.log([2 / 3, 1 / 3]), rtol=1e-6)
    ids, lp, cnt = oracle.topk_capture(z, 3, 1.0, 1.0)
    assert ids.tolist() == [[0, 1, 2]] and cnt.tolist() == [3]  # the tie 2/3 goes to the lower id
    np.testing.assert_allclose(lp[0], np.log([0.5, 0.25, 0.125]), rtol=1e-6)


def test_topk_capture_equal_logits_and_short_rows():
    z = np.full((2, 300), 1.25, dtype=np.float32)
    ids, lp, cnt = oracle.topk_capture(z, 128)
    assert np.all(ids == np.arange(128)) and np.all(cnt == 128)
    np.testing.assert_allclose(lp, -np.log(300.0), rtol=1e-6)
    ids, lp, cnt = oracle.topk_capture(z[:, :5], 8)  # K > V: every id, then padding
    assert ids[0].tolist() == [0, 1, 2, 3, 4, -1, -1, -1] and cnt.tolist() == [5, 5]


def test_topk_capture_geometric_closed_form():
    # z_v = -v ln 2 at inv_t = 1: p_v = 2^-v / S with S = 2 (1 - 2^-V)
    V, K = 60, 16
    z = (-np.arange(V) * np.log(2.0)).astype(np.float32)[None, :]
    S = 2.0 * (1.0 - 2.0 ** -V)
    zz = z[0].astype(np.float64)
    ids, lp, cnt = oracle.topk_capture(z, K)
    assert ids[0].tolist() == list(range(K))
    np.testing.assert_allclose(lp[0], zz[:K] - np.log(np.exp(zz).sum()), rtol=1e-6)
    np.testing.assert_allclose(lp[0], -np.arange(K) * np.log(2.0) - np.log(S), rtol=1e-5)
    # top_p 0.9: the mass before entry n is (1 - 2^-n) / (1 - 2^-V); it first reaches 0.9 at n = 4
    ids, lp, cnt = oracle.topk_capture(z, K, 1.0, 0.9)
    assert cnt.tolist() == [4] and ids[0, :4].tolist() == [0, 1, 2, 3]
    nuc = (1.0 - 2.0 ** -4) / (1.0 - 2.0 ** -V)
    np.testing.assert_allclose(lp[0, :4], -np.arange(4) * np.log(2.0) - np.log(S) - np.log(nuc), rtol=1e-5)


@pytest.mark.parametrize("inv_t,top_p", [(1.0, 1.0), (1 / 0.7, 1.0), (1 / 0.7, 0.95), (2.0, 0.5)])
def test_topk_capture_selection_invariants(inv_t, top_p):
    rng = np.random.default_rng(int(inv_t * 10 + top_p * 100))
    T, V, K = 6, 2000, 64
    z = (rng.standard_normal((T, V)) * 3.0).astype(np.float32)
    z[:, 100:140] = z[:, 99:100]  # a run of equal values
    ids, lp, cnt = oracle.topk_capture(z, K, inv_t, top_p)
    for t in range(T):
        c = cnt[t]
        sel = ids[t, :c]
        assert np.all(ids[t, c:] == -1) and len(set(sel.tolist())) == c
        rest = np.setdiff1d(np.arange(V), sel)
        # every selected value is at least every unselected one; among equal values the lower ids win
        assert z[t, sel].min() >= z[t, rest].max()
        edge = z[t, sel].min()
        assert np.all(rest[z[t, rest] == edge] > sel[z[t, sel] == edge].max())
        # sorted by value, larger first
        assert np.all(np.diff(z[t, sel].astype(np.float64)) <= 0)
        ls = log_softmax(z[t].astype(np.float64) * inv_t)
        if top_p == 1.0:
            assert c == K
            np.testing.assert_allclose(lp[t, :c], ls[sel], rtol=1e-6, atol=1e-6)
        else:
            # brute force: the nucleus is the shortest sorted prefix whose preceding mass is below top_p
            order = np.lexsort((np.arange(V), -z[t].astype(np.float64)))
            before = np.concatenate([[0.0], np.cumsum(np.exp(ls[order]))[:-1]])
            n_keep = int((before < top_p).sum())
            assert c == min(K, n_keep)
            nuc = np.exp(ls[order[:n_keep]]).sum()
            np.testing.assert_allclose(lp[t, :c], ls[sel] - np.log(nuc), rtol=1e-6, atol=1e-6)


# --------------------------------------------------------------------------
# The LM head followed by score centering (z = bf16(H W^T); dH = g W, dW = g^T H).


def _lmhead_case(rng, T=4, d=5, V=12, K=3, inv_t=1.0):
    # small integers: z = H W^T is an integer of a few bits, exact in bf16
    H = rng.integers(-2, 3, size=(T, d)).astype(np.float64)
    W = rng.integers(-2, 3, size=(V, d)).astype(np.float64)
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(T)]).astype(np.int32)
    lp = np.log(rng.dirichlet(np.ones(K), size=T) * 0.8).astype(np.float32)
    sampled = rng.integers(0, V, size=T).astype(np.int32)
    resp = np.array([0, 1, -1, 1][:T], dtype=np.int32)
    adv = np.array([0.9, -1.3], dtype=np.float32)
    batch = dict(rec_ids=ids, rec_logprobs=lp, rec_count=None, sampled=sampled, rollout_logprob=None,
                 row_response=resp, adv=adv)
    return H, W, batch


@pytest.mark.parametrize("inv_t,seed", [(1.0, 41), (1 / 0.7, 42)])
def test_lmhead_gradients_match_central_differences(inv_t, seed):
    rng = np.random.default_rng(seed)
    H, W, batch = _lmhead_case(rng, inv_t=inv_t)
    scale = 0.25
    prm = oracle.make_params(inv_temperature=inv_t, grad_scale=scale)
    dH, dW, la, out, zb = oracle.lmhead_rows(bf16_bits(H), bf16_bits(W), batch, prm)
    assert np.array_equal(bf16_values(zb), H @ W.T)  # exact here: the rounding is the identity
    T = H.shape[0]
    # the batch loss with every row's stop-gradient constants c held at the base point
    consts = []
    for t in range(T):
        if batch["row_response"][t] < 0:
            consts.append(None)
            continue
        p0 = softmax((H[t] @ W.T) * inv_t)
        ids = batch["rec_ids"][t]
        c = np.exp(batch["rec_logprobs"][t].astype(np.float64)) - out["rho"][t] * p0[ids]
        consts.append((ids, c, int(batch["sampled"][t]), float(batch["adv"][batch["row_response"][t]])))

    def loss(HH, WW):
        tot = 0.0
        for t, k in enumerate(consts):
            if k is None:
                continue
            ids, c, a, A = k
            l = log_softmax((HH[t] @ WW.T) * inv_t)
            tot += -A * (l[a] - np.dot(c, l[ids]))
        return scale * tot

    np.testing.assert_allclose(loss(H, W), scale * out["loss"].sum(), rtol=1e-12)
    h = 1e-6
    fdH = np.zeros_like(H)
    for i in np.ndindex(H.shape):
        e = np.zeros_like(H)
        e[i] = h
        fdH[i] = (loss(H + e, W) - loss(H - e, W)) / (2 * h)
    fdW = np.zeros_like(W)
    for i in np.ndindex(W.shape):
        e = np.zeros_like(W)
        e[i] = h
        fdW[i] = (loss(H, W + e) - loss(H, W - e)) / (2 * h)
    np.testing.assert_allclose(dH, fdH, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dW, fdW, rtol=1e-6, atol=1e-8)
    assert np.all(dH[2] == 0)  # the padding row contributes nothing


def test_lmhead_with_identity_head_reduces_to_the_row_oracle():
    # W = I (V = d): z = bf16(H), dH is the rows' gradient itself and dW = g^T H.
    rng = np.random.default_rng(43)
    T, d, K = 6, 40, 8
    Hb = bf16_bits(rng.standard_normal((T, d)) * 2.0)
    Wb = bf16_bits(np.eye(d))
    ids = np.stack([rng.choice(d, K, replace=False) for _ in range(T)]).astype(np.int32)
    lp = np.log(rng.dirichlet(np.ones(K), size=T) * 0.9).astype(np.float32)
    batch = dict(rec_ids=ids, rec_logprobs=lp, rec_count=None, sampled=rng.integers(0, d, T).astype(np.int32),
                 rollout_logprob=None, row_response=np.array([0, 0, 1, 1, -1, 0], np.int32),
                 adv=np.array([1.1, -0.4], np.float32))
    prm = oracle.make_params()
    dH, dW, la, out, zb = oracle.lmhead_rows(Hb, Wb, batch, prm)
    assert np.array_equal(zb, Hb)
    g, la2, out2, _ = oracle.rows(dict(batch, logits=Hb, V=d), prm)
    np.testing.assert_array_equal(dH, g)
    np.testing.assert_allclose(dW, g.T @ bf16_values(Hb), rtol=1e-15, atol=0)
    np.testing.assert_array_equal(la, la2)


def test_lmhead_logits_are_the_rounded_fp64_products():
    # Non-dyadic inputs: each logit is the FP64 product H W^T (exact here: 24
    # products of bf16 values need far fewer than 53 bits) rounded once by the
    # scalar bf16 rounding pinned above; some entries round up in magnitude, so
    # truncation would differ there.
    rng = np.random.default_rng(45)
    T, d, V, K = 5, 24, 40, 4
    Hb = bf16_bits(rng.standard_normal((T, d)))
    Wb = bf16_bits(rng.standard_normal((V, d)) * 0.3)
    batch = dict(rec_ids=np.stack([rng.choice(V, K, replace=False) for _ in range(T)]).astype(np.int32),
                 rec_logprobs=np.log(rng.dirichlet(np.ones(K), size=T) * 0.8).astype(np.float32), rec_count=None,
                 sampled=rng.integers(0, V, T).astype(np.int32), rollout_logprob=None,
                 row_response=np.array([0, 0, 1, 1, -1], np.int32), adv=np.array([0.7, -1.2], np.float32))
    _, _, _, _, zb = oracle.lmhead_rows(Hb, Wb, batch, oracle.make_params())
    prod = bf16_values(Hb) @ bf16_values(Wb).T
    expected = np.array([oracle.bf16_bits(float(x)) for x in prod.ravel()], dtype=np.uint16).reshape(T, V)
    np.testing.assert_array_equal(zb, expected)
    assert np.any(np.abs(bf16_values(expected)) > np.abs(prod))


def test_bf16_round_array_matches_the_scalar_rounding():
    rng = np.random.default_rng(44)
    x = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-6, 6, 2000), [0.0, -0.0, 1.0 + 2.0**-8]])
    got = oracle.bf16_round_array(x)
    ref = np.array([oracle.bf16_bits(float(v)) for v in x], dtype=np.uint16)
    np.testing.assert_array_equal(got, ref)
    assert got[-1] == 0x3F80  # the tie 1 + 2^-8 rounds to even (1.0)
