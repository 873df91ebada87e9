"""Helpers for the parity tests: run the CUDA library, run the oracle, compare.

Tolerances (stated by the method's target accuracy and derived where it
gives none):

* gradient elements: |g_gpu - g_oracle| <= 1 bf16 ulp of g_oracle + 1e-7
  (times |grad_scale| when a scale other than 1 is used);
* log p_a: |delta| <= 1e-4;
* row sums: the bf16 output row sums to within 1e-3 |A| (scaled) plus half
  an ulp per element (rounding alone can exceed the bare bound on flat
  rows); the kernel's FP32 sum before rounding to within 1e-3 |A| max(1,
  rho), a bound on FP32 rounding derived in `fp32_row_sum_bound`;
* diagnostics: relative 1e-4 with small absolute floors, as listed in
  `check_diag`.

The oracle always gets its inputs from the seeded generator and its own
advantages (oracle.group_advantages), never from the CUDA path.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import precision_off_policy_gb300 as sc
import synth

CLAMP_BITS = oracle.FLAG_CLAMP_PI | oracle.FLAG_CLAMP_MU
IS_BITS = oracle.FLAG_IS_TRUNC | oracle.FLAG_IS_REJECT | oracle.FLAG_CLIPPED


def ulp_bf16(x):
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0**-126)))
    return np.exp2(e - 7)


def bits_to_f64(bits):
    return oracle.bf16_to_double(bits)


def oracle_adv(batch) -> np.ndarray:
    """FP32 advantages from the oracle's own group statistics."""
    r = batch["rewards"].detach().cpu().numpy()
    return oracle.group_advantages(r, batch["n_groups"], batch["group_size"], True, 1e-6).astype(np.float32)


def sc_params(batch, **kw):
    kw.setdefault("K_max", batch["rec_ids"].shape[1])
    kw.setdefault("inv_temperature", batch["inv_temperature"])
    return sc.params(**kw)


def oracle_params(p: sc.Params):
    # The library takes its scalars in FP32; the oracle takes the same values.
    return oracle.make_params(is_mode=p.is_mode, tis_max=p.tis_max, mis_min=p.mis_min, mis_max=p.mis_max,
                              centering=bool(p.centering), inv_temperature=float(np.float32(p.inv_temperature)),
                              grad_scale=float(np.float32(p.grad_scale)), clip_low=p.clip_low,
                              clip_high=p.clip_high)


def run_gpu(batch, p, adv: np.ndarray, inplace=False, with_rollout=True, stream=None):
    """Runs sc_center_forward_backward on cuda:0.  Returns (grad, logp, diag, status) on the device.

    When V is not a multiple of 8 the rows are stored with a stride rounded up
    to 8 entries (the ABI's 16-byte row alignment); the returned gradient is
    then the [T, V] view."""
    dev = torch.device("cuda")
    b = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in batch.items()}
    T, V = b["logits"].shape
    stride = (V + 7) // 8 * 8
    diag = torch.zeros((T, 16), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if stride == V:
        logits = b["logits"].clone() if inplace else b["logits"]
    else:
        logits = torch.zeros((T, stride), dtype=torch.bfloat16, device=dev)
        logits[:, :V] = b["logits"]
    grad = logits if inplace else torch.empty((T, stride), dtype=torch.bfloat16, device=dev)
    _, lp, d = sc.sc_center_forward_backward(
        logits, b["rec_ids"], b["rec_logprobs"], b["rec_count"], b["sampled"],
        b["rollout_logprob"] if with_rollout else None, b["row_response"],
        torch.as_tensor(adv, device=dev), p, V=V, grad_out=grad, diag_out=diag, status=status,
        stream=stream)
    torch.cuda.synchronize()
    return grad[:, :V], lp, d, status


def host_batch(batch, adv, with_rollout=True) -> dict:
    bn = synth.to_numpy(batch)
    bn["adv"] = adv
    if not with_rollout:
        bn["rollout_logprob"] = None
    return bn


def check_rows(bn: dict, p: sc.Params, rows, g_bits: np.ndarray, logp: np.ndarray, diag: np.ndarray,
               nthreads: int = 0, what: str = ""):
    """Compares GPU rows with the oracle element by element.  Returns the oracle outputs."""
    rows = np.asarray(rows, dtype=np.int64)
    po = oracle_params(p)
    G, LA, OUT, _ = oracle.rows(bn, po, rows, nthreads=nthreads)
    g = bits_to_f64(g_bits)
    scale = max(1.0, abs(float(np.float32(p.grad_scale))))
    tol = ulp_bf16(G) + 1e-7 * scale
    err = np.abs(g - G)
    bad = err > tol
    if bad.any():
        r, v = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {bad.sum()} gradient elements out of tolerance; first at row {rows[r]} v={v}: "
            f"gpu={g[r, v]!r} oracle={G[r, v]!r} tol={tol[r, v]!r}; flags={OUT['flags'][r]:#x}")
    np.testing.assert_allclose(logp, LA, rtol=0, atol=1e-4, err_msg=f"{what}: log p_a")
    rl = bn.get("rollout_logprob")
    d_or = LA - rl[rows].astype(np.float64) if rl is not None else np.zeros_like(LA)
    check_diag(diag, OUT, p, what, d_or)
    check_row_sums(g, diag, OUT, p, what)
    return G, LA, OUT


def check_diag(d: np.ndarray, o: np.ndarray, p: sc.Params, what: str, d_or=None):
    masked = (o["flags"] & (oracle.FLAG_MASKED | oracle.FLAG_BAD_RESPONSE | oracle.FLAG_BAD_SAMPLED)) != 0
    # flags: exact, except decisions taken at a floating-point threshold
    # (clamps, importance-weight bounds), compared only away from it below.
    np.testing.assert_array_equal(d["flags"] & ~np.uint32(CLAMP_BITS | IS_BITS),
                                  o["flags"] & ~np.uint32(CLAMP_BITS | IS_BITS), err_msg=f"{what}: flags")
    np.testing.assert_array_equal(d["n_valid_k"], o["n_valid_k"], err_msg=f"{what}: n_valid_k")
    if masked.any():
        for f in ["loss", "logp_a", "P_H", "rho", "entropy", "row_sum"]:
            assert np.all(d[f][masked] == 0), f"{what}: {f} nonzero on masked rows"
    v = ~masked
    if not v.any():
        return
    dv, ov = d[v], o[v]
    near = lambda x, thr, rel: np.abs(x - thr) <= rel * thr
    for bit, field in [(oracle.FLAG_CLAMP_PI, "tail_pi"), (oracle.FLAG_CLAMP_MU, "tail_mu")]:
        sure = ~near(ov[field], 1e-6, 1e-3)
        np.testing.assert_array_equal((dv["flags"] & bit)[sure], (ov["flags"] & bit)[sure], err_msg=f"{what}: {field} clamp")
    for f, rtol, atol in [("P_H", 1e-4, 1e-6), ("Q_H", 1e-5, 1e-6), ("entropy", 1e-4, 1e-5)]:
        np.testing.assert_allclose(dv[f], ov[f], rtol=rtol, atol=atol, err_msg=f"{what}: {f}")
    np.testing.assert_allclose(dv["tail_pi"], ov["tail_pi"], rtol=1e-3, atol=1e-9, err_msg=f"{what}: tail_pi")
    np.testing.assert_allclose(dv["tail_mu"], ov["tail_mu"], rtol=1e-3, atol=2e-7, err_msg=f"{what}: tail_mu")
    np.testing.assert_allclose(dv["rho"], ov["rho"], rtol=2e-3, atol=0, err_msg=f"{what}: rho")
    np.testing.assert_allclose(dv["s"], ov["s"], rtol=2e-3, atol=1e-6, err_msg=f"{what}: s")
    np.testing.assert_allclose(dv["adv"], ov["adv"], rtol=0, atol=0, err_msg=f"{what}: adv")
    A = np.abs(ov["adv"] * ov["is_weight"])
    # loss = -A_w (log p_a - sum_H c log p): log p_a carries 1e-4, the centred sum
    # the same relative error.
    lossscale = A * (1.0 + np.abs(ov["logp_a"])) + np.abs(ov["loss"])
    assert np.all(np.abs(dv["loss"] - ov["loss"]) <= 1e-4 * lossscale + 1e-6), f"{what}: loss"
    # k3 = e^d - 1 - d with d carrying the 1e-4 of log p_a: |dk3| <= |e^d - 1| * 1e-4
    dd = np.zeros(v.sum()) if d_or is None else d_or[v]
    dk3 = 1e-4 * np.abs(np.expm1(dd)) + 1e-4 * np.abs(ov["k3"]) + 1e-6
    assert np.all(np.abs(dv["k3"] - ov["k3"]) <= dk3), f"{what}: k3"
    np.testing.assert_allclose(dv["is_weight"], ov["is_weight"], rtol=1e-3, atol=1e-7, err_msg=f"{what}: is_weight")


def fp32_row_sum_bound(o: np.ndarray, p: sc.Params) -> np.ndarray:
    """Bound on the kernel's FP32 row sum (diag field `row_sum`).

    The kernel forms it as the sum of the values its write pass stores,
    beta p_v on every entry, plus, for the recorded ids and the sampled token,
    the difference between their own gradient and beta p_v.  Those terms add
    up to at most |a| (s + 1 + Q_H + rho P_H) <= 5 |a| max(1, rho) in absolute
    value (a = grad_scale A_w / T, s <= 1 + rho), and FP32 rounding of the
    terms (each exponent argument rounded once, at most 2^-24 |y| with |y| <=
    64 in the bits that matter) and of the summation tree (at most a few
    hundred additions deep for any launch plan) stays below 400 * 2^-24 of
    that sum: under 1.2e-4 |a| max(1, rho).  The check uses 1e-3 |a|
    max(1, rho).  When rho >> 1 (the trainer's tail mass clamped at 1e-6)
    beta = -a s is of order a rho and the cancellation between the write
    pass's sum and the corrections is real; the bf16 output itself holds the
    patched values and needs no rho (see check_row_sums)."""
    a = np.abs(o["adv"] * o["is_weight"]) * abs(float(np.float32(p.grad_scale))) * float(np.float32(p.inv_temperature))
    return 1e-3 * a * np.maximum(1.0, o["rho"]) + 1e-7


def bf16_row_sum_allowance(g: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp per nonzero element: the most round-to-nearest-even can
    move a row's sum."""
    return 0.5 * ulp_bf16(g).sum(axis=1) * (np.abs(g) > 0).any(axis=1)


def check_row_sums(g: np.ndarray, d: np.ndarray, o: np.ndarray, p: sc.Params, what: str):
    """Every gradient row sums to zero.  The FP32 row sum the kernel reports is
    held to fp32_row_sum_bound; the bf16 output row to the target 1e-3 |a|
    (a = grad_scale A_w / T) plus the rounding allowance, with no rho factor:
    its entries sum to at most 4 |a| in absolute value in every regime."""
    assert np.all(np.abs(d["row_sum"]) <= fp32_row_sum_bound(o, p)), f"{what}: FP32 row sum"
    a = np.abs(o["adv"] * o["is_weight"]) * abs(float(np.float32(p.grad_scale))) * float(np.float32(p.inv_temperature))
    assert np.all(np.abs(g.sum(axis=1)) <= 1e-3 * a + bf16_row_sum_allowance(g) + 1e-7), f"{what}: bf16 row sum"


def bare_row_sum_fraction(g: np.ndarray, o: np.ndarray, p: sc.Params) -> float:
    """Fraction of the rows with a nonzero advantage whose bf16 output sums to
    within the bare 1e-3 |a|, with no rounding allowance."""
    a = np.abs(o["adv"] * o["is_weight"]) * abs(float(np.float32(p.grad_scale))) * float(np.float32(p.inv_temperature))
    live = a > 0
    if not live.any():
        return 1.0
    return float(np.mean(np.abs(g.sum(axis=1))[live] <= 1e-3 * a[live]))


def grad_bits(g: torch.Tensor, rows) -> np.ndarray:
    idx = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=g.device)
    return g.index_select(0, idx).cpu().view(torch.int16).numpy().view(np.uint16)


def diag_rows(d: torch.Tensor, rows) -> np.ndarray:
    idx = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=d.device)
    return sc.diag_to_numpy(d.index_select(0, idx))
