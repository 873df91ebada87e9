"""GPU parity of the LM head followed by score centering against the FP64 oracle.

With dyadic inputs (hidden on a 1/8 grid, the head on a 1/16 grid) the
logits H W^T are exact in FP32, so the library and the oracle round the same
logits to bf16 and the comparison isolates the kernels: the score-centered
gradient g is within one bf16 ulp (+1e-7) per element (the fused kernel's
bar), so dH = g W and dW = g^T H are within the sums of those errors times
|W| and |H|, plus the bf16 rounding of dH and FP32 accumulation.  With
random bf16 weights the library's FP32 accumulation can round a logit to the
neighbouring bf16 value where the exact sum lies near a rounding boundary;
there the check is on the relative Frobenius error.
"""

import numpy as np
import pytest
import torch

import oracle
import precision_off_policy_gb300 as sc
import synth
from sc_parity import bits_to_f64, ulp_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sc.build()
    sc.lib()


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _case(b, block_rows, grad_scale):
    dev = torch.device("cuda")
    x = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in b.items()}
    r = b["rewards"].numpy()
    adv = oracle.group_advantages(r, b["n_groups"], b["group_size"], True, 1e-6).astype(np.float32)
    p = sc.params(K_max=b["K"], grad_scale=grad_scale)
    T = b["hidden"].shape[0]
    diag = torch.zeros((T, 16), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    dh, dw, lp, _ = sc.sc_lmhead_forward_backward(
        x["hidden"], x["w"], x["rec_ids"], x["rec_logprobs"], None, x["sampled"], x["rollout_logprob"],
        x["row_response"], torch.as_tensor(adv, device=dev), p, block_rows=block_rows, diag_out=diag, status=status)
    torch.cuda.synchronize()
    batch = dict(rec_ids=b["rec_ids"].numpy(), rec_logprobs=b["rec_logprobs"].numpy(), rec_count=None,
                 sampled=b["sampled"].numpy(), rollout_logprob=b["rollout_logprob"].numpy(),
                 row_response=b["row_response"].numpy(), adv=adv)
    prm = oracle.make_params(grad_scale=float(np.float32(grad_scale)))
    Hb, Wb = _bits(b["hidden"]), _bits(b["w"])
    dH, dW, la, out, zb = oracle.lmhead_rows(Hb, Wb, batch, prm)
    G, _, _, _ = oracle.rows(dict(batch, logits=zb, V=b["V"]), prm)
    return dict(dh=bits_to_f64(_bits(dh)), dw=dw.cpu().numpy().astype(np.float64), lp=lp.cpu().numpy(),
                status=int(status.item()), flags=sc.diag_to_numpy(diag)["flags"], dH=dH, dW=dW, la=la, G=G,
                H=bits_to_f64(Hb), W=bits_to_f64(Wb), out=out)


@pytest.mark.parametrize("block_rows", [16, 40, 1024])
def test_dyadic_inputs_match_the_oracle(block_rows):
    b = synth.lmhead_batch(40, 64, 1003, K=32, seed=11)
    n_valid = int((b["row_response"] >= 0).sum())
    r = _case(b, block_rows, 1.0 / n_valid)
    assert r["status"] == 0
    eg = ulp_bf16(r["G"]) + 1e-7
    aG = np.abs(r["G"])
    tol_dh = eg @ np.abs(r["W"]) + ulp_bf16(r["dH"]) + 1e-6 * (aG @ np.abs(r["W"])) + 1e-12
    tol_dw = eg.T @ np.abs(r["H"]) + 1e-6 * (aG.T @ np.abs(r["H"])) + 1e-12
    err_h = np.abs(r["dh"] - r["dH"])
    err_w = np.abs(r["dw"] - r["dW"])
    assert np.all(err_h <= tol_dh), f"dH off by {err_h.max():.3g} (ratio {(err_h / tol_dh).max():.3g})"
    assert np.all(err_w <= tol_dw), f"dW off by {err_w.max():.3g} (ratio {(err_w / tol_dw).max():.3g})"
    valid = b["row_response"].numpy() >= 0
    np.testing.assert_allclose(r["lp"][valid], r["la"][valid], rtol=0, atol=1e-4)
    assert np.all(r["lp"][~valid] == 0) and np.all(r["dh"][~valid] == 0)
    assert np.all((r["flags"][~valid] & sc.FLAG_MASKED) != 0)


def test_random_weights_relative_error():
    b = synth.lmhead_batch(64, 256, 4096, K=64, seed=12, dyadic=False)
    r = _case(b, 24, 1.0 / 64)
    assert r["status"] == 0
    for got, ref, name in [(r["dh"], r["dH"], "dH"), (r["dw"], r["dW"], "dW")]:
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel <= 1e-2, f"{name}: relative Frobenius error {rel:.3g}"
    valid = b["row_response"].numpy() >= 0
    np.testing.assert_allclose(r["lp"][valid], r["la"][valid], rtol=0, atol=1e-3)


def test_rejects_bad_shapes_on_the_host():
    dev = torch.device("cuda")
    b = synth.lmhead_batch(8, 64, 100, K=8, seed=13)
    x = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in b.items()}
    adv = torch.zeros(4, dtype=torch.float32, device=dev)
    p = sc.params(K_max=8)
    with pytest.raises(sc.ScError):
        sc.sc_lmhead_forward_backward(x["hidden"][:, :60].contiguous(), x["w"][:, :60].contiguous(), x["rec_ids"],
                                      x["rec_logprobs"], None, x["sampled"], None, x["row_response"], adv, p)
    with pytest.raises(sc.ScError):
        sc.sc_lmhead_forward_backward(x["hidden"], x["w"], x["rec_ids"], x["rec_logprobs"], None, x["sampled"], None,
                                      x["row_response"], adv, p, block_rows=0)
