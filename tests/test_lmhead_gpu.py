"""GPU parity of the LM head followed by score centering against the FP64 oracle.

With dyadic inputs (hidden on a 1/8 grid, the head on a 1/16 grid) the
logits H W^T are exact in FP32 for any d up to 2^14, so the library and the
oracle round the same logits to bf16 and the comparison isolates the kernels:
the score-centered gradient g is within one bf16 ulp (+1e-7) per element (the
fused kernel's bar), so dH = g W and dW = g^T H are, element by element,
within the sums of those errors times |W| and |H|, plus the bf16 rounding of
dH and FP32 accumulation (1e-6 of the sums of |g||W| and |g||H|).  The
element-wise cases run at the full sizes of the tensor-core tiles (d = 4096,
V = 151936, several row blocks, so dW is stored by the first block and added
to by the others).  With random bf16 weights the library's FP32 accumulation
can round a logit to the neighbouring bf16 value where the exact sum lies
near a rounding boundary, so that case is only a sanity check on the
relative Frobenius error.
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


def _case(b, block_rows, grad_scale, dw_rows=None):
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
    dH, dW, la, out, zb = oracle.lmhead_rows(Hb, Wb, batch, prm, dw_rows=dw_rows)
    G, _, _, _ = oracle.rows(dict(batch, logits=zb, V=b["V"]), prm)
    dw_gpu = dw if dw_rows is None else dw[torch.as_tensor(np.asarray(dw_rows), device=dw.device)]
    return dict(dh=bits_to_f64(_bits(dh)), dw=dw_gpu.cpu().numpy().astype(np.float64), lp=lp.cpu().numpy(),
                status=int(status.item()), flags=sc.diag_to_numpy(diag)["flags"], dH=dH, dW=dW, la=la, G=G,
                H=bits_to_f64(Hb), W=bits_to_f64(Wb), out=out)


def _check_elementwise(b, r, dw_rows=None):
    assert r["status"] == 0
    eg = ulp_bf16(r["G"]) + 1e-7
    aG = np.abs(r["G"])
    W, H = np.abs(r["W"]), np.abs(r["H"])
    tol_dh = eg @ W + ulp_bf16(r["dH"]) + 1e-6 * (aG @ W) + 1e-12
    sel = slice(None) if dw_rows is None else np.asarray(dw_rows)
    tol_dw = eg[:, sel].T @ H + 1e-6 * (aG[:, sel].T @ H) + 1e-12
    err_h = np.abs(r["dh"] - r["dH"])
    err_w = np.abs(r["dw"] - r["dW"])
    assert np.all(err_h <= tol_dh), f"dH off by {err_h.max():.3g} (ratio {(err_h / tol_dh).max():.3g})"
    assert np.all(err_w <= tol_dw), f"dW off by {err_w.max():.3g} (ratio {(err_w / tol_dw).max():.3g})"
    valid = b["row_response"].numpy() >= 0
    np.testing.assert_allclose(r["lp"][valid], r["la"][valid], rtol=0, atol=1e-4)
    assert np.all(r["lp"][~valid] == 0) and np.all(r["dh"][~valid] == 0)
    assert np.all((r["flags"][~valid] & sc.FLAG_MASKED) != 0)


@pytest.mark.parametrize("block_rows", [16, 40, 1024])
def test_dyadic_inputs_match_the_oracle(block_rows):
    # V = 1003 and d = 64: ragged tiles in every product (the logits' last
    # columns and dW's last rows)
    b = synth.lmhead_batch(40, 64, 1003, K=32, seed=11)
    n_valid = int((b["row_response"] >= 0).sum())
    _check_elementwise(b, _case(b, block_rows, 1.0 / n_valid))


@pytest.mark.slow
@pytest.mark.parametrize("block_rows", [128, 100])
def test_dyadic_full_tiles_element_by_element(block_rows):
    # d = 4096, V = 151936, 256 rows in 2 or 3 blocks: dH on every element,
    # dW on 384 sampled vocabulary rows (its full FP64 copy would take 5 GB)
    b = synth.lmhead_batch(256, 4096, 151936, K=128, seed=21, n_resp=8)
    n_valid = int((b["row_response"] >= 0).sum())
    rng = np.random.default_rng(block_rows)
    ids = b["rec_ids"].numpy().ravel()
    dw_rows = np.unique(np.concatenate([[0, 151935], rng.choice(ids, 128), rng.choice(151936, 254)]))
    _check_elementwise(b, _case(b, block_rows, 1.0 / n_valid, dw_rows=dw_rows), dw_rows)


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
