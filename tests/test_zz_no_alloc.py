"""The allocation-free variant of the fused call, against the regular one.

Some callers of this library are handed their input and output buffers and
nothing more (a plugin inside a framework that has already planned all of its
device memory, an embedded runtime that reserved its memory at start-up), so
they cannot pass the small workspace the regular call needs.
sc_center_forward_backward_noalloc serves them with a workspace kept inside
the library.  This test calls it through the C ABI twice in a row and checks
both results against the regular call on the same inputs, with the
tolerances of the parity tests.

The file name makes pytest collect it last; it also runs on its own in a
fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import precision_off_policy_gb300 as sc
import synth
from sc_parity import bits_to_f64, oracle_adv, sc_params, ulp_bf16

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _outputs(T, V, dev):
    return (torch.empty((T, V), dtype=torch.bfloat16, device=dev), torch.empty(T, dtype=torch.float32, device=dev),
            torch.zeros((T, 16), dtype=torch.int32, device=dev), torch.zeros(1, dtype=torch.int32, device=dev))


def test_noalloc_call_matches_the_regular_call_twice_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sc.build()
    L = sc.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    # 1024 rows at the full vocabulary: rows dealt round robin and handed out
    # at run time, padding rows included
    cfg = synth.config("C2", n_prompts=1, n_per_prompt=2, L_pad=512, len_lo=64, len_hi=512)
    b = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in synth.make_batch(cfg).items()}
    T, V = b["logits"].shape
    p = sc_params(b)
    adv = torch.as_tensor(oracle_adv(b), device=dev)
    stream = torch.cuda.current_stream(dev)

    g_ref, lp_ref, d_ref, st_ref = _outputs(T, V, dev)
    sc.sc_center_forward_backward(b["logits"], b["rec_ids"], b["rec_logprobs"], b["rec_count"], b["sampled"],
                                  b["rollout_logprob"], b["row_response"], adv, p, grad_out=g_ref, logp_out=lp_ref,
                                  diag_out=d_ref, status=st_ref, stream=stream)
    torch.cuda.synchronize()
    G = bits_to_f64(g_ref.view(torch.int16).cpu().numpy().view(np.uint16))
    tol = ulp_bf16(G) + 1e-7

    for call in range(2):
        g, lp, d, st = _outputs(T, V, dev)
        status = L.sc_center_forward_backward_noalloc(
            _ptr(b["logits"]), T, V, V, _ptr(b["rec_ids"]), _ptr(b["rec_logprobs"]), _ptr(b["rec_count"]),
            _ptr(b["sampled"]), _ptr(b["rollout_logprob"]), _ptr(b["row_response"]), _ptr(adv), adv.numel(),
            ctypes.byref(p), _ptr(g), V, _ptr(lp), _ptr(d), _ptr(st), ctypes.c_void_p(stream.cuda_stream))
        assert status == sc.SC_OK, L.sc_last_error().decode()
        torch.cuda.synchronize()
        assert int(st.item()) == int(st_ref.item()) == 0, f"call {call}: device status {int(st.item()):#x}"
        err = np.abs(bits_to_f64(g.view(torch.int16).cpu().numpy().view(np.uint16)) - G)
        assert np.all(err <= tol), f"call {call}: gradient off by {err.max()}"
        assert np.all(np.abs(lp.cpu().numpy() - lp_ref.cpu().numpy()) <= 1e-4), f"call {call}: log p_a"
        dn, dr = sc.diag_to_numpy(d), sc.diag_to_numpy(d_ref)
        assert np.array_equal(dn["flags"], dr["flags"]) and np.array_equal(dn["n_valid_k"], dr["n_valid_k"])
        for field in ("loss", "P_H", "Q_H", "rho", "s", "entropy", "row_sum"):
            np.testing.assert_allclose(dn[field], dr[field], rtol=1e-5, atol=1e-6, err_msg=f"call {call}: {field}")
