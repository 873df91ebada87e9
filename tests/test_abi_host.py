"""Host-side checks of the C ABI: no GPU needed.

The library must load, export every function `include/sc.h` declares, and
reject bad arguments on the host -- before any CUDA call -- with the status
codes the header documents.  Pointer arguments here are fake addresses that
are never dereferenced: validation fails before anything touches them.
"""

import ctypes
import os
import re

import pytest

import precision_off_policy_gb300 as sc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sc.h")


@pytest.fixture(scope="module")
def L():
    sc.build()
    return sc.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(sc_\w+)\s*\(", text, re.M)))


def test_header_declares_the_documented_entry_points():
    names = declared_functions()
    assert "sc_group_advantages" in names and "sc_center_forward_backward" in names
    assert set(names) == set(sc.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_struct_layouts_match_header(L):
    assert ctypes.sizeof(sc.Params) == 64
    assert sc.DIAG_DTYPE.itemsize == 64
    p = sc.Params()
    assert L.sc_params_default(ctypes.byref(p)) == sc.SC_OK
    assert (p.K_max, p.is_mode, p.tis_max, p.mis_min, p.mis_max, p.centering) == (128, 0, 2.0, 0.5, 5.0, 1)
    assert (p.inv_temperature, p.grad_scale, p.cluster_size, p.threads, p.stages) == (1.0, 1.0, 0, 0, 0)
    assert (p.clip_low, p.clip_high, p.flag_layout) == (pytest.approx(0.2), pytest.approx(0.3), 0)
    assert (p.wait_limit_us, p.test_stall) == (0, 0)
    assert L.sc_params_default(None) == sc.SC_ERR_NULL
    assert L.sc_abi_version() == 106
    assert L.sc_status_string(sc.SC_ERR_ALIGN) == b"misaligned pointer or stride"


FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced


def call_center(L, T=4, V=64, lstride=64, gstride=64, logits=FAKE, grad=FAKE * 2, ids=FAKE * 3,
                lps=FAKE * 4, cnt=None, samp=FAKE * 5, roll=None, resp=FAKE * 6, adv=FAKE * 7, n_resp=2,
                logp=FAKE * 8, diag=None, status=None, ws=FAKE * 11, **pk):
    raw_centering = pk.pop("centering", None)
    p = sc.params(**{"K_max": 8, **pk})
    if raw_centering is not None:
        p.centering = raw_centering  # bypass the binding's bool() to reach the C check
    return L.sc_center_forward_backward(logits, T, V, lstride, ids, lps, cnt, samp, roll, resp, adv, n_resp,
                                        ctypes.byref(p), grad, gstride, logp, diag, status, ws, None)


def err(L):
    return L.sc_last_error().decode()


@pytest.mark.parametrize("kw,status", [
    (dict(V=0), sc.SC_ERR_SHAPE),
    (dict(V=(1 << 20) + 1, lstride=(1 << 20) + 8, gstride=(1 << 20) + 8), sc.SC_ERR_SHAPE),
    (dict(T=-1), sc.SC_ERR_SHAPE),
    (dict(K_max=1025), sc.SC_ERR_SHAPE),
    (dict(K_max=-1), sc.SC_ERR_SHAPE),
    (dict(n_resp=-1), sc.SC_ERR_SHAPE),
    (dict(lstride=32), sc.SC_ERR_SHAPE),
    (dict(inv_temperature=0.0), sc.SC_ERR_ARG),
    (dict(inv_temperature=float("inf")), sc.SC_ERR_ARG),
    (dict(grad_scale=float("nan")), sc.SC_ERR_ARG),
    (dict(is_mode=4), sc.SC_ERR_ARG),
    (dict(is_mode=3, roll=FAKE * 9), sc.SC_ERR_ARG),                              # clip needs centering 0
    (dict(is_mode=3, roll=FAKE * 9, centering=0, clip_low=1.0), sc.SC_ERR_ARG),
    (dict(is_mode=3, roll=FAKE * 9, centering=0, clip_high=-0.1), sc.SC_ERR_ARG),
    (dict(is_mode=3, roll=FAKE * 9, centering=0, clip_high=float("inf")), sc.SC_ERR_ARG),
    (dict(is_mode=3, centering=0), sc.SC_ERR_NULL),                                # clip needs the old logprob
    (dict(is_mode=1, roll=FAKE * 9, tis_max=0.0), sc.SC_ERR_ARG),
    (dict(is_mode=2, roll=FAKE * 9, mis_min=3.0, mis_max=1.0), sc.SC_ERR_ARG),
    (dict(is_mode=1), sc.SC_ERR_NULL),
    (dict(centering=2), sc.SC_ERR_ARG),
    (dict(cluster_size=17), sc.SC_ERR_ARG),
    (dict(threads=100), sc.SC_ERR_ARG),
    (dict(stages=5), sc.SC_ERR_ARG),
    (dict(flag_layout=3), sc.SC_ERR_ARG),
    (dict(flag_layout=-1), sc.SC_ERR_ARG),
    (dict(wait_limit_us=-1), sc.SC_ERR_ARG),
    (dict(wait_limit_us=60000001), sc.SC_ERR_ARG),
    (dict(test_stall=2), sc.SC_ERR_ARG),
    (dict(logits=None), sc.SC_ERR_NULL),
    (dict(grad=None), sc.SC_ERR_NULL),
    (dict(logp=None), sc.SC_ERR_NULL),
    (dict(samp=None), sc.SC_ERR_NULL),
    (dict(resp=None), sc.SC_ERR_NULL),
    (dict(adv=None), sc.SC_ERR_NULL),
    (dict(ids=None), sc.SC_ERR_NULL),
    (dict(ws=None), sc.SC_ERR_NULL),
    (dict(ws=FAKE * 11 + 8), sc.SC_ERR_ALIGN),
    (dict(logits=FAKE + 2), sc.SC_ERR_ALIGN),
    (dict(grad=FAKE * 2 + 8), sc.SC_ERR_ALIGN),
    (dict(lstride=68), sc.SC_ERR_ALIGN),
    (dict(gstride=66), sc.SC_ERR_ALIGN),
    (dict(samp=FAKE * 5 + 2), sc.SC_ERR_ALIGN),
    (dict(diag=FAKE * 10 + 4), sc.SC_ERR_ALIGN),
    (dict(grad=FAKE + 64), sc.SC_ERR_ARG),                       # partial overlap with logits
    (dict(grad=FAKE, gstride=72, lstride=64), sc.SC_ERR_ARG),    # same base, different stride
])
def test_center_rejects_bad_arguments_on_the_host(L, kw, status):
    assert call_center(L, **kw) == status, err(L)
    assert err(L) != ""


def test_center_empty_batch_is_a_no_op(L):
    assert call_center(L, T=0, logits=None, grad=None, samp=None, resp=None, logp=None, ws=None) == sc.SC_OK
    assert err(L) == ""


def test_center_null_params(L):
    assert L.sc_center_forward_backward(FAKE, 1, 8, 8, None, None, None, FAKE, None, FAKE, FAKE, 1, None,
                                        FAKE * 2, 8, FAKE * 3, None, None, FAKE * 4, None) == sc.SC_ERR_NULL


def test_no_gpu_reaches_cuda_not_a_crash(L):
    # Arguments that pass validation reach the CUDA runtime; without a GPU
    # that reports an error status instead of crashing.
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call_center(L) in (sc.SC_ERR_CUDA, sc.SC_ERR_UNSUPPORTED)


def call_center_noalloc(L, **kw):
    """The allocation-free entry point with call_center's arguments (no workspace)."""
    kw = dict(kw)
    kw.pop("ws", None)
    T, V = kw.pop("T", 4), kw.pop("V", 8)
    p = sc.params(K_max=8)
    return L.sc_center_forward_backward_noalloc(kw.get("logits", FAKE), T, V, 8, FAKE * 5, FAKE * 6, None,
                                                kw.get("samp", FAKE * 7), None, kw.get("resp", FAKE * 10),
                                                FAKE * 12, 2, ctypes.byref(p), kw.get("grad", FAKE * 2), 8,
                                                kw.get("logp", FAKE * 8), None, None, None)


def test_noalloc_empty_batch_is_a_no_op(L):
    assert call_center_noalloc(L, T=0, logits=None, grad=None, samp=None, resp=None, logp=None) == sc.SC_OK
    assert err(L) == ""


@pytest.mark.parametrize("kw,status", [
    (dict(logits=FAKE + 2), sc.SC_ERR_ALIGN),
    (dict(samp=None), sc.SC_ERR_NULL),
    (dict(grad=None), sc.SC_ERR_NULL),
    (dict(V=0), sc.SC_ERR_SHAPE),
])
def test_noalloc_checks_its_arguments_before_anything_else(L, kw, status):
    # the same host-side checks as the regular call, before the library's
    # array is looked up or cleared (these fail even without a GPU)
    assert call_center_noalloc(L, **kw) == status, err(L)
    assert err(L) != ""


def test_noalloc_without_a_gpu_reports_a_status(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call_center_noalloc(L) in (sc.SC_ERR_CUDA, sc.SC_ERR_UNSUPPORTED)
    assert err(L) != ""


@pytest.mark.parametrize("args,status", [
    ((FAKE, -1, 4, 1, 1e-6, FAKE * 2), sc.SC_ERR_SHAPE),
    ((FAKE, 2, 0, 1, 1e-6, FAKE * 2), sc.SC_ERR_SHAPE),
    ((FAKE, 2, 65537, 1, 1e-6, FAKE * 2), sc.SC_ERR_SHAPE),
    ((FAKE, 2, 4, 1, -1.0, FAKE * 2), sc.SC_ERR_ARG),
    ((FAKE, 2, 4, 1, float("nan"), FAKE * 2), sc.SC_ERR_ARG),
    ((None, 2, 4, 1, 1e-6, FAKE * 2), sc.SC_ERR_NULL),
    ((FAKE, 2, 4, 1, 1e-6, None), sc.SC_ERR_NULL),
    ((FAKE + 2, 2, 4, 1, 1e-6, FAKE * 2), sc.SC_ERR_ALIGN),
    ((FAKE, 2, 4, 1, 1e-6, FAKE + 4), sc.SC_ERR_ARG),  # partial overlap
    ((None, 0, 4, 1, 1e-6, None), sc.SC_OK),            # nothing to do
])
def test_group_advantages_host_validation(L, args, status):
    assert L.sc_group_advantages(*args, None) == status, err(L)


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(sc._build_mod, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(sc, "_lib", None)
    with pytest.raises(sc.ScError):
        sc.lib()
    monkeypatch.undo()
    assert sc.lib() is not None


@pytest.mark.parametrize("args,status", [
    ((FAKE, FAKE * 2, -1, 4, FAKE * 3, FAKE * 4), sc.SC_ERR_SHAPE),
    ((FAKE, FAKE * 2, 8, -1, FAKE * 3, FAKE * 4), sc.SC_ERR_SHAPE),
    ((None, FAKE * 2, 8, 4, FAKE * 3, FAKE * 4), sc.SC_ERR_NULL),
    ((FAKE, None, 8, 4, FAKE * 3, FAKE * 4), sc.SC_ERR_NULL),
    ((FAKE, FAKE * 2, 8, 4, None, FAKE * 4), sc.SC_ERR_NULL),
    ((FAKE, FAKE * 2, 8, 4, FAKE * 3, None), sc.SC_ERR_NULL),
    ((FAKE + 2, FAKE * 2, 8, 4, FAKE * 3, FAKE * 4), sc.SC_ERR_ALIGN),
    ((FAKE, FAKE * 2 + 1, 8, 4, FAKE * 3, FAKE * 4), sc.SC_ERR_ALIGN),
])
def test_rollout_mean_rejects_bad_arguments_on_the_host(L, args, status):
    assert L.sc_rollout_mean_advantages(*args, None) == status, err(L)


def test_rollout_mean_no_responses_is_a_no_op(L):
    assert L.sc_rollout_mean_advantages(None, None, 8, 0, None, None, None) == sc.SC_OK


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), sc.SC_ERR_SHAPE),
    (dict(V=0), sc.SC_ERR_SHAPE),
    (dict(K=0), sc.SC_ERR_SHAPE),
    (dict(K=1025), sc.SC_ERR_SHAPE),
    (dict(stride=60), sc.SC_ERR_SHAPE),
    (dict(inv_t=0.0), sc.SC_ERR_ARG),
    (dict(top_p=0.0), sc.SC_ERR_ARG),
    (dict(top_p=1.5), sc.SC_ERR_ARG),
    (dict(logits=None), sc.SC_ERR_NULL),
    (dict(ids=None), sc.SC_ERR_NULL),
    (dict(lps=None), sc.SC_ERR_NULL),
    (dict(logits=FAKE + 4), sc.SC_ERR_ALIGN),
    (dict(stride=66), sc.SC_ERR_ALIGN),
    (dict(cnt=FAKE * 4 + 2), sc.SC_ERR_ALIGN),
    (dict(ws=FAKE * 5 + 8), sc.SC_ERR_ALIGN),
])
def test_topk_capture_rejects_bad_arguments_on_the_host(L, kw, status):
    a = dict(logits=FAKE, T=3, V=64, stride=64, inv_t=1.0, K=8, top_p=1.0, ids=FAKE * 2, lps=FAKE * 3, cnt=None,
             ws=None)
    a.update(kw)
    assert L.sc_topk_capture(a["logits"], a["T"], a["V"], a["stride"], a["inv_t"], a["K"], a["top_p"], a["ids"],
                             a["lps"], a["cnt"], a["ws"], None) == status, err(L)


def test_topk_capture_empty_batch_is_a_no_op(L):
    assert L.sc_topk_capture(None, 0, 64, 64, 1.0, 8, 1.0, None, None, None, None, None) == sc.SC_OK


def call_lmhead(L, T=4, d=64, V=100, hidden=FAKE, w=FAKE * 2, ids=FAKE * 3, lps=FAKE * 4, samp=FAKE * 5,
                resp=FAKE * 6, adv=FAKE * 7, dh=FAKE * 8, dw=FAKE * 9, logp=FAKE * 10, ws=FAKE * 256,
                ws_bytes=None, block_rows=2, **pk):
    p = sc.params(**{"K_max": 8, **pk})
    if ws_bytes is None:
        ws_bytes = L.sc_lmhead_workspace_bytes(min(block_rows, T) if block_rows > 0 else 1, V, d if d > 0 else 8)
    return L.sc_lmhead_forward_backward(hidden, w, T, d, V, ids, lps, None, samp, None, resp, adv, 2,
                                        ctypes.byref(p), block_rows, dh, dw, logp, None, None, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(d=60), sc.SC_ERR_SHAPE),
    (dict(d=0), sc.SC_ERR_SHAPE),
    (dict(V=0), sc.SC_ERR_SHAPE),
    (dict(T=-1), sc.SC_ERR_SHAPE),
    (dict(block_rows=0), sc.SC_ERR_SHAPE),
    (dict(K_max=2000), sc.SC_ERR_SHAPE),
    (dict(inv_temperature=0.0), sc.SC_ERR_ARG),
    (dict(hidden=None), sc.SC_ERR_NULL),
    (dict(dw=None), sc.SC_ERR_NULL),
    (dict(ws=None), sc.SC_ERR_NULL),
    (dict(logp=None), sc.SC_ERR_NULL),
    (dict(ids=None), sc.SC_ERR_NULL),
    (dict(hidden=FAKE + 8), sc.SC_ERR_ALIGN),
    (dict(ws=FAKE * 256 + 16), sc.SC_ERR_ALIGN),
    (dict(ws_bytes=256 + 2 * 104 * 2 - 1), sc.SC_ERR_SHAPE),   # short of two rows of logits
])
def test_lmhead_rejects_bad_arguments_on_the_host(L, kw, status):
    assert call_lmhead(L, **kw) == status, err(L)


def test_lmhead_workspace_size(L):
    assert L.sc_lmhead_workspace_bytes(0, 100, 64) == 0
    small = L.sc_lmhead_workspace_bytes(1, 100, 64)
    assert small == 256 + 256  # the fixed part and one row of logits, padded
    # 4096 rows, d = 4096, V = 151936 (148 SMs without a GPU): the block of
    # logits and two FP32 slices of dH (32 x 16 output tiles split in two)
    big = L.sc_lmhead_workspace_bytes(4096, 151936, 4096)
    assert big == 256 + 4096 * 151936 * 2 + 2 * 4096 * 4096 * 4 and big % 256 == 0


@pytest.mark.parametrize("args,status", [
    ((FAKE, -1, 1.0, FAKE * 2), sc.SC_ERR_SHAPE),
    ((FAKE, 4, 1.0, None), sc.SC_ERR_NULL),
    ((None, 4, 1.0, FAKE * 2), sc.SC_ERR_NULL),
    ((FAKE, 4, float("inf"), FAKE * 2), sc.SC_ERR_ARG),
    ((FAKE + 4, 4, 1.0, FAKE * 2), sc.SC_ERR_ALIGN),
    ((FAKE, 4, 1.0, FAKE * 2 + 2), sc.SC_ERR_ALIGN),
])
def test_batch_loss_rejects_bad_arguments_on_the_host(L, args, status):
    assert L.sc_batch_loss(*args, None) == status, err(L)
