"""GB300 (sm_103a) score centering: Python binding of the C ABI in ``include/sc.h``.

This module only marshals arguments.  Every step of the computation runs in
the CUDA library ``_build/libsc_gb300.so`` (built by :func:`build`); there is
no fallback, and calls raise if the library is missing or the device cannot
run it.  PyTorch provides device memory and streams.

Entry points (same names as the C ABI):

* :func:`sc_group_advantages` -- GRPO group-std advantages (docs "Score
  Centering" page, section "Training").
* :func:`sc_center_forward_backward` -- the fused score-centered forward and
  backward over ``[T, V]`` bf16 logits (section "Score Centering").
"""

from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import build as _build_mod

__all__ = [
    "build", "lib", "ScError", "Params", "params", "DIAG_DTYPE", "DIAG_FIELDS",
    "sc_group_advantages", "sc_center_forward_backward", "sc_plan_query", "diag_to_numpy",
    "ScoreCenteredLoss", "score_centered_loss",
    "sc_rollout_mean_advantages", "sc_topk_capture", "SC_IS_NONE", "SC_IS_TIS", "SC_IS_MIS", "SC_IS_CLIP",
    "WORKSPACE_BYTES", "workspace", "reset_workspaces", "sc_lmhead_forward_backward", "sc_batch_loss",
    "sc_gemm_bf16", "GEMM_BF16", "GEMM_FP32", "GEMM_FP32_ADD",
]

SC_OK, SC_ERR_NULL, SC_ERR_ALIGN, SC_ERR_SHAPE, SC_ERR_ARG, SC_ERR_CUDA, SC_ERR_UNSUPPORTED = range(7)
SC_IS_NONE, SC_IS_TIS, SC_IS_MIS, SC_IS_CLIP = 0, 1, 2, 3
SC_FLAGS_ENTRY, SC_FLAGS_VECTOR = 1, 2  # recorded-id flag layouts (0 = automatic)
SC_STATUS_DATA, SC_STATUS_TIMEOUT_LOAD, SC_STATUS_TIMEOUT_EXCHANGE = 0x1, 0x2, 0x4

FLAG_MASKED = 0x1
FLAG_BAD_ID = 0x2
FLAG_DUP_ID = 0x4
FLAG_BAD_SAMPLED = 0x8
FLAG_BAD_COUNT = 0x10
FLAG_BAD_RESPONSE = 0x20
FLAG_CLAMP_PI = 0x40
FLAG_CLAMP_MU = 0x80
FLAG_IS_TRUNC = 0x100
FLAG_IS_REJECT = 0x200
FLAG_CLIPPED = 0x400

# Symbols declared in include/sc.h.
EXPORTS = ["sc_params_default", "sc_group_advantages", "sc_batch_loss", "sc_gemm_bf16", "sc_rollout_mean_advantages", "sc_topk_capture",
           "sc_center_forward_backward", "sc_center_forward_backward_noalloc", "sc_lmhead_workspace_bytes",
           "sc_lmhead_forward_backward", "sc_plan_query",
           "sc_status_string", "sc_last_error", "sc_abi_version"]


class ScError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"status {status}: {message}")
        self.status = status


class Params(ctypes.Structure):
    _fields_ = [
        ("K_max", ctypes.c_int),
        ("is_mode", ctypes.c_int),
        ("tis_max", ctypes.c_float),
        ("mis_min", ctypes.c_float),
        ("mis_max", ctypes.c_float),
        ("centering", ctypes.c_int),
        ("inv_temperature", ctypes.c_float),
        ("grad_scale", ctypes.c_float),
        ("cluster_size", ctypes.c_int),
        ("threads", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("clip_low", ctypes.c_float),
        ("clip_high", ctypes.c_float),
        ("flag_layout", ctypes.c_int),
        ("wait_limit_us", ctypes.c_int),
        ("test_stall", ctypes.c_int),
    ]


DIAG_FIELDS = ["loss", "logp_a", "P_H", "tail_pi", "Q_H", "tail_mu", "rho", "s", "entropy", "k3",
               "is_weight", "row_sum", "adv", "n_valid_k", "flags", "reserved"]
DIAG_DTYPE = np.dtype({"names": DIAG_FIELDS,
                       "formats": ["<f4"] * 13 + ["<i4", "<u4", "<u4"]})
assert DIAG_DTYPE.itemsize == 64

_lock = threading.Lock()
_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library for sm_103a (in-tree) and return its path."""
    return _build_mod.build(force=force, verbose=verbose)


def lib():
    """The loaded CUDA library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build_mod.LIB_PATH
            if not os.path.exists(path):
                raise ScError(SC_ERR_UNSUPPORTED,
                              f"CUDA library {path} is missing: run precision_off_policy_gb300.build()")
            L = ctypes.CDLL(path)
            vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float
            L.sc_params_default.argtypes = [ctypes.POINTER(Params)]
            L.sc_params_default.restype = i32
            L.sc_group_advantages.argtypes = [vp, i32, i32, i32, f32, vp, vp]
            L.sc_group_advantages.restype = i32
            L.sc_batch_loss.argtypes = [vp, i64, f32, vp, vp]
            L.sc_batch_loss.restype = i32
            L.sc_gemm_bf16.argtypes = [vp, i64, i32, vp, i64, i32, vp, i64, i32, i64, i64, i64, vp, vp]
            L.sc_gemm_bf16.restype = i32
            L.sc_rollout_mean_advantages.argtypes = [vp, vp, i64, i32, vp, vp, vp]
            L.sc_rollout_mean_advantages.restype = i32
            L.sc_topk_capture.argtypes = [vp, i64, i32, i64, f32, i32, f32, vp, vp, vp, vp, vp]
            L.sc_topk_capture.restype = i32
            L.sc_center_forward_backward.argtypes = [vp, i64, i32, i64, vp, vp, vp, vp, vp, vp, vp, i32,
                                                     ctypes.POINTER(Params), vp, i64, vp, vp, vp, vp, vp]
            L.sc_center_forward_backward.restype = i32
            L.sc_center_forward_backward_noalloc.argtypes = [vp, i64, i32, i64, vp, vp, vp, vp, vp, vp, vp, i32,
                                                             ctypes.POINTER(Params), vp, i64, vp, vp, vp, vp]
            L.sc_center_forward_backward_noalloc.restype = i32
            L.sc_lmhead_workspace_bytes.argtypes = [i64, i32, i32]
            L.sc_lmhead_workspace_bytes.restype = ctypes.c_size_t
            L.sc_lmhead_forward_backward.argtypes = [vp, vp, i64, i32, i32, vp, vp, vp, vp, vp, vp, vp, i32,
                                                     ctypes.POINTER(Params), i64, vp, vp, vp, vp, vp, vp,
                                                     ctypes.c_size_t, vp]
            L.sc_lmhead_forward_backward.restype = i32
            L.sc_plan_query.argtypes = [i32, ctypes.POINTER(Params)] + [ctypes.POINTER(i32)] * 6
            L.sc_plan_query.restype = i32
            L.sc_status_string.argtypes = [i32]
            L.sc_status_string.restype = ctypes.c_char_p
            L.sc_last_error.argtypes = []
            L.sc_last_error.restype = ctypes.c_char_p
            L.sc_abi_version.argtypes = []
            L.sc_abi_version.restype = i32
            _lib = L
    return _lib


def _check(status: int):
    if status != SC_OK:
        L = lib()
        raise ScError(status, f"{L.sc_status_string(status).decode()}: {L.sc_last_error().decode()}")


def params(K_max=128, is_mode=SC_IS_NONE, tis_max=2.0, mis_min=0.5, mis_max=5.0, centering=True,
           inv_temperature=1.0, grad_scale=1.0, cluster_size=0, threads=0, stages=0, clip_low=0.2,
           clip_high=0.3, flag_layout=0, wait_limit_us=0, test_stall=0) -> Params:
    """Defaults are the settings table of the docs' "Score Centering" section
    and the clip widths of the page's `grpo` preset.  wait_limit_us: how long
    a wait inside the fused kernel may take before the launch gives up (0 =
    1 s); test_stall: the test hook of the C header (0 in normal use)."""
    return Params(int(K_max), int(is_mode), float(tis_max), float(mis_min), float(mis_max),
                  int(bool(centering)), float(inv_temperature), float(grad_scale), int(cluster_size),
                  int(threads), int(stages), float(clip_low), float(clip_high), int(flag_layout),
                  int(wait_limit_us), int(test_stall))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, dev, ndim=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != dev:
        raise ValueError(f"{name} is on {t.device}, expected {dev}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


def _check_rows(T, **named):
    """Each given per-row tensor is 1-D with T entries."""
    for name, t in named.items():
        if t is not None and (t.dim() != 1 or t.shape[0] != T):
            raise ValueError(f"{name} must have T = {T} entries, got shape {tuple(t.shape)}")


def _check_row_inputs(T, K_max, rec_ids, rec_logprobs, rec_count, sampled_id, rollout_logprob, row_response,
                      logp_out, diag_out, status):
    """The per-row inputs and outputs shared by the fused call and the LM head
    hold what the kernels read or write (the C ABI takes plain pointers, so a
    short buffer is refused here, before any launch)."""
    if K_max > 0:
        for name, t in (("rec_ids", rec_ids), ("rec_logprobs", rec_logprobs)):
            if t is None or tuple(t.shape) != (T, K_max):
                raise ValueError(f"{name} must be [T, K_max] = [{T}, {K_max}]")
    _check_rows(T, rec_count=rec_count, sampled_id=sampled_id, rollout_logprob=rollout_logprob,
                row_response=row_response, logp_out=logp_out)
    if diag_out is not None and (tuple(diag_out.shape) != (T, 16) or not diag_out.is_contiguous()):
        raise ValueError("diag_out must be a contiguous int32 [T, 16] tensor")
    if status is not None and status.numel() < 1:
        raise ValueError("status must hold one int32")


def _check_center_buffers(T, V, K_max, logits, grad_out, rec_ids, rec_logprobs, rec_count, sampled_id,
                          rollout_logprob, row_response, logp_out, diag_out, status):
    """Shapes of the fused call's buffers: logits and grad_out rows hold at
    least V entries, grad_out has T rows, the per-row tensors T entries."""
    if logits.shape[1] < V:
        raise ValueError(f"logits rows hold {logits.shape[1]} entries, fewer than V = {V}")
    if grad_out.shape[0] != T or grad_out.shape[1] < V:
        raise ValueError(f"grad_out must be [T = {T}, >= V = {V}], got {tuple(grad_out.shape)}")
    _check_row_inputs(T, K_max, rec_ids, rec_logprobs, rec_count, sampled_id, rollout_logprob, row_response,
                      logp_out, diag_out, status)


def _check_topk_buffers(T, V, K, logits, ids_out, logprobs_out, count_out):
    """Shapes of the top-K capture's buffers."""
    if logits.shape[1] < V:
        raise ValueError(f"logits rows hold {logits.shape[1]} entries, fewer than V = {V}")
    for name, t in (("ids_out", ids_out), ("logprobs_out", logprobs_out)):
        if tuple(t.shape) != (T, K):
            raise ValueError(f"{name} must be [T, K] = [{T}, {K}], got {tuple(t.shape)}")
    _check_rows(T, count_out=count_out)


def _check_lmhead_buffers(T, d, V, K_max, dhidden, dw, rec_ids, rec_logprobs, rec_count, sampled_id,
                          rollout_logprob, row_response, logp_out, diag_out, status):
    """Shapes of the LM head call's buffers: dhidden [T, d] and dw [V, d],
    contiguous, and the per-row tensors as for the fused call."""
    if tuple(dhidden.shape) != (T, d) or not dhidden.is_contiguous():
        raise ValueError(f"dhidden must be a contiguous [T, d] = [{T}, {d}] tensor")
    if tuple(dw.shape) != (V, d) or not dw.is_contiguous():
        raise ValueError(f"dw must be a contiguous [V, d] = [{V}, {d}] tensor")
    _check_row_inputs(T, K_max, rec_ids, rec_logprobs, rec_count, sampled_id, rollout_logprob, row_response,
                      logp_out, diag_out, status)


def _rows(t, name):
    """Row stride of a 2-D tensor whose rows are contiguous."""
    if t.stride(1) != 1:
        raise ValueError(f"{name} rows must be contiguous")
    return t.stride(0) if t.shape[0] > 1 else max(t.stride(0), t.shape[1])


def sc_group_advantages(rewards: torch.Tensor, n_groups: int, group_size: int,
                        normalize_std: bool = True, eps: float = 1e-6,
                        out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """FP32 rewards [n_groups * group_size] (device) -> FP32 advantages."""
    dev = rewards.device
    if dev.type != "cuda":
        raise ValueError("rewards must be on a CUDA device")
    _need(rewards, "rewards", torch.float32, dev)
    if not rewards.is_contiguous() or rewards.numel() != n_groups * group_size:
        raise ValueError("rewards must be contiguous with n_groups * group_size entries")
    if out is None:
        out = torch.empty_like(rewards)
    _need(out, "out", torch.float32, dev)
    if out.numel() != rewards.numel() or not out.is_contiguous():
        raise ValueError("out must be contiguous with as many entries as rewards")
    _check(lib().sc_group_advantages(_ptr(rewards), int(n_groups), int(group_size),
                                     int(bool(normalize_std)), float(eps), _ptr(out), _stream(stream)))
    return out


def sc_rollout_mean_advantages(adv: torch.Tensor, row_response: torch.Tensor, out: torch.Tensor | None = None,
                               counts: torch.Tensor | None = None, stream=None):
    """Per-rollout mean: adv[r] / (valid tokens of response r), 0 if none.

    adv float32 [n_resp], row_response int32 [T] on the same CUDA device.
    Returns (adv_out, counts int32 [n_resp]); ``out`` may be ``adv``.
    """
    dev = adv.device
    if dev.type != "cuda":
        raise ValueError("adv must be on a CUDA device")
    _need(adv, "adv", torch.float32, dev, 1)
    _need(row_response, "row_response", torch.int32, dev, 1)
    n = adv.numel()
    out = torch.empty_like(adv) if out is None else out
    counts = torch.empty(n, dtype=torch.int32, device=dev) if counts is None else counts
    _need(out, "out", torch.float32, dev, 1)
    _need(counts, "counts", torch.int32, dev, 1)
    for name, t in [("adv", adv), ("row_response", row_response), ("out", out), ("counts", counts)]:
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if out.numel() != n or counts.numel() != n:
        raise ValueError("out and counts must have n_resp entries")
    _check(lib().sc_rollout_mean_advantages(_ptr(adv), _ptr(row_response), int(row_response.numel()), int(n),
                                            _ptr(counts), _ptr(out), _stream(stream)))
    return out, counts


def sc_topk_capture(logits: torch.Tensor, K: int, inv_temperature: float = 1.0, top_p: float = 1.0,
                    ids_out: torch.Tensor | None = None, logprobs_out: torch.Tensor | None = None,
                    count_out: torch.Tensor | None = None, V: int | None = None, stream=None,
                    workspace_buf: torch.Tensor | None = None, dynamic: bool = True):
    """Sampler-side top-K capture.  logits: FP32 [T, >=V] on a CUDA device with
    contiguous rows.  Returns (ids int32 [T, K], logprobs float32 [T, K],
    count int32 [T]).  With ``dynamic`` the last rows are handed out at run
    time through the binding's workspace for this device and stream (or
    ``workspace_buf``); without, every row is dealt at launch."""
    dev = logits.device
    if dev.type != "cuda":
        raise ValueError("logits must be on a CUDA device")
    _need(logits, "logits", torch.float32, dev, 2)
    T = logits.shape[0]
    V = logits.shape[1] if V is None else int(V)
    K = int(K)
    ids_out = torch.empty((T, K), dtype=torch.int32, device=dev) if ids_out is None else ids_out
    logprobs_out = torch.empty((T, K), dtype=torch.float32, device=dev) if logprobs_out is None else logprobs_out
    count_out = torch.empty(T, dtype=torch.int32, device=dev) if count_out is None else count_out
    _need(ids_out, "ids_out", torch.int32, dev, 2)
    _need(logprobs_out, "logprobs_out", torch.float32, dev, 2)
    _need(count_out, "count_out", torch.int32, dev, 1)
    for name, t in [("ids_out", ids_out), ("logprobs_out", logprobs_out), ("count_out", count_out)]:
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    _check_topk_buffers(T, V, K, logits, ids_out, logprobs_out, count_out)
    if T == 0:
        return ids_out, logprobs_out, count_out
    ws = None
    if dynamic:
        ws = workspace(dev, stream) if workspace_buf is None else workspace_buf
        if ws.device != dev or ws.numel() * ws.element_size() < WORKSPACE_BYTES:
            raise ValueError(f"workspace_buf must hold {WORKSPACE_BYTES} bytes on {dev}")
    _check(lib().sc_topk_capture(_ptr(logits), T, V, _rows(logits, "logits"), float(inv_temperature), K,
                                 float(top_p), _ptr(ids_out), _ptr(logprobs_out), _ptr(count_out), _ptr(ws),
                                 _stream(stream)))
    return ids_out, logprobs_out, count_out


WORKSPACE_BYTES = 64  # SC_WORKSPACE_BYTES
_workspaces = {}


def workspace(device, stream=None) -> torch.Tensor:
    """The binding's workspace for calls on (device, stream): 64 zeroed bytes,
    created on first use.  Calls on one stream run one after another, so they
    share it; another stream gets its own."""
    dev = torch.device(device)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    key = (dev.index, int(stream.cuda_stream))
    with _lock:
        ws = _workspaces.get(key)
        if ws is None:
            # allocated and zeroed on the stream the calls run on, so that the
            # zero fill is ordered before the first launch that uses it
            with torch.cuda.stream(stream):
                ws = torch.zeros(WORKSPACE_BYTES // 8, dtype=torch.int64, device=dev)
            _workspaces[key] = ws
    return ws


def reset_workspaces() -> None:
    """Zero every workspace the binding holds (needed only after a launch that
    did not complete, e.g. a CUDA error)."""
    with _lock:
        for (dev_index, stream_ptr), ws in _workspaces.items():
            with torch.cuda.stream(torch.cuda.ExternalStream(stream_ptr, device=torch.device("cuda", dev_index))):
                ws.zero_()


def sc_center_forward_backward(logits: torch.Tensor, rec_ids: torch.Tensor | None,
                               rec_logprobs: torch.Tensor | None, rec_count: torch.Tensor | None,
                               sampled_id: torch.Tensor, rollout_logprob: torch.Tensor | None,
                               row_response: torch.Tensor, adv: torch.Tensor, p: Params,
                               V: int | None = None, grad_out: torch.Tensor | None = None,
                               logp_out: torch.Tensor | None = None,
                               diag_out: torch.Tensor | None = None,
                               status: torch.Tensor | None = None, stream=None,
                               workspace_buf: torch.Tensor | None = None):
    """Score-centered forward/backward.

    logits: bf16 [T, >=V] on a CUDA device with contiguous rows; rec_ids int32
    and rec_logprobs float32 [T, K_max]; rec_count int32 [T] or None;
    sampled_id, row_response int32 [T]; rollout_logprob float32 [T] or None;
    adv float32 [n_resp].  grad_out may be ``logits`` (in place).  diag_out,
    when given, is an int32 [T, 16] tensor (64-byte records, see
    :func:`diag_to_numpy`); status an int32 [1] tensor.  workspace_buf: 64
    zeroed bytes on the device (SC_WORKSPACE_BYTES in the C header); by
    default the binding's own for this device and stream (:func:`workspace`).
    Returns (grad_out, logp_out, diag_out).
    """
    dev = logits.device
    if dev.type != "cuda":
        raise ValueError("logits must be on a CUDA device")
    _need(logits, "logits", torch.bfloat16, dev, 2)
    T = logits.shape[0]
    V = logits.shape[1] if V is None else int(V)
    K_max = int(p.K_max)
    for name, t, dt, nd in [("rec_ids", rec_ids, torch.int32, 2), ("rec_logprobs", rec_logprobs, torch.float32, 2),
                            ("rec_count", rec_count, torch.int32, 1), ("sampled_id", sampled_id, torch.int32, 1),
                            ("rollout_logprob", rollout_logprob, torch.float32, 1),
                            ("row_response", row_response, torch.int32, 1), ("adv", adv, torch.float32, 1)]:
        _need(t, name, dt, dev, nd)
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if grad_out is None:
        grad_out = torch.empty((T, V), dtype=torch.bfloat16, device=dev)
    _need(grad_out, "grad_out", torch.bfloat16, dev, 2)
    if logp_out is None:
        logp_out = torch.empty(T, dtype=torch.float32, device=dev)
    _need(logp_out, "logp_out", torch.float32, dev, 1)
    _need(diag_out, "diag_out", torch.int32, dev, 2)
    _need(status, "status", torch.int32, dev, 1)
    _check_center_buffers(T, V, K_max, logits, grad_out, rec_ids, rec_logprobs, rec_count, sampled_id,
                          rollout_logprob, row_response, logp_out, diag_out, status)
    if T == 0:
        return grad_out, logp_out, diag_out
    if workspace_buf is None:
        workspace_buf = workspace(dev, stream)
    elif workspace_buf.device != dev or workspace_buf.numel() * workspace_buf.element_size() < WORKSPACE_BYTES:
        raise ValueError(f"workspace_buf must hold {WORKSPACE_BYTES} bytes on {dev}")
    _check(lib().sc_center_forward_backward(
        _ptr(logits), T, V, _rows(logits, "logits"), _ptr(rec_ids) if K_max else None,
        _ptr(rec_logprobs) if K_max else None, _ptr(rec_count), _ptr(sampled_id), _ptr(rollout_logprob),
        _ptr(row_response), _ptr(adv), int(adv.numel()), ctypes.byref(p), _ptr(grad_out),
        _rows(grad_out, "grad_out"), _ptr(logp_out), _ptr(diag_out), _ptr(status), _ptr(workspace_buf),
        _stream(stream)))
    return grad_out, logp_out, diag_out


def sc_batch_loss(diag: torch.Tensor, grad_scale: float, out: torch.Tensor | None = None, stream=None):
    """grad_scale * sum of the rows' losses of a fused call's diagnostics
    (int32 [T, 16] on a CUDA device), summed by the library in a fixed order.
    Returns a float32 [1] device tensor (``out`` when given)."""
    dev = diag.device
    if dev.type != "cuda":
        raise ValueError("diag must be on a CUDA device")
    _need(diag, "diag", torch.int32, dev, 2)
    if diag.shape[1] != 16 or not diag.is_contiguous():
        raise ValueError("diag must be a contiguous int32 [T, 16] tensor")
    out = torch.empty(1, dtype=torch.float32, device=dev) if out is None else out
    _need(out, "out", torch.float32, dev)
    if out.numel() < 1:
        raise ValueError("out must hold one float32")
    _check(lib().sc_batch_loss(_ptr(diag), int(diag.shape[0]), float(grad_scale), _ptr(out), _stream(stream)))
    return out


GEMM_BF16, GEMM_FP32, GEMM_FP32_ADD = 0, 1, 2


def sc_gemm_bf16(a: torch.Tensor, b: torch.Tensor, c: torch.Tensor, a_kmajor: bool = True, b_kmajor: bool = True,
                 c_mode: int = GEMM_BF16, status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """C = A . B on the tensor cores (the LM head's products).

    a: bf16, [M, K] when ``a_kmajor`` else [K, M]; b: bf16, [N, K] when
    ``b_kmajor`` else [K, N]; rows contiguous.  c: row-major [M, N], bf16
    (GEMM_BF16) or float32 (GEMM_FP32: written; GEMM_FP32_ADD: C += A . B).
    """
    dev = a.device
    if dev.type != "cuda":
        raise ValueError("a must be on a CUDA device")
    _need(a, "a", torch.bfloat16, dev, 2)
    _need(b, "b", torch.bfloat16, dev, 2)
    _need(c, "c", torch.bfloat16 if c_mode == GEMM_BF16 else torch.float32, dev, 2)
    _need(status, "status", torch.int32, dev, 1)
    M, K = (a.shape[0], a.shape[1]) if a_kmajor else (a.shape[1], a.shape[0])
    N, Kb = (b.shape[0], b.shape[1]) if b_kmajor else (b.shape[1], b.shape[0])
    if Kb != K:
        raise ValueError(f"inner sizes differ: {K} and {Kb}")
    if tuple(c.shape[:1]) != (M,) or c.shape[1] < N:
        raise ValueError(f"c must be [M = {M}, >= N = {N}]")
    _check(lib().sc_gemm_bf16(_ptr(a), _rows(a, "a"), 0 if a_kmajor else 1, _ptr(b), _rows(b, "b"),
                              0 if b_kmajor else 1, _ptr(c), _rows(c, "c"), int(c_mode), M, N, K, _ptr(status),
                              _stream(stream)))
    return c


def sc_plan_query(V: int, p: Params) -> dict:
    """The launch plan the library uses for V on the current device."""
    out = [ctypes.c_int(0) for _ in range(6)]
    _check(lib().sc_plan_query(int(V), ctypes.byref(p), *[ctypes.byref(o) for o in out]))
    return dict(zip(["cluster_size", "threads", "slice", "smem_bytes", "max_clusters", "flag_layout"],
                    [o.value for o in out]))


def diag_to_numpy(diag: torch.Tensor) -> np.ndarray:
    """int32 [T, 16] diagnostics tensor -> numpy structured array [T]."""
    return diag.detach().cpu().contiguous().numpy().view(DIAG_DTYPE).reshape(-1)


class ScoreCenteredLoss(torch.autograd.Function):
    """Autograd wrapper of :func:`sc_center_forward_backward`.

    The forward pass is one library launch: it produces the per-row losses and
    the finished gradient with respect to the logits, which is saved.  The
    returned loss is ``grad_scale * sum_t loss_t`` (a token mean when
    grad_scale = 1 / N_tokens), summed by the library (:func:`sc_batch_loss`),
    whose gradient is exactly the saved one; the backward pass returns it
    scaled by the incoming gradient (torch's one multiplication, when the
    incoming gradient is not 1).  Outputs: (loss, logp [T], diag int32
    [T, 16]); the last two carry no gradient.
    """

    @staticmethod
    def forward(ctx, logits, rec_ids, rec_logprobs, rec_count, sampled_id, rollout_logprob, row_response, adv,
                p, stream=None):
        T = logits.shape[0]
        diag = torch.empty((T, 16), dtype=torch.int32, device=logits.device)
        grad, logp, diag = sc_center_forward_backward(
            logits.detach(), rec_ids, rec_logprobs, rec_count, sampled_id, rollout_logprob, row_response, adv, p,
            diag_out=diag, stream=stream)
        ctx.save_for_backward(grad)
        loss = sc_batch_loss(diag, float(np.float32(p.grad_scale)), stream=stream).reshape(())
        ctx.mark_non_differentiable(logp, diag)
        return loss, logp, diag

    @staticmethod
    def backward(ctx, g_loss, g_logp, g_diag):
        (grad,) = ctx.saved_tensors
        return (grad * g_loss.to(grad.dtype),) + (None,) * 9


def score_centered_loss(logits, rec_ids, rec_logprobs, rec_count, sampled_id, rollout_logprob, row_response, adv,
                        p, stream=None):
    """Differentiable score-centered loss (see :class:`ScoreCenteredLoss`)."""
    return ScoreCenteredLoss.apply(logits, rec_ids, rec_logprobs, rec_count, sampled_id, rollout_logprob,
                                   row_response, adv, p, stream)


_lmhead_workspaces = {}


def sc_lmhead_forward_backward(hidden: torch.Tensor, w: torch.Tensor, rec_ids, rec_logprobs, rec_count,
                               sampled_id, rollout_logprob, row_response, adv, p: Params, block_rows: int = 1024,
                               dhidden: torch.Tensor | None = None, dw: torch.Tensor | None = None,
                               logp_out: torch.Tensor | None = None, diag_out: torch.Tensor | None = None,
                               status: torch.Tensor | None = None, stream=None,
                               workspace_buf: torch.Tensor | None = None):
    """The LM head followed by score centering: z = H W^T in row blocks, the
    fused kernel on each block, dH = g W and dW = g^T H.

    hidden bf16 [T, d], w bf16 [V, d] (contiguous, d % 8 == 0); the other
    inputs as :func:`sc_center_forward_backward`.  Returns (dhidden bf16
    [T, d], dw float32 [V, d], logp_out, diag_out).  workspace_buf: a uint8
    tensor of sc_lmhead_workspace_bytes(block_rows, V, d) zero-initialised
    bytes; by default the binding's own for this device, stream and size.
    """
    dev = hidden.device
    if dev.type != "cuda":
        raise ValueError("hidden must be on a CUDA device")
    _need(hidden, "hidden", torch.bfloat16, dev, 2)
    _need(w, "w", torch.bfloat16, dev, 2)
    if not hidden.is_contiguous() or not w.is_contiguous():
        raise ValueError("hidden and w must be contiguous")
    T, d = hidden.shape
    V = w.shape[0]
    if w.shape[1] != d:
        raise ValueError("w must be [V, d] with the hidden size d")
    K_max = int(p.K_max)
    for name, t, dt, nd in [("rec_ids", rec_ids, torch.int32, 2), ("rec_logprobs", rec_logprobs, torch.float32, 2),
                            ("rec_count", rec_count, torch.int32, 1), ("sampled_id", sampled_id, torch.int32, 1),
                            ("rollout_logprob", rollout_logprob, torch.float32, 1),
                            ("row_response", row_response, torch.int32, 1), ("adv", adv, torch.float32, 1)]:
        _need(t, name, dt, dev, nd)
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    dhidden = torch.empty((T, d), dtype=torch.bfloat16, device=dev) if dhidden is None else dhidden
    dw = torch.empty((V, d), dtype=torch.float32, device=dev) if dw is None else dw
    logp_out = torch.empty(T, dtype=torch.float32, device=dev) if logp_out is None else logp_out
    _need(dhidden, "dhidden", torch.bfloat16, dev, 2)
    _need(dw, "dw", torch.float32, dev, 2)
    _need(logp_out, "logp_out", torch.float32, dev, 1)
    _need(diag_out, "diag_out", torch.int32, dev, 2)
    _need(status, "status", torch.int32, dev, 1)
    _check_lmhead_buffers(T, d, V, K_max, dhidden, dw, rec_ids, rec_logprobs, rec_count, sampled_id,
                          rollout_logprob, row_response, logp_out, diag_out, status)
    if T == 0:
        return dhidden, dw, logp_out, diag_out
    L = lib()
    need = int(L.sc_lmhead_workspace_bytes(min(int(block_rows), T), V, d))
    if workspace_buf is None:
        s_obj = torch.cuda.current_stream(dev) if stream is None else stream
        key = (dev.index, int(s_obj.cuda_stream), need)
        with _lock:
            workspace_buf = _lmhead_workspaces.get(key)
            if workspace_buf is None:
                with torch.cuda.stream(s_obj):  # zero fill ordered before the first call on s_obj
                    workspace_buf = torch.zeros(need, dtype=torch.uint8, device=dev)
                _lmhead_workspaces[key] = workspace_buf
    if workspace_buf.device != dev or workspace_buf.numel() * workspace_buf.element_size() < need:
        raise ValueError(f"workspace_buf must hold {need} bytes on {dev}")
    _check(L.sc_lmhead_forward_backward(
        _ptr(hidden), _ptr(w), T, d, V, _ptr(rec_ids) if K_max else None, _ptr(rec_logprobs) if K_max else None,
        _ptr(rec_count), _ptr(sampled_id), _ptr(rollout_logprob), _ptr(row_response), _ptr(adv), int(adv.numel()),
        ctypes.byref(p), int(block_rows), _ptr(dhidden), _ptr(dw), _ptr(logp_out), _ptr(diag_out), _ptr(status),
        _ptr(workspace_buf), int(workspace_buf.numel() * workspace_buf.element_size()), _stream(stream)))
    return dhidden, dw, logp_out, diag_out
