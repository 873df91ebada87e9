"""FP64 CPU oracle for score centering -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never does, and this package
imports nothing from it: the two share no code.

The arithmetic lives in ``sc_oracle.c`` (plain C, double precision, one row
at a time).  This module compiles it with gcc on first use (or via
:func:`build`) and exposes it to Python through ctypes with numpy arrays.
The formulas follow the "Score Centering" section of the Agent Lightning
docs page "Score Centering"; the C file states them and every reading taken
where the page is silent.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sc_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libsc_oracle.so")

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

IS_NONE, IS_TIS, IS_MIS, IS_CLIP = 0, 1, 2, 3


class Params(ctypes.Structure):
    _fields_ = [
        ("is_mode", ctypes.c_int),
        ("tis_max", ctypes.c_double),
        ("mis_min", ctypes.c_double),
        ("mis_max", ctypes.c_double),
        ("centering", ctypes.c_int),
        ("inv_temperature", ctypes.c_double),
        ("grad_scale", ctypes.c_double),
        ("clip_low", ctypes.c_double),
        ("clip_high", ctypes.c_double),
    ]


class RowOut(ctypes.Structure):
    _fields_ = [
        ("loss", ctypes.c_double),
        ("logp_a", ctypes.c_double),
        ("P_H", ctypes.c_double),
        ("tail_pi", ctypes.c_double),
        ("Q_H", ctypes.c_double),
        ("tail_mu", ctypes.c_double),
        ("rho", ctypes.c_double),
        ("s", ctypes.c_double),
        ("entropy", ctypes.c_double),
        ("k3", ctypes.c_double),
        ("is_weight", ctypes.c_double),
        ("row_sum", ctypes.c_double),
        ("adv", ctypes.c_double),
        ("n_valid_k", ctypes.c_int),
        ("flags", ctypes.c_uint),
    ]


ROW_OUT_FIELDS = [f for f, _ in RowOut._fields_]
ROW_OUT_DTYPE = np.dtype(
    {
        "names": ROW_OUT_FIELDS,
        "formats": ["<f8"] * 13 + ["<i4", "<u4"],
        "offsets": [getattr(RowOut, f).offset for f in ROW_OUT_FIELDS],
        "itemsize": ctypes.sizeof(RowOut),
    }
)

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``sc_oracle.c`` into a shared library with gcc; return its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    # -ffp-contract=off keeps every multiply and add separately rounded, so the
    # oracle gives the same bits on x86-64 and aarch64.
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    """The loaded oracle.  ``SC_ORACLE_LIB`` names another compiled copy to load
    instead (the mutation tests point it at copies with a planted mistake)."""
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("SC_ORACLE_LIB") or build()
            L = ctypes.CDLL(path)
            L.sco_bf16_to_double.restype = ctypes.c_double
            L.sco_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.sco_double_to_bf16_rne.restype = ctypes.c_uint16
            L.sco_double_to_bf16_rne.argtypes = [ctypes.c_double]
            L.sco_round_bf16_n.restype = None
            L.sco_round_bf16_n.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p]
            L.sco_group_advantages.restype = ctypes.c_int
            L.sco_group_advantages.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_double, ctypes.c_void_p]
            L.sco_rollout_mean_advantages.restype = ctypes.c_int
            L.sco_rollout_mean_advantages.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong,
                                                      ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
            L.sco_topk_capture.restype = ctypes.c_int
            L.sco_topk_capture.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_longlong,
                                           ctypes.c_double, ctypes.c_int, ctypes.c_double, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_void_p]
            L.sco_row.restype = ctypes.c_uint
            L.sco_row.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                  ctypes.c_double, ctypes.POINTER(Params), ctypes.c_void_p,
                                  ctypes.POINTER(RowOut)]
            L.sco_rows.restype = ctypes.c_int
            L.sco_rows.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_longlong,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_int, ctypes.POINTER(Params), ctypes.c_void_p,
                                   ctypes.c_longlong, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_int]
            L.sco_row_out_size.restype = ctypes.c_int
            L.sco_params_size.restype = ctypes.c_int
            assert L.sco_row_out_size() == ctypes.sizeof(RowOut)
            assert L.sco_params_size() == ctypes.sizeof(Params)
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def make_params(is_mode=IS_NONE, tis_max=2.0, mis_min=0.5, mis_max=5.0, centering=True,
                inv_temperature=1.0, grad_scale=1.0, clip_low=0.2, clip_high=0.3) -> Params:
    """Defaults are the settings table of the docs' "Score Centering" section
    and, for the clipped GRPO baseline (is_mode 3), the clip widths of the
    page's `grpo` preset."""
    return Params(int(is_mode), float(tis_max), float(mis_min), float(mis_max), int(bool(centering)),
                  float(inv_temperature), float(grad_scale), float(clip_low), float(clip_high))


def bf16_to_double(bits) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_round(x: float) -> float:
    """Round to the nearest bf16 value (ties to even); returns it as a float."""
    return float(lib().sco_bf16_to_double(lib().sco_double_to_bf16_rne(float(x))))


def bf16_bits(x: float) -> int:
    return int(lib().sco_double_to_bf16_rne(float(x)))


def group_advantages(rewards, n_groups: int, group_size: int, normalize_std: bool = True,
                     eps: float = 1e-6) -> np.ndarray:
    r = np.ascontiguousarray(rewards, dtype=np.float32)
    if r.size != n_groups * group_size:
        raise ValueError("rewards size does not match n_groups * group_size")
    out = np.zeros(n_groups * group_size, dtype=np.float64)
    rc = lib().sco_group_advantages(_ptr(r), n_groups, group_size, int(bool(normalize_std)),
                                    float(eps), _ptr(out))
    if rc != 0:
        raise ValueError("sco_group_advantages rejected its arguments")
    return out


def rollout_mean_advantages(adv, row_response, n_resp: int):
    """Per-rollout mean loss: (adv[r] / valid tokens of response r, counts)."""
    a = np.ascontiguousarray(adv, dtype=np.float64)
    rr = np.ascontiguousarray(row_response, dtype=np.int32)
    counts = np.zeros(n_resp, dtype=np.int64)
    out = np.zeros(n_resp, dtype=np.float64)
    if a.size != n_resp:
        raise ValueError("adv must have n_resp entries")
    rc = lib().sco_rollout_mean_advantages(_ptr(a), _ptr(rr) if rr.size else None, rr.size, n_resp,
                                           _ptr(counts), _ptr(out))
    if rc != 0:
        raise ValueError("sco_rollout_mean_advantages rejected its arguments")
    return out, counts


def topk_capture(logits, K: int, inv_temperature: float = 1.0, top_p: float = 1.0):
    """Sampler-side capture of the top-K behaviour probabilities (FP32 logits
    [T, V]).  Returns (ids int32 [T, K], logprobs float32 [T, K], count int32 [T])."""
    z = np.ascontiguousarray(logits, dtype=np.float32)
    if z.ndim != 2:
        raise ValueError("logits must be [T, V]")
    T, V = z.shape
    ids = np.zeros((T, K), dtype=np.int32)
    lp = np.zeros((T, K), dtype=np.float32)
    cnt = np.zeros(T, dtype=np.int32)
    rc = lib().sco_topk_capture(_ptr(z), T, V, V, float(inv_temperature), int(K), float(top_p), _ptr(ids),
                                _ptr(lp), _ptr(cnt))
    if rc != 0:
        raise ValueError("sco_topk_capture rejected its arguments")
    return ids, lp, cnt


def row(z_bits, ids, logprobs, a: int, A: float, params: Params | None = None,
        rollout_logprob: float | None = None):
    """One unmasked row.  Returns (grad[V] float64, RowOut as a dict)."""
    z = np.ascontiguousarray(z_bits, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    lp = np.ascontiguousarray(logprobs, dtype=np.float32)
    if ids.shape != lp.shape:
        raise ValueError("ids and logprobs differ in length")
    p = params if params is not None else make_params()
    g = np.zeros(z.size, dtype=np.float64)
    out = RowOut()
    f = lib().sco_row(_ptr(z), z.size, _ptr(ids) if ids.size else None, _ptr(lp) if lp.size else None,
                      ids.size, int(a), float(rollout_logprob or 0.0), int(rollout_logprob is not None),
                      float(A), ctypes.byref(p), _ptr(g), ctypes.byref(out))
    if f == 0xFFFFFFFF:
        raise ValueError("sco_row rejected its arguments")
    return g, {k: getattr(out, k) for k in ROW_OUT_FIELDS}


def rows(batch: dict, params: Params, row_idx=None, nthreads: int = 0):
    """Rows of a batch laid out like the library call (numpy arrays).

    ``batch`` keys: logits (uint16 [T, row_stride]), V, rec_ids (int32 [T, K_max]),
    rec_logprobs (float32 [T, K_max]), rec_count (int32 [T] or None),
    sampled (int32 [T]), rollout_logprob (float32 [T] or None),
    row_response (int32 [T]), adv (float32 [n_resp]).
    Returns (grad float64 [n, V], logp_a float64 [n], out structured [n], threads).
    """
    z = np.ascontiguousarray(batch["logits"], dtype=np.uint16)
    T = z.shape[0]
    stride = z.shape[1]
    V = int(batch.get("V", stride))
    ids = np.ascontiguousarray(batch["rec_ids"], dtype=np.int32)
    lp = np.ascontiguousarray(batch["rec_logprobs"], dtype=np.float32)
    K_max = ids.shape[1] if ids.ndim == 2 else 0
    cnt = batch.get("rec_count")
    cnt = None if cnt is None else np.ascontiguousarray(cnt, dtype=np.int32)
    sampled = np.ascontiguousarray(batch["sampled"], dtype=np.int32)
    rl = batch.get("rollout_logprob")
    rl = None if rl is None else np.ascontiguousarray(rl, dtype=np.float32)
    resp = np.ascontiguousarray(batch["row_response"], dtype=np.int32)
    adv = np.ascontiguousarray(batch["adv"], dtype=np.float32)
    if row_idx is None:
        row_idx = np.arange(T, dtype=np.int64)
    row_idx = np.ascontiguousarray(row_idx, dtype=np.int64)
    n = row_idx.size
    g = np.zeros((n, V), dtype=np.float64)
    la = np.zeros(n, dtype=np.float64)
    out = np.zeros(n, dtype=ROW_OUT_DTYPE)
    used = lib().sco_rows(_ptr(z), T, V, stride, _ptr(ids) if K_max else None,
                          _ptr(lp) if K_max else None, _ptr(cnt), K_max, _ptr(sampled), _ptr(rl),
                          _ptr(resp), _ptr(adv), adv.size, ctypes.byref(params), _ptr(row_idx), n,
                          _ptr(g), _ptr(la), out.ctypes.data, int(nthreads))
    if used < 0:
        raise ValueError("sco_rows rejected its arguments")
    return g, la, out, used


def bf16_round_array(x) -> np.ndarray:
    """Every entry of x rounded to bf16 (ties to even); uint16 bit patterns, same shape."""
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(a.shape, dtype=np.uint16)
    lib().sco_round_bf16_n(_ptr(a), a.size, _ptr(out))
    return out


def lmhead_rows(hidden_bits, w_bits, batch: dict, params: Params, nthreads: int = 0, dw_rows=None):
    """The LM head followed by score centering, for a BF16 trainer.

    The trainer's logits are z = bf16(H W^T): H [T, d] and W [V, d] are bf16
    values, their products summed in FP64 and rounded once to bf16 (ties to
    even).  Every row then gets the score-centered gradient g of the row
    oracle (``rows``), and the gradients of the batch loss
    grad_scale * sum_t loss_t with respect to the LM head's inputs follow from
    z's linearity: dH = g W and dW = g^T H, in FP64 from the unrounded g.

    hidden_bits: uint16 [T, d]; w_bits: uint16 [V, d]; batch: the keys of
    ``rows`` except logits (V taken from w_bits).  dw_rows: indices of the
    rows of dW to return (all when None; a full FP64 dW at V = 151936 and
    d = 4096 takes 5 GB).
    Returns (dH [T, d], dW [len(dw_rows) or V, d], logp_a [T], out [T],
    z_bits [T, V]).
    """
    Hb = np.ascontiguousarray(hidden_bits, dtype=np.uint16)
    Wb = np.ascontiguousarray(w_bits, dtype=np.uint16)
    if Hb.ndim != 2 or Wb.ndim != 2 or Hb.shape[1] != Wb.shape[1]:
        raise ValueError("hidden must be [T, d] and w [V, d] with the same d")
    H = bf16_to_double(Hb)
    W = bf16_to_double(Wb)
    z_bits = bf16_round_array(H @ W.T)
    b = dict(batch)
    b["logits"] = z_bits
    b["V"] = Wb.shape[0]
    g, la, out, _ = rows(b, params, None, nthreads)
    gw = g if dw_rows is None else g[:, np.asarray(dw_rows, dtype=np.int64)]
    return g @ W, gw.T @ H, la, out, z_bits
