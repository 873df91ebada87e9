#!/usr/bin/env python3
"""Benchmark of the score-centering hot path on GB300.

One step = one pass of the whole hot path over one batch: the group
advantages (sc_group_advantages) and the fused score-centered forward and
backward (sc_center_forward_backward) over the quick-check batch -- 2 prompts
x 4 responses x 512 tokens = 4096 rows (lengths U[64, 512], the rest padding),
V = 151936, K = 128 recorded ids, synthetic inputs from ``synth``.

Prints one JSON line.  `value` is valid (unmasked) tokens per second over all
ranks with inputs resident in HBM; `e2e` is the same metric through the same
calls with pinned host buffers copied in and the step's results (per-row
losses and log p_a) copied back inside the timed region; `roofline` relates
the fused kernel's algorithmic bytes to the measured HBM copy bandwidth;
`cpu_baseline` times the FP64 CPU oracle on this machine's cores on a bounded
sample of the same batch; `secondary` times the sampler-side top-K capture
(sc_topk_capture) on the batch's FP32 sampler logits.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
For N > 1 launch under torch.distributed.run: every rank processes its own
batch (weak scaling); the only exchange is the global valid-token count,
all-reduced once per batch to set grad_scale = 1 / N_tokens.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "score-centered tokens/s at V=151936 bf16; HBM GB/s as % of GB300 peak"
WORKLOAD = "C2"
WORKLOAD_TEXT = ("quick-check batch: 2 prompts x 4 responses x 512 tokens = 4096 rows, lengths U[64,512] "
                 "padded, V=151936, K=128, logits N(0,3^2)+Zipf bias, sampler noise N(0,0.05^2)")
WORKLOADS = {
    "C3": ("full-step batch: 32 prompts x 4 responses, lengths U[256,4096] padded to 4096 = 524288 rows in "
           "32 chunks of 16384, V=151936, K=128, Bernoulli(0.6) rewards with 10% forced to 0"),
    "C4": ("large-vocab peaked case: 16384 rows (8 x 4 responses x 512 tokens), V=248320, K=128, "
           "logits Student-t(3) x 6, sampler noise N(0,0.2^2)"),
    "C5": ("ragged sampler case: 65536 rows (8 x 8 responses x 1024 tokens), V=151936, recorded count "
           "U{1..128} from T=0.7 top-p 0.95 sampling, 5% of sampled tokens outside the recorded ids"),
}
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["precision_off_policy_gb300/csrc/sc_center.cu", "precision_off_policy_gb300/csrc/sc_device.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "center_kernel_C2_traffic.txt")


def strip_c_comments(text: str) -> str:
    """C/C++ source without its comments (newlines inside block comments kept);
    string and character literals are copied as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            j = n if j < 0 else j + 2
            out.append("\n" * text.count("\n", i, j))
            i = j
        else:
            out.append(c)
            i += 1
    return "".join(out)


def kernel_source_hash() -> str:
    """Hash of the fused kernel's code: its sources without comments, blank
    lines and trailing blanks, so that editing a comment does not change the
    kernel the committed counters were taken on."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            lines = (ln.rstrip() for ln in strip_c_comments(f.read()).split("\n"))
        h.update("\n".join(ln for ln in lines if ln).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_traffic(launch_rows: int):
    """DRAM bytes per launch from the committed ncu summary (`key: value`
    lines), if it was taken on the current kernel source; else None."""
    t = {}
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if line.startswith("#") or ":" not in line:
                    continue
                k, v = line.split(":", 1)
                t[k.strip()] = v.strip()
    except OSError:
        return None
    if t.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return float(t["dram_bytes_per_launch"]) * launch_rows / float(t["rows_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def algorithmic_bytes(batch) -> int:
    """Minimum bytes one launch must move: per valid row the logits read and
    gradient write (4 V), the recorded head (8 per id used: its count clamped
    to [0, K], 4 more for the count itself), its metadata (row_response,
    sampled id, rollout logprob, advantage: 16) and outputs (log p_a 4,
    diagnostics 64); per padding row the zero gradient (2 V), row_response and
    sampled id (8) and outputs (68)."""
    V = batch["V"]
    resp = batch["row_response"].cpu().numpy()
    valid = int((resp >= 0).sum())
    masked = resp.size - valid
    cnt = batch["rec_count"]
    if cnt is not None:
        c = np.asarray(cnt.cpu().numpy() if hasattr(cnt, "cpu") else cnt)
        k_total = int(np.clip(c[resp >= 0], 0, batch["K"]).sum())
    else:
        k_total = valid * batch["K"]
    extra_cnt = 4 * valid if cnt is not None else 0
    return valid * (4 * V + 16 + 68) + 8 * k_total + extra_cnt + masked * (2 * V + 8 + 68)


def topk_secondary(batch, dev, peak, peak_kind, reps=10):
    """The sampler-side top-K capture on the batch's sampler logits (FP32
    trainer logits plus the sampler's N(0, 0.05^2) perturbation), K = 128,
    with and without the nucleus: CUDA-event time per launch and the fraction
    of the HBM copy bandwidth for reading each logit once."""
    import precision_off_policy_gb300 as sc

    cfg = synth.config(WORKLOAD)
    g = torch.Generator(device=dev).manual_seed(cfg["seed"] + 77)
    z = batch["logits"].float()
    z.add_(torch.randn(z.shape, generator=g, device=dev), alpha=cfg["sigma_s"])
    T, V = z.shape
    K = batch["K"]
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    lps = torch.empty((T, K), dtype=torch.float32, device=dev)
    cnt = torch.empty(T, dtype=torch.int32, device=dev)
    st = torch.cuda.Stream(device=dev)
    out = []
    alg = T * (4 * V + 8 * K + 4)
    for inv_t, top_p in [(1.0, 1.0), (1.0 / 0.7, 0.95)]:
        with torch.cuda.stream(st):
            for _ in range(3):
                sc.sc_topk_capture(z, K, inv_t, top_p, ids_out=ids, logprobs_out=lps, count_out=cnt, stream=st)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(reps):
                sc.sc_topk_capture(z, K, inv_t, top_p, ids_out=ids, logprobs_out=lps, count_out=cnt, stream=st)
            e1.record(st)
        st.synchronize()
        ms = e0.elapsed_time(e1) / reps
        achieved = alg / (ms / 1e3) / 1e9
        out.append({"kernel": "topk_kernel", "call": "sc_topk_capture",
                    "workload": f"{WORKLOAD} sampler logits FP32 [{T}, {V}], K={K}, inv_t={inv_t:.4g}, top_p={top_p}",
                    "rows_per_s": T / (ms / 1e3), "ms_per_launch": ms,
                    "mean_count": float(cnt.float().mean().item()),
                    "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                                 "frac": achieved / peak, "peak_source": peak_kind,
                                 "algorithmic_bytes_per_launch": alg}})
    del z
    return out


NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s GB300 figure the target is stated against


def bare_row_sum_fraction(grad, diag, p):
    """Fraction of the rows with a nonzero advantage whose bf16 gradient row
    sums to within the bare 1e-3 |a| (a = grad_scale A_w / T), with no
    allowance for the bf16 rounding of its entries (computed on the device)."""
    import precision_off_policy_gb300 as sc

    d = sc.diag_to_numpy(diag)
    a = np.abs(d["adv"] * d["is_weight"]) * float(np.float32(p.inv_temperature)) * abs(float(np.float32(p.grad_scale)))
    gs = np.abs(grad.double().sum(dim=1).cpu().numpy())
    live = a > 0
    return float(np.mean(gs[live] <= 1e-3 * a[live])) if live.any() else 1.0


def config_secondary(name, dev, peak, peak_kind, reps=10, warmup=3):
    """One whole step of the hot path over configuration `name` -- for each of
    its chunks the group advantages and the fused call -- with every chunk's
    inputs resident in HBM (inputs far larger than L2).  Times the step
    (CUDA events around `reps` steps) and the fused kernel alone (events
    around reps x chunks back-to-back fused launches, no other kernel between
    them), and relates the fused launches' algorithmic bytes to the measured
    and to the nominal HBM bandwidth."""
    import precision_off_policy_gb300 as sc

    cfg = synth.config(name)
    n_ch = synth.n_chunks(cfg)
    t0 = time.perf_counter()
    chunks = [synth.make_batch(cfg, chunk=c, device=dev) for c in range(n_ch)]
    gen_s = time.perf_counter() - t0
    b0 = chunks[0]
    T, V, K = b0["logits"].shape[0], b0["V"], b0["K"]
    n_valid = sum(b["n_valid"] for b in chunks)
    total_rows = sum(b["logits"].shape[0] for b in chunks)
    p = sc.params(K_max=K, inv_temperature=b0["inv_temperature"], grad_scale=1.0 / max(1, n_valid))
    plan = sc.sc_plan_query(V, p)
    grad = torch.empty((T, V), dtype=torch.bfloat16, device=dev)
    logp = torch.empty(T, dtype=torch.float32, device=dev)
    diag = torch.empty((T, 16), dtype=torch.int32, device=dev)
    advs = [torch.empty_like(b["rewards"]) for b in chunks]
    st = torch.cuda.Stream(device=dev)

    def fused(b, adv):
        sc.sc_center_forward_backward(b["logits"], b["rec_ids"], b["rec_logprobs"], b["rec_count"], b["sampled"],
                                      b["rollout_logprob"], b["row_response"], adv, p, grad_out=grad,
                                      logp_out=logp, diag_out=diag, stream=st)

    def step():
        for b, adv in zip(chunks, advs):
            sc.sc_group_advantages(b["rewards"], b["n_groups"], b["group_size"], out=adv, stream=st)
            fused(b, adv)

    with torch.cuda.stream(st):
        for _ in range(warmup):
            step()
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(st)
        for _ in range(reps):
            step()
        e1.record(st)
        for _ in range(reps):
            for b, adv in zip(chunks, advs):
                fused(b, adv)
        e2.record(st)
    st.synchronize()
    step_ms = e0.elapsed_time(e1) / reps
    kernel_ms = e1.elapsed_time(e2) / reps  # all chunks' fused launches of one step
    alg = sum(algorithmic_bytes(b) for b in chunks)
    achieved = alg / (kernel_ms / 1e3) / 1e9
    bare = bare_row_sum_fraction(grad, diag, p)  # the last chunk's rows
    del chunks, grad, advs
    torch.cuda.empty_cache()
    return {"workload": f"{name} {WORKLOADS[name]}", "call": "sc_group_advantages + sc_center_forward_backward",
            "rows": total_rows, "valid_rows": n_valid, "chunks": n_ch, "V": V, "K": K, "plan": plan,
            "ms_per_step": step_ms, "tokens_per_s": n_valid / (step_ms / 1e3),
            "kernel_ms_per_step": kernel_ms, "kernel_tokens_per_s": n_valid / (kernel_ms / 1e3),
            "row_sum_bare_fraction_last_chunk": bare, "input_generation_s": gen_s,
            "roofline": {"bound": "hbm", "kernel": "center_kernel", "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_kind,
                         "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                         "algorithmic_bytes_per_step": alg}}


def bf16_peak():
    """Measured dense bf16 TFLOP/s (the sustained figure: the call below runs
    for tens of milliseconds back to back)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured (sustained)"
    except (OSError, KeyError, ValueError):
        return 1700.0, "fallback (sustained)"


def lmhead_secondary(batch, adv, dev, d=4096, reps=5):
    """The LM head followed by score centering on the batch's 4096 rows:
    random bf16 hidden states [T, d] and head [V, d] (logits of standard
    deviation near 3), the batch's recorded ids, sampled tokens and responses.
    Three products of 2 T d V flops each per call (logits, dH, dW), all on the
    library's tensor-core GEMM.  Timed as one block of all T rows and as
    blocks of 1024 (dW then added to by the later blocks); each product also
    timed alone at the one-block shapes."""
    import precision_off_policy_gb300 as sc

    T, V, K = batch["logits"].shape[0], batch["V"], batch["K"]
    g = torch.Generator(device=dev).manual_seed(4242)
    hidden = torch.randn((T, d), generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn((V, d), generator=g, device=dev) * (3.0 / d ** 0.5)).to(torch.bfloat16)
    dh = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((V, d), dtype=torch.float32, device=dev)
    logp = torch.empty(T, dtype=torch.float32, device=dev)
    p = sc.params(K_max=K, grad_scale=1.0 / max(1, batch["n_valid"]))
    st = torch.cuda.Stream(device=dev)
    peak, kind = bf16_peak()
    flops = 3 * 2.0 * T * d * V

    def timed(fn, n):
        with torch.cuda.stream(st):
            for _ in range(2):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(n):
                fn()
            e1.record(st)
        st.synchronize()
        return e0.elapsed_time(e1) / n

    out = []
    for block_rows in (T, 1024):
        def call():
            sc.sc_lmhead_forward_backward(hidden, w, batch["rec_ids"], batch["rec_logprobs"], batch["rec_count"],
                                          batch["sampled"], batch["rollout_logprob"], batch["row_response"], adv, p,
                                          block_rows=block_rows, dhidden=dh, dw=dw, logp_out=logp, stream=st)
        ms = timed(call, reps)
        achieved = flops / (ms / 1e3) / 1e12
        out.append({"kernel": "gemm_kernel (tcgen05) x 3 + center_kernel", "call": "sc_lmhead_forward_backward",
                    "workload": f"{WORKLOAD} rows: T={T}, d={d}, V={V}, K={K}, blocks of {block_rows} rows",
                    "ms_per_call": ms, "tokens_per_s": batch["n_valid"] / (ms / 1e3),
                    "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                                 "frac": achieved / peak, "peak_source": kind, "flops_per_call": flops}})
    # each product alone (one block of T rows): z = H W^T, dH = g W, dW = g^T H
    z = torch.empty((T, V), dtype=torch.bfloat16, device=dev)
    gemms = {"z = H W^T (A, B K-major; bf16 out)": lambda: sc.sc_gemm_bf16(hidden, w, z, True, True, sc.GEMM_BF16,
                                                                           stream=st),
             "dH = g W (B N-major; bf16 out)": lambda: sc.sc_gemm_bf16(z, w, dh, True, False, sc.GEMM_BF16, stream=st),
             "dW = g^T H (A M-major, B N-major; FP32 out)": lambda: sc.sc_gemm_bf16(z, hidden, dw, False, False,
                                                                                    sc.GEMM_FP32, stream=st)}
    for name, fn in gemms.items():
        ms = timed(fn, reps)
        achieved = 2.0 * T * d * V / (ms / 1e3) / 1e12
        out.append({"kernel": "gemm_kernel (tcgen05)", "call": "sc_gemm_bf16", "workload": f"{name}: T={T}, d={d}, V={V}",
                    "ms_per_call": ms, "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                                                    "unit": "TFLOP/s", "frac": achieved / peak, "peak_source": kind,
                                                    "flops_per_call": 2.0 * T * d * V}})
    del hidden, w, dh, dw, z
    return out


def cpu_baseline(batch, p, adv, min_seconds=10.0, max_passes=50):
    """The FP64 oracle over the whole batch on all host cores, repeated until
    about `min_seconds` of wall time have been spent (a stable figure)."""
    import oracle

    bn = synth.to_numpy(batch)
    bn["adv"] = adv
    T = bn["logits"].shape[0]
    rows = np.arange(T)
    prm = oracle.make_params(inv_temperature=float(np.float32(p.inv_temperature)),
                             grad_scale=float(np.float32(p.grad_scale)))
    valid = int((bn["row_response"] >= 0).sum())
    used, passes = 0, 0
    t0 = time.perf_counter()
    while passes < max_passes and (passes == 0 or time.perf_counter() - t0 < min_seconds):
        for r0 in range(0, T, 512):  # bounded memory: 512 rows of FP64 gradients at a time
            _, _, _, u = oracle.rows(bn, prm, rows[r0:r0 + 512])
            used = max(used, u)
        passes += 1
    dt = time.perf_counter() - t0
    return {"value": valid * passes / dt, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"{passes} passes over the {T} rows of the {WORKLOAD} batch ({valid} valid), "
                      f"{dt:.1f} s wall"}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus and not (world == 1 and n_gpus == 1):
        if world == 1:
            raise SystemExit(f"--gpus {n_gpus} needs torch.distributed.run with {n_gpus} processes")
    return world, rank, local


def run_reference(args):
    world, rank, _ = dist_setup(args.gpus)
    if rank != 0:
        return 0
    import oracle

    cfg = synth.config(WORKLOAD)
    rows_per_step = 128
    batch = make_host_rows(cfg, rows_per_step * 2)
    adv = oracle.group_advantages(batch["rewards"].numpy(), batch["n_groups"], batch["group_size"], True,
                                  1e-6).astype(np.float32)
    bn = synth.to_numpy(batch)
    bn["adv"] = adv
    prm = oracle.make_params(grad_scale=1.0)
    times, valids, used = [], [], 0
    T = bn["logits"].shape[0]
    for s in range(args.warmup + args.steps):
        r0 = (s * rows_per_step) % T
        rows = np.arange(r0, min(T, r0 + rows_per_step))
        t0 = time.perf_counter()
        _, _, _, u = oracle.rows(bn, prm, rows)
        dt = time.perf_counter() - t0
        used = max(used, u)
        if s >= args.warmup:
            times.append(dt)
            valids.append(int((bn["row_response"][rows] >= 0).sum()))
    value = sum(valids) / sum(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{WORKLOAD} {WORKLOAD_TEXT}", "rows_per_step": rows_per_step,
                   "V": cfg["V"], "K": cfg["K"]},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                         "sample": f"{rows_per_step} rows of the {WORKLOAD} batch per step (host-generated)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def make_host_rows(cfg, n):
    """The first `n` rows of the workload generated on the host (same recipe)."""
    n_resp = max(cfg["n_per_prompt"], (n + cfg["L_pad"] - 1) // cfg["L_pad"])
    n_prompts = max(1, (n_resp + cfg["n_per_prompt"] - 1) // cfg["n_per_prompt"])
    sub = synth.config(cfg, n_prompts=min(n_prompts, cfg["n_prompts"]))
    return synth.make_batch(sub, device="cpu")


def profile_run(args):
    """Small launches for a profiler (no timing, no JSON line):
    `topk`: three launches of the top-K capture on the quick-check batch's
    sampler logits at --top-p / --inv-t; `gemm`: the logits product at 1024
    rows (H [1024, 4096] W^T, V = 151936, bf16 out) and the head-gradient
    product on a quarter vocabulary (g^T [37984, 1024] H [1024, 4096], FP32
    out), one launch each."""
    import precision_off_policy_gb300 as sc

    sc.build()
    dev = torch.device("cuda", 0)
    if args.profile == "topk":
        cfg = synth.config(WORKLOAD)
        b = synth.make_batch(cfg, device=dev)
        g = torch.Generator(device=dev).manual_seed(cfg["seed"] + 77)
        z = b["logits"].float()
        z.add_(torch.randn(z.shape, generator=g, device=dev), alpha=cfg["sigma_s"])
        del b
        for _ in range(3):
            sc.sc_topk_capture(z, cfg["K"], args.inv_t, args.top_p)
    else:
        g = torch.Generator(device=dev).manual_seed(1)
        T, d = 1024, 4096
        H = torch.randn((T, d), generator=g, device=dev).to(torch.bfloat16)
        W = (torch.randn((151936, d), generator=g, device=dev) * 0.05).to(torch.bfloat16)
        z = torch.empty((T, 151936), dtype=torch.bfloat16, device=dev)
        G = (torch.randn((T, 37984), generator=g, device=dev) * 0.01).to(torch.bfloat16)
        dw = torch.empty((37984, d), dtype=torch.float32, device=dev)
        sc.sc_gemm_bf16(H, W, z, True, True, sc.GEMM_BF16)
        sc.sc_gemm_bf16(G, H, dw, False, False, sc.GEMM_FP32)
    torch.cuda.synchronize()
    print("profile run done")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration lines")
    ap.add_argument("--profile", choices=["topk", "gemm"], default=None,
                    help="only run a few launches of one kernel for a profiler")
    ap.add_argument("--top-p", type=float, default=1.0)
    ap.add_argument("--inv-t", type=float, default=1.0)
    args = ap.parse_args()
    if args.profile:
        return profile_run(args)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    import precision_off_policy_gb300 as sc
    from precision_off_policy_gb300 import dp

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    sc.build()

    cfg = synth.config(WORKLOAD, seed=synth.CONFIGS[WORKLOAD]["seed"] + 1000 * rank)
    batch = synth.make_batch(cfg, device=dev)
    T, V, K = batch["logits"].shape[0], batch["V"], batch["K"]
    n_valid = batch["n_valid"]
    # global generated-token count for the token-mean loss (int64 all-reduce)
    grad_scale = dp.token_mean_scale(dp.global_valid_tokens(n_valid, device=dev))
    p = sc.params(K_max=K, inv_temperature=batch["inv_temperature"], grad_scale=grad_scale)
    plan = sc.sc_plan_query(V, p)

    stream = torch.cuda.Stream(device=dev)
    grad = torch.empty((T, V), dtype=torch.bfloat16, device=dev)
    logp = torch.empty(T, dtype=torch.float32, device=dev)
    diag = torch.empty((T, 16), dtype=torch.int32, device=dev)
    adv = torch.empty_like(batch["rewards"])

    def step(s):
        sc.sc_group_advantages(batch["rewards"], batch["n_groups"], batch["group_size"], out=adv, stream=s)
        sc.sc_center_forward_backward(batch["logits"], batch["rec_ids"], batch["rec_logprobs"], batch["rec_count"],
                                      batch["sampled"], batch["rollout_logprob"], batch["row_response"], adv, p,
                                      grad_out=grad, logp_out=logp, diag_out=diag, stream=s)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(stream)
    stream.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---- device-resident timing ----------------------------------------------
    # The fused kernel is launched with programmatic stream serialisation: its
    # shared-memory set-up overlaps the previous kernel's tail.  An event
    # recorded between two kernels ends that overlap, so the fused launch is
    # bracketed by events on every EVENT_EVERY-th step only; its duration is
    # the mean over those launches (which lose their own overlap: a slightly
    # long, conservative figure), and `value` is the whole timed region.
    EVENT_EVERY = 8
    timed = [i for i in range(args.steps) if i % EVENT_EVERY == 0]
    ev = {i: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for i in timed}
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clocks:
        barrier()
        start.record(stream)
        for i in range(args.steps):
            sc.sc_group_advantages(batch["rewards"], batch["n_groups"], batch["group_size"], out=adv, stream=stream)
            if i in ev:
                ev[i][0].record(stream)
            sc.sc_center_forward_backward(batch["logits"], batch["rec_ids"], batch["rec_logprobs"],
                                          batch["rec_count"], batch["sampled"], batch["rollout_logprob"],
                                          batch["row_response"], adv, p, grad_out=grad, logp_out=logp,
                                          diag_out=diag, stream=stream)
            if i in ev:
                ev[i][1].record(stream)
        stop.record(stream)
        # The fused kernel alone: back-to-back launches with events only around
        # the whole run (each launch's set-up overlaps the previous one's tail,
        # as in the timed steps), so its mean cannot exceed a step.
        b2b = min(args.steps, 400)
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record(stream)
        for i in range(b2b):
            sc.sc_center_forward_backward(batch["logits"], batch["rec_ids"], batch["rec_logprobs"],
                                          batch["rec_count"], batch["sampled"], batch["rollout_logprob"],
                                          batch["row_response"], adv, p, grad_out=grad, logp_out=logp,
                                          diag_out=diag, stream=stream)
        k1.record(stream)
        barrier()
    elapsed_ms = start.elapsed_time(stop)
    kernel_ms = [a.elapsed_time(b) for a, b in ev.values()]
    b2b_ms = k0.elapsed_time(k1) / b2b
    bare = bare_row_sum_fraction(grad, diag, p)
    t_max = torch.tensor([elapsed_ms], dtype=torch.float64, device=dev)
    tok = torch.tensor([n_valid * args.steps], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t_max, op=dist.ReduceOp.MAX)
        dist.all_reduce(tok)
    elapsed_ms = float(t_max.item())
    value = float(tok.item()) / (elapsed_ms / 1e3)

    # ---- end to end: pinned host buffers in, the step's result back ----------
    # Every step copies its inputs in from pinned host memory and reads its
    # result back: the per-row losses and log p_a (the diagnostics records and
    # logp_out).  The gradient stays on the device, where the backward pass of
    # the LM head consumes it.  Three device buffer sets and three streams:
    # step i+1's inputs copy in (copy-in stream) while step i computes (compute
    # stream) and step i-1's results copy out (copy-out stream).  Host outputs
    # alternate between two pinned buffers.
    host_in = {k: batch[k].cpu().pin_memory() for k in
               ["logits", "rec_ids", "rec_logprobs", "sampled", "rollout_logprob", "row_response", "rewards"]}
    host_out = [dict(logp=torch.empty(T, dtype=torch.float32).pin_memory(),
                     diag=torch.empty((T, 16), dtype=torch.int32).pin_memory()) for _ in range(2)]
    del grad
    torch.cuda.empty_cache()
    sets = []
    for _ in range(3):
        sets.append(dict(inp={k: torch.empty_like(v, device=dev) for k, v in host_in.items()},
                         grad=torch.empty((T, V), dtype=torch.bfloat16, device=dev),
                         logp=torch.empty(T, dtype=torch.float32, device=dev),
                         diag=torch.empty((T, 16), dtype=torch.int32, device=dev),
                         adv=torch.empty_like(batch["rewards"]),
                         loaded=torch.cuda.Event(), computed=torch.cuda.Event(), done=torch.cuda.Event()))
    copy_in = torch.cuda.Stream(device=dev)
    copy_out = torch.cuda.Stream(device=dev)
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out[0].values())

    def e2e_run(n):
        for i in range(n):
            bs = sets[i % 3]
            copy_in.wait_event(bs["done"])  # the set's previous step has been copied out
            with torch.cuda.stream(copy_in):
                for k, v in host_in.items():
                    bs["inp"][k].copy_(v, non_blocking=True)
                bs["loaded"].record(copy_in)
            stream.wait_event(bs["loaded"])
            with torch.cuda.stream(stream):
                x = bs["inp"]
                sc.sc_group_advantages(x["rewards"], batch["n_groups"], batch["group_size"], out=bs["adv"],
                                       stream=stream)
                sc.sc_center_forward_backward(x["logits"], x["rec_ids"], x["rec_logprobs"], None, x["sampled"],
                                              x["rollout_logprob"], x["row_response"], bs["adv"], p,
                                              grad_out=bs["grad"], logp_out=bs["logp"], diag_out=bs["diag"],
                                              stream=stream)
                bs["computed"].record(stream)
            copy_out.wait_event(bs["computed"])
            with torch.cuda.stream(copy_out):
                ho = host_out[i % 2]
                ho["logp"].copy_(bs["logp"], non_blocking=True)
                ho["diag"].copy_(bs["diag"], non_blocking=True)
                bs["done"].record(copy_out)

    e2e_run(3)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_in.wait_event(e0)
    copy_out.wait_event(e0)
    e2e_run(args.e2e_steps)
    stream.wait_stream(copy_out)  # the last step's outputs are on the host
    e1.record(stream)
    barrier()
    e2e_ms = torch.tensor([e0.elapsed_time(e1)], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(e2e_ms, op=dist.ReduceOp.MAX)
    e2e_value = n_valid * world * args.e2e_steps / (float(e2e_ms.item()) / 1e3)

    # ---- roofline of the fused kernel ----------------------------------------
    alg = algorithmic_bytes(batch)
    k_avg_ms = b2b_ms
    achieved = alg / (k_avg_ms / 1e3) / 1e9
    peak, peak_kind = hbm_peak()
    traffic = measured_traffic(T)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD} {WORKLOAD_TEXT}", "rows": T, "valid_rows": n_valid, "V": V, "K": K,
                   "io": "bf16 logits in, bf16 gradient out, FP32 arithmetic",
                   "parallelism": f"dp{world} (rows sharded, no data-path collective)",
                   "l2": "inputs larger than L2 (1.24 GB of logits per step)",
                   "plan": plan},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_kind,
                     "kernel": "center_kernel", "algorithmic_bytes_per_launch": alg,
                     "kernel_ms": k_avg_ms, "timed_launches": b2b,
                     "timing": "CUDA events around back-to-back fused launches on the launching stream",
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "kernel_ms_bracketed_in_steps": statistics.fmean(kernel_ms)},
        "row_sum_bare_fraction": bare,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": args.e2e_steps},
        "gpu_launches": 2 * args.steps + b2b,
        "clocks": clocks.summary(),
    }
    del sets
    torch.cuda.empty_cache()
    line["secondary"] = topk_secondary(batch, dev, peak, peak_kind)
    line["secondary"].extend(lmhead_secondary(batch, adv, dev))
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        adv_or = oracle.group_advantages(batch["rewards"].cpu().numpy(), batch["n_groups"], batch["group_size"],
                                         True, 1e-6).astype(np.float32)
        line["cpu_baseline"] = cpu_baseline(batch, p, adv_or)
    if not args.no_configs:
        # the other workloads, one after another (each holds its own inputs)
        del batch
        torch.cuda.empty_cache()
        line["configs"] = [config_secondary(name, dev, peak, peak_kind) for name in ("C4", "C5", "C3")]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
