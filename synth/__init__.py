"""Seeded synthetic inputs for score centering.

This module is shared by the tests, the benchmark and the smoke check.  It
holds none of the score-centering arithmetic: it only simulates what a
trainer and a low-precision sampler would hand to the loss -- bf16 trainer
logits, the sampler's recorded top-K ids with their log-probabilities, the
sampled token and its rollout log-probability, the row -> response map with
padding, and rewards.

The pages train Qwen3.5-9B on INTELLECT-2 math prompts; neither the model nor
the dataset is available, so these recipes stand in for them with the shapes
of the five workload configurations:

* C1  tiny oracle case: 2 prompts x 4 responses x 8 tokens, V = 1024, K = 128,
  logits N(0, 2^2), sampler noise N(0, 0.05^2), rewards Bernoulli(0.5).
* C2  quick-check batch: 2 x 4 responses x 512 tokens (lengths U[64, 512],
  padded), V = 151936, logits N(0, 3^2) plus a Zipf-shaped bias
  -1.1 ln(rank) over a seeded permutation of the vocabulary, noise
  N(0, 0.05^2), rewards Bernoulli(0.3).
* C3  full-step batch: 32 x 4 responses, lengths U[256, 4096] padded to 4096,
  streamed in 16384-row chunks (4 responses per chunk), V = 151936, C2's
  logit recipe, rewards Bernoulli(0.6) with 10% of responses forced to 0.
* C4  large-vocab peaked case: 8 x 4 responses x 512 tokens, V = 248320,
  logits Student-t(3) x 6, noise N(0, 0.2^2), rewards Bernoulli(0.5).
* C5  ragged sampler case: 8 x 8 responses x 1024 tokens, V = 151936, C2's
  logit recipe; the sampler draws at temperature 0.7 with top-p 0.95; the
  recorded count per row is U{1..128} (capped by the nucleus size); 5% of
  sampled tokens are drawn outside the recorded ids; rewards {0, 1} with one
  all-ones and one all-zeros group.
* C2R the quick-check batch where the trainer's policy sits on the sampler's
  recorded ids: after the sampler's top-K is recorded, the trainer logits of
  the recorded ids are raised by U[10, 30] per row (then rounded to bf16),
  so the trainer's unrecorded mass falls to about e^-10 .. e^-30 while the
  sampler's stays where it was.

The sampler distribution mu is softmax((trainer logits + noise) / T_s) in
FP32; the recorded ids are mu's top-K with FP32 log mu (their sum stays
below one); the sampled token is drawn from mu by the Gumbel-max rule.
"""

from __future__ import annotations

import copy
import math

import torch

BASE = dict(
    n_prompts=2, n_per_prompt=4, L_pad=8, len_lo=None, len_hi=None, V=1024, K=128,
    logits="normal", sigma=2.0, zipf=0.0, sigma_s=0.05, temperature=1.0, top_p=1.0,
    k_uniform=False, p_outside=0.0, p_reward=0.5, force_zero_frac=0.0, force_equal_groups=0,
    chunk_rows=None, head_boost=None, seed=1,
)

CONFIGS = {
    "C1": dict(BASE, seed=1),
    "C2": dict(BASE, L_pad=512, len_lo=64, len_hi=512, V=151936, sigma=3.0, zipf=1.1, p_reward=0.3,
               seed=2),
    "C3": dict(BASE, n_prompts=32, L_pad=4096, len_lo=256, len_hi=4096, V=151936, sigma=3.0, zipf=1.1,
               p_reward=0.6, force_zero_frac=0.1, chunk_rows=16384, seed=3),
    "C4": dict(BASE, n_prompts=8, L_pad=512, V=248320, logits="student3", sigma=6.0, sigma_s=0.2,
               p_reward=0.5, seed=4),
    "C5": dict(BASE, n_prompts=8, n_per_prompt=8, L_pad=1024, V=151936, sigma=3.0, zipf=1.1,
               temperature=0.7, top_p=0.95, k_uniform=True, p_outside=0.05, force_equal_groups=2,
               seed=5),
    # The quick-check batch with a trainer that has moved almost all of its
    # mass onto the sampler's recorded ids: 1 - P_H far below 1e-6 on most
    # rows while the sampler's own tail 1 - Q_H stays large.
    "C2R": dict(BASE, L_pad=512, len_lo=64, len_hi=512, V=151936, sigma=3.0, zipf=1.1, p_reward=0.3,
                head_boost=(10.0, 30.0), seed=12),
}


def config(name_or_cfg, **overrides) -> dict:
    """A configuration by name (C1..C5) or dict, with fields overridden."""
    cfg = copy.deepcopy(CONFIGS[name_or_cfg] if isinstance(name_or_cfg, str) else name_or_cfg)
    for k, v in overrides.items():
        if k not in cfg:
            raise KeyError(k)
        cfg[k] = v
    return cfg


def n_rows(cfg) -> int:
    return cfg["n_prompts"] * cfg["n_per_prompt"] * cfg["L_pad"]


def n_chunks(cfg) -> int:
    rows = cfg["chunk_rows"] or n_rows(cfg)
    return (n_rows(cfg) + rows - 1) // rows


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def responses(cfg):
    """Per-response lengths and rewards (host tensors, from the config seed)."""
    g = _gen(cfg["seed"] * 1000 + 7, "cpu")
    n_resp = cfg["n_prompts"] * cfg["n_per_prompt"]
    L = cfg["L_pad"]
    if cfg["len_lo"] is None:
        lengths = torch.full((n_resp,), L, dtype=torch.int64)
    else:
        lengths = torch.randint(cfg["len_lo"], cfg["len_hi"] + 1, (n_resp,), generator=g)
    rewards = (torch.rand(n_resp, generator=g) < cfg["p_reward"]).float()
    if cfg["force_zero_frac"] > 0:
        forced = torch.rand(n_resp, generator=g) < cfg["force_zero_frac"]
        rewards[forced] = 0.0  # truncated responses score 0
    n = cfg["n_per_prompt"]
    for grp in range(min(cfg["force_equal_groups"], cfg["n_prompts"])):
        rewards[grp * n:(grp + 1) * n] = 1.0 if grp % 2 == 0 else 0.0
    return lengths, rewards


def _vocab_bias(cfg, device):
    if cfg["zipf"] == 0.0:
        return None
    g = _gen(cfg["seed"] * 1000 + 11, "cpu")
    rank = torch.randperm(cfg["V"], generator=g).to(torch.float32) + 1.0
    return (-cfg["zipf"] * torch.log(rank)).to(device)


def _logits_f32(cfg, rows, g, device, bias):
    V = cfg["V"]
    if cfg["logits"] == "normal":
        z = torch.randn(rows, V, generator=g, device=device) * cfg["sigma"]
    elif cfg["logits"] == "student3":
        nrm = torch.randn(rows, V, generator=g, device=device)
        chi = torch.zeros(rows, V, device=device)
        for _ in range(3):
            chi += torch.randn(rows, V, generator=g, device=device) ** 2
        z = nrm / torch.sqrt(chi / 3.0) * cfg["sigma"]
    else:
        raise ValueError(cfg["logits"])
    if bias is not None:
        z += bias
    return z


def _gumbel_argmax(logw, g):
    u = torch.rand(logw.shape, generator=g, device=logw.device).clamp_(1e-20, 1.0 - 1e-7)
    return torch.argmax(logw - torch.log(-torch.log(u)), dim=1)


def make_batch(cfg, chunk: int = 0, device="cpu", row_block: int = 1024) -> dict:
    """Rows of chunk `chunk` of the configuration, generated on `device`.

    Returns a dict of tensors on `device`: logits (bf16 [T, V]), rec_ids
    (int32 [T, K]), rec_logprobs (f32 [T, K]), rec_count (int32 [T] or None),
    sampled (int32 [T]), rollout_logprob (f32 [T]), row_response (int32 [T],
    -1 for padding, indices local to the chunk), rewards (f32 [n_resp] of
    the chunk's responses), plus n_groups, group_size, inv_temperature,
    V, K and the number of valid rows.
    """
    cfg = config(cfg) if isinstance(cfg, str) else cfg
    device = torch.device(device)
    V, K, L = cfg["V"], cfg["K"], cfg["L_pad"]
    lengths, rewards = responses(cfg)
    total = n_rows(cfg)
    per_chunk = cfg["chunk_rows"] or total
    r0 = chunk * per_chunk
    r1 = min(total, r0 + per_chunk)
    if r0 >= total:
        raise IndexError("chunk out of range")
    T = r1 - r0
    resp_first = r0 // L
    resp_last = (r1 - 1) // L
    rows = torch.arange(r0, r1)
    resp_global = rows // L
    valid = (rows % L) < lengths[resp_global]
    row_response = torch.where(valid, resp_global - resp_first, torch.full_like(resp_global, -1))
    chunk_rewards = rewards[resp_first:resp_last + 1].clone()
    n = cfg["n_per_prompt"]
    if resp_first % n != 0 or (resp_last + 1) % n != 0:
        raise ValueError("chunks must hold whole groups")

    bias = _vocab_bias(cfg, device)
    inv_ts = 1.0 / cfg["temperature"]
    logits = torch.empty(T, V, dtype=torch.bfloat16, device=device)
    rec_ids = torch.empty(T, K, dtype=torch.int32, device=device)
    rec_lp = torch.empty(T, K, dtype=torch.float32, device=device)
    rec_count = torch.full((T,), K, dtype=torch.int32, device=device) if cfg["k_uniform"] else None
    sampled = torch.empty(T, dtype=torch.int32, device=device)
    rollout = torch.empty(T, dtype=torch.float32, device=device)
    g = _gen(cfg["seed"] * 1_000_003 + chunk, device)
    for b0 in range(0, T, row_block):
        b1 = min(T, b0 + row_block)
        nb = b1 - b0
        z = _logits_f32(cfg, nb, g, device, bias).to(torch.bfloat16)
        logits[b0:b1] = z
        zs = z.float() + torch.randn(nb, V, generator=g, device=device) * cfg["sigma_s"]
        logq = torch.log_softmax(zs * inv_ts, dim=1)  # the sampler's tempered distribution
        if cfg["top_p"] < 1.0:
            srt, idx = torch.sort(logq, dim=1, descending=True)
            cum = torch.cumsum(srt.exp(), dim=1)
            keep_sorted = (cum - srt.exp()) < cfg["top_p"]  # smallest prefix reaching top_p
            n_keep = keep_sorted.sum(1)
            keep = torch.zeros_like(keep_sorted).scatter_(1, idx, keep_sorted)
            mu_lp = torch.where(keep, logq, torch.full_like(logq, -math.inf))
            mu_lp = mu_lp - torch.logsumexp(mu_lp, dim=1, keepdim=True)
            del srt, idx, cum, keep_sorted, keep
        else:
            n_keep = torch.full((nb,), V, device=device)
            mu_lp = logq
        top_lp, top_id = torch.topk(mu_lp, K, dim=1)
        rec_ids[b0:b1] = top_id.to(torch.int32)
        rec_lp[b0:b1] = top_lp
        if cfg["k_uniform"]:
            kt = torch.randint(1, K + 1, (nb,), generator=g, device=device)
            cnt = torch.minimum(kt, n_keep.clamp(max=K).to(kt.dtype))
            rec_count[b0:b1] = cnt.to(torch.int32)
        else:
            cnt = torch.full((nb,), K, device=device)
        if cfg["head_boost"] is not None:
            # the trainer's logits of the recorded ids raised by a per-row amount
            lo_b, hi_b = cfg["head_boost"]
            boost = lo_b + (hi_b - lo_b) * torch.rand(nb, generator=g, device=device)
            pos = (torch.arange(K, device=device)[None, :] < cnt[:, None]).float()
            zb = z.float().scatter_add_(1, top_id, pos * boost[:, None])
            logits[b0:b1] = zb.to(torch.bfloat16)
            del zb, pos
        if cfg["p_outside"] > 0:
            in_head = torch.zeros(nb, V, dtype=torch.bool, device=device)
            pos = torch.arange(K, device=device)[None, :] < cnt[:, None]
            in_head.scatter_(1, top_id, pos)
            outside = torch.rand(nb, generator=g, device=device) < cfg["p_outside"]
            # 95%: mu restricted to the recorded ids; 5%: the untruncated tempered
            # distribution restricted to the unrecorded ids.
            w_in = torch.where(in_head, mu_lp, torch.full_like(mu_lp, -math.inf))
            w_out = torch.where(in_head, torch.full_like(logq, -math.inf), logq)
            a_in = _gumbel_argmax(w_in, g)
            a_out = _gumbel_argmax(w_out, g)
            a = torch.where(outside, a_out, a_in)
            lp_a = torch.where(outside, logq.gather(1, a[:, None])[:, 0], mu_lp.gather(1, a[:, None])[:, 0])
            del in_head, w_in, w_out
        else:
            a = _gumbel_argmax(mu_lp, g)
            lp_a = mu_lp.gather(1, a[:, None])[:, 0]
        sampled[b0:b1] = a.to(torch.int32)
        rollout[b0:b1] = lp_a
        del z, zs, logq, mu_lp
    return dict(
        logits=logits, rec_ids=rec_ids, rec_logprobs=rec_lp, rec_count=rec_count, sampled=sampled,
        rollout_logprob=rollout, row_response=row_response.to(torch.int32).to(device),
        rewards=chunk_rewards.to(device), n_groups=chunk_rewards.numel() // n, group_size=n,
        inv_temperature=1.0 / cfg["temperature"], V=V, K=K, n_valid=int(valid.sum()),
    )


def to_numpy(batch: dict) -> dict:
    """Host numpy copies of a batch, with bf16 logits as uint16 bit patterns."""
    out = {}
    for k, v in batch.items():
        if isinstance(v, torch.Tensor):
            t = v.detach().cpu()
            out[k] = t.view(torch.int16).numpy().view("uint16") if t.dtype == torch.bfloat16 else t.numpy()
        else:
            out[k] = v
    return out


def lmhead_batch(T: int, d: int, V: int, K: int = 128, seed: int = 7, dyadic: bool = True, sigma_s: float = 0.05,
                 n_resp: int = 4, pad_frac: float = 0.2) -> dict:
    """Inputs of the LM head followed by score centering (CPU tensors).

    hidden bf16 [T, d] and w bf16 [V, d].  With `dyadic`, hidden lies on a
    1/8 grid in [-1, 1] and w on a 1/16 grid in [-1, 1], so every product and
    every sum of d <= 2048 of them is exact in FP32: the trainer's logits
    H W^T need no rounding before their single rounding to bf16.  Otherwise
    both are N(0, 1) scaled so the logits have a standard deviation near 3.
    The sampler's view: FP32 logits H W^T (computed here in FP32 on the CPU,
    as a sampler would) plus N(0, sigma_s^2) noise; the recorded ids are its
    top-K with FP32 log-probabilities, the sampled token is drawn from it.
    The last rows of every response are padding (about pad_frac of them).
    """
    g = torch.Generator().manual_seed(seed)
    if dyadic:
        H = torch.randint(-8, 9, (T, d), generator=g).float() / 8.0
        W = torch.randint(-16, 17, (V, d), generator=g).float() / 16.0
        W = W * (3.0 / (math.sqrt(d) * 0.6))
        W = torch.round(W * 16.0) / 16.0  # back on the 1/16 grid
        W = W.clamp(-1.0, 1.0)
    else:
        H = torch.randn(T, d, generator=g)
        W = torch.randn(V, d, generator=g) * (3.0 / math.sqrt(d))
    hidden = H.to(torch.bfloat16)
    w = W.to(torch.bfloat16)
    z = hidden.float() @ w.float().T
    zs = z + torch.randn(z.shape, generator=g) * sigma_s
    mu = torch.softmax(zs, dim=1)
    Kp = min(K, V)
    top = torch.topk(mu, Kp, dim=1)
    rec_ids = top.indices.to(torch.int32)
    rec_lp = torch.log(top.values).to(torch.float32)
    gum = -torch.log(-torch.log(torch.rand(zs.shape, generator=g).clamp_min(1e-20)))
    sampled = torch.argmax(torch.log(mu.clamp_min(1e-38)) + gum, dim=1).to(torch.int32)
    rl = torch.log(mu.gather(1, sampled.long()[:, None])[:, 0]).to(torch.float32)
    per = max(1, T // n_resp)
    resp = torch.arange(T, dtype=torch.int32) // per
    resp = torch.clamp(resp, max=n_resp - 1)
    pos = torch.arange(T) - resp.long() * per
    resp = torch.where(pos >= int(round(per * (1 - pad_frac))), torch.full_like(resp, -1), resp)
    rewards = (torch.rand(n_resp, generator=g) < 0.5).float()
    return dict(hidden=hidden, w=w, rec_ids=rec_ids, rec_logprobs=rec_lp, rec_count=None, sampled=sampled,
                rollout_logprob=rl, row_response=resp, rewards=rewards, n_groups=1, group_size=n_resp, K=Kp, V=V,
                inv_temperature=1.0)
