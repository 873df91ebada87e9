"""Data-parallel helpers for the score-centering loss.

Rows are independent, so the path shards over rows with no data-path
exchange.  Two things span ranks:

* the loss is a mean over every generated token of the whole step (the
  docs' "Score Centering" section reduces over all of them), so every rank
  needs the global count of valid rows: one int64 all-reduce per batch;
* advantages are normalised within a group of responses to one prompt, so a
  shard boundary must not cut a group: :func:`shard_groups` splits whole
  groups.

Token counts stay integers until the final division, which is done in double
precision (the devotd.net release note, section 4, keeps token counts unrounded).
"""

from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist


def shard_groups(n_groups: int, world_size: int, rank: int) -> range:
    """Contiguous block of whole groups owned by `rank` (sizes differ by at most one)."""
    if world_size < 1 or not 0 <= rank < world_size or n_groups < 0:
        raise ValueError("bad world_size / rank / n_groups")
    base, extra = divmod(n_groups, world_size)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def global_valid_tokens(n_valid_local: int, group=None, device=None) -> int:
    """Sum of the ranks' valid-row counts (int64 all-reduce; local count if not distributed)."""
    t = torch.tensor([int(n_valid_local)], dtype=torch.int64, device=device)
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return int(t.item())


def token_mean_scale(n_valid_global: int) -> float:
    """grad_scale for a global token mean: 1 / N in double, rounded once to FP32."""
    if n_valid_global <= 0:
        return 0.0
    return float(np.float32(1.0 / float(n_valid_global)))
