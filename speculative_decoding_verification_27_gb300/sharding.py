"""Partition of a verify batch over ranks (one process per GPU).

Requests are independent: each rank can verify a contiguous range of requests
with its own spec_verify call, and no data crosses ranks. In the packed
ragged layout a contiguous request range [lo, hi) owns contiguous blocks of
every array:

  target rows / uniforms / out_tokens / out_probs   [cu[lo] + lo, cu[hi] + hi)
  draft rows / draft tokens                         [cu[lo], cu[hi])
  out_len / mode                                    [lo, hi)

so a shard is a set of slices plus the rebased offsets cu[lo:hi+1] - cu[lo],
and the global outputs are the ranks' outputs concatenated in rank order.

The split balances the logit bytes each rank must read: a sampling request
reads 2 K_b + 1 rows (K_b + 1 target rows and K_b draft rows, or only the
target rows with one-hot proposals), a greedy request K_b + 1.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


def request_weights(cu_draft: np.ndarray, greedy: np.ndarray | None, has_draft: bool) -> np.ndarray:
    """Logit rows each request reads."""
    K = np.diff(np.asarray(cu_draft, np.int64))
    w = K + 1
    if has_draft:
        g = np.zeros(K.size, bool) if greedy is None else np.asarray(greedy, bool)
        w = w + np.where(g, 0, K)
    return w


def partition_requests(cu_draft: np.ndarray, world: int, greedy: np.ndarray | None = None,
                       has_draft: bool = True) -> np.ndarray:
    """[world + 1] request boundaries: rank r verifies requests [bounds[r], bounds[r + 1]).

    Rank r's range ends at the first request whose cumulative weight reaches
    (r + 1) / world of the total, so every rank gets within one request's
    weight of an equal share. Ranks may get no request when B < world.
    """
    if world < 1:
        raise ValueError("world must be >= 1")
    w = request_weights(cu_draft, greedy, has_draft)
    B = w.size
    cum = np.concatenate([[0], np.cumsum(w)])
    total = int(cum[-1])
    bounds = np.empty(world + 1, np.int64)
    bounds[0], bounds[-1] = 0, B
    for r in range(1, world):
        # smallest b with cum[b] * world >= r * total
        bounds[r] = int(np.searchsorted(cum * world, r * total, side="left"))
    return np.maximum.accumulate(np.minimum(bounds, B))


@dataclass(frozen=True)
class Shard:
    lo: int   # first request
    hi: int   # one past the last request
    t0: int   # first target row
    t1: int
    d0: int   # first draft row
    d1: int

    @property
    def B(self) -> int:
        return self.hi - self.lo


def shard_of(cu_draft: np.ndarray, lo: int, hi: int) -> Shard:
    cu = np.asarray(cu_draft, np.int64)
    return Shard(lo, hi, int(cu[lo] + lo), int(cu[hi] + hi), int(cu[lo]), int(cu[hi]))


def local_batch(batch, shard: Shard):
    """The shard as a batch of its own (views of the global arrays, offsets rebased)."""
    from .workloads import VerifyBatch

    s = shard
    cu = np.asarray(batch.cu_draft[s.lo:s.hi + 1], np.int64)
    cu_local = (cu - cu[0]).astype(np.int32)
    mode = None if batch.mode is None else batch.mode[s.lo:s.hi]
    draft = None if batch.draft is None else batch.draft[s.d0:s.d1]
    return VerifyBatch(f"{batch.name}[{s.lo}:{s.hi}]", batch.target[s.t0:s.t1], draft,
                       batch.draft_tokens[s.d0:s.d1], cu_local, batch.uniforms[s.t0:s.t1],
                       batch.temperature, mode, dict(batch.meta, shard=(s.lo, s.hi)))


def merge_outputs(parts):
    """Concatenates per-rank (out_tokens, out_len, out_probs) in rank order."""
    tok = np.concatenate([p[0] for p in parts])
    ln = np.concatenate([p[1] for p in parts])
    pr = None if parts[0][2] is None else np.concatenate([p[2] for p in parts])
    return tok, ln, pr


def gather_outputs(tok, ln, pr, group=None):
    """Every rank's shard outputs (numpy out_tokens, out_len, out_probs or
    None), gathered over a torch.distributed group and concatenated in rank
    order: the global outputs, on every rank. The arrays are a few KB per
    rank (tokens and lengths), so they travel as pickled objects."""
    import torch.distributed as dist

    parts = [None] * dist.get_world_size(group)
    dist.all_gather_object(parts, (tok, ln, pr), group=group)
    return merge_outputs(parts)
