"""Vocabulary-sharded verify-and-commit: the library's sv_vshard_* kernels
with the two exchanges between shards in between.

Each shard holds a contiguous slice [v0, v0 + Vs) of the vocabulary for every
target (and draft) row, as a tensor-parallel LM head leaves it; the shards
cover [0, V) in order. The kernels do every step of the method; this module
only moves their small outputs between shards:

  stats  (every shard)  -> all-gather [S, rows] -> decide (every shard, alike)
  masses (every shard)  -> all-gather [S, B]    -> draw (the owning shard)
  draw_tok / draw_prob  -> max over shards      -> finish

Two ways to hold the shards: all of them in this process (`LocalShards`,
e.g. on one GPU), or one per rank of a torch.distributed group
(`GroupShards`; rank order is vocabulary order).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import List, Optional, Sequence

import torch

from . import api

STAT_WORDS = 8  # sv_shard_stat: 32 bytes as 8 int32 words


@dataclass
class Shard:
    target: torch.Tensor            # [R_t, Vs] slice of the target logits
    draft: Optional[torch.Tensor]   # [R_d, Vs] slice of the draft logits, or None (one-hot)
    v0: int                         # first vocabulary index of the slice


class LocalShards:
    """Every shard in this process: gathers stack the shards' parts in order
    and the max is taken over them."""

    def gather(self, parts: Sequence[torch.Tensor]) -> torch.Tensor:
        return torch.stack(list(parts))

    def max(self, parts: Sequence[torch.Tensor]) -> torch.Tensor:
        out = parts[0].clone()
        for p in parts[1:]:
            torch.maximum(out, p, out=out)
        return out

    def bit_or(self, t: torch.Tensor) -> torch.Tensor:
        return t  # the local shards already share one status word

    def first_index(self, n_local: int) -> int:
        return 0

    def count(self, n_local: int) -> int:
        return n_local


class GroupShards:
    """One shard per rank of a torch.distributed process group. With the
    gloo backend the exchanges go through host copies."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.host = dist.get_backend(group) == "gloo"

    def _io(self, t: torch.Tensor):
        return t.cpu() if self.host and t.is_cuda else t

    def gather(self, parts: Sequence[torch.Tensor]) -> torch.Tensor:
        assert len(parts) == 1, "one shard per rank"
        t = self._io(parts[0].contiguous())
        out = [torch.empty_like(t) for _ in range(self.world)]
        self.dist.all_gather(out, t, group=self.group)
        return torch.stack(out).to(parts[0].device)

    def max(self, parts: Sequence[torch.Tensor]) -> torch.Tensor:
        assert len(parts) == 1, "one shard per rank"
        t = self._io(parts[0].clone())
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX, group=self.group)
        return t.to(parts[0].device)

    def bit_or(self, t: torch.Tensor) -> torch.Tensor:
        u = self._io(t.clone())
        self.dist.all_reduce(u, op=self.dist.ReduceOp.BOR, group=self.group)
        return u.to(t.device)

    def first_index(self, n_local: int) -> int:
        return self.rank

    def count(self, n_local: int) -> int:
        return self.world


def _fns():
    lib = api.load()
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.sv_vshard_jobs_bytes.argtypes = [i32]
    lib.sv_vshard_jobs_bytes.restype = ctypes.c_size_t
    lib.sv_vshard_stats.argtypes = [P, ctypes.c_int, i32, i32, i64, i32, i32, i32, i32, P, P, f32, P, P, P]
    lib.sv_vshard_decide.argtypes = [P, P, i32, i32, i32, i32, P, P, P, P, f32, P, P, P, P, P, P]
    lib.sv_vshard_masses.argtypes = [P, P, ctypes.c_int, i32, i64, i32, i32, i32, P, P, P, f32, P, P]
    lib.sv_vshard_draw.argtypes = [P, P, ctypes.c_int, i32, i64, i32, i32, i32, i32, i32, P, P, P, P, P, f32,
                                   P, P, P, P]
    lib.sv_vshard_finish.argtypes = [P, i32, i32, P, P, P, P, P, P]
    for n in ("sv_vshard_stats", "sv_vshard_decide", "sv_vshard_masses", "sv_vshard_draw", "sv_vshard_finish"):
        getattr(lib, n).restype = ctypes.c_int
    return lib


def spec_verify_vsharded(shards: List[Shard], V: int, draft_tokens: torch.Tensor, cu_draft: torch.Tensor,
                         uniforms: torch.Tensor, temperature: float, mode: Optional[torch.Tensor] = None, *,
                         exchange=None, out_tokens=None, out_len=None, out_probs=None, status=None,
                         stream=None):
    """Verify-and-commit over vocabulary shards; the result (out_tokens,
    out_len, out_probs, status bits) is that of spec_verify on the whole
    vocabulary. `shards` are the shards this process holds, in vocabulary
    order; `exchange` is LocalShards() (the default) or GroupShards(group).
    Every process ends with the same outputs."""
    lib = _fns()
    ex = exchange if exchange is not None else LocalShards()
    t0 = shards[0].target
    dev = t0.device
    dtype = api._dtype(t0)
    B = cu_draft.shape[0] - 1
    R_t = t0.shape[0]
    R_d = int(draft_tokens.shape[0]) if draft_tokens is not None else 0
    has_draft = shards[0].draft is not None
    S = ex.count(len(shards))
    first = ex.first_index(len(shards))
    T = float(temperature)
    st = api._stream(stream)
    if out_tokens is None:
        out_tokens = torch.full((R_t,), -1, dtype=torch.int32, device=dev)
    if out_len is None:
        out_len = torch.zeros(B, dtype=torch.int32, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    P = api._ptr
    chk = api._check
    # 1. statistics of every local shard's slices
    tstats, dstats = [], []
    for sh in shards:
        Vs = sh.target.shape[1]
        ts = torch.empty((R_t, STAT_WORDS), dtype=torch.int32, device=dev)
        chk("sv_vshard_stats", lib.sv_vshard_stats(P(sh.target), dtype, R_t, Vs, sh.target.stride(0), sh.v0, V,
                                                   0, B, P(cu_draft), P(draft_tokens), T, P(ts), P(status), st))
        tstats.append(ts)
        if has_draft:
            ds = torch.empty((max(R_d, 1), STAT_WORDS), dtype=torch.int32, device=dev)
            chk("sv_vshard_stats", lib.sv_vshard_stats(P(sh.draft), dtype, R_d, Vs, sh.draft.stride(0), sh.v0, V,
                                                       1, B, P(cu_draft), P(draft_tokens), T, P(ds), P(status),
                                                       st))
            dstats.append(ds)
    all_t = ex.gather(tstats)                       # [S, R_t, 8]
    all_d = ex.gather(dstats) if has_draft else None
    if has_draft and R_d == 0:
        all_d = None
    # 2. decisions, alike on every shard
    jobs = torch.empty(max(int(lib.sv_vshard_jobs_bytes(B)), 16), dtype=torch.uint8, device=dev)
    chk("sv_vshard_decide", lib.sv_vshard_decide(P(all_t), P(all_d), S, V, B, R_t, P(cu_draft), P(draft_tokens),
                                                 P(mode), P(uniforms), T, P(out_tokens), P(out_len),
                                                 P(out_probs), P(jobs), P(status), st))
    # 3. residual masses of every local shard
    masses = []
    for k, sh in enumerate(shards):
        m = torch.empty(max(B, 1), dtype=torch.float64, device=dev)
        Vs = sh.target.shape[1]
        chk("sv_vshard_masses", lib.sv_vshard_masses(P(sh.target), P(sh.draft), dtype, Vs, sh.target.stride(0),
                                                     sh.v0, B, R_t, P(cu_draft), P(tstats[k]), P(jobs), T,
                                                     P(m), st))
        masses.append(m)
    all_m = ex.gather(masses)                       # [S, B]
    # 4. the draw, in the shard that owns it
    toks, probs = [], []
    for k, sh in enumerate(shards):
        dt_ = torch.empty(max(B, 1), dtype=torch.int32, device=dev)
        dp_ = torch.empty((max(B, 1), 2), dtype=torch.float32, device=dev)
        Vs = sh.target.shape[1]
        chk("sv_vshard_draw", lib.sv_vshard_draw(P(sh.target), P(sh.draft), dtype, Vs, sh.target.stride(0), sh.v0,
                                                 first + k, S, B, R_t, P(cu_draft), P(all_m), P(all_t), P(jobs),
                                                 P(uniforms), T, P(dt_), P(dp_), P(status), st))
        toks.append(dt_)
        probs.append(dp_)
    draw_tok = ex.max(toks)
    draw_prob = ex.max(probs)
    # 5. the drawn tokens into the outputs
    chk("sv_vshard_finish", lib.sv_vshard_finish(P(jobs), B, R_t, P(draw_tok), P(draw_prob), P(out_tokens),
                                                 P(out_probs), P(status), st))
    status.copy_(ex.bit_or(status))  # every shard's data-error bits
    return out_tokens, out_len, out_probs, status


def split_vocab(V: int, S: int) -> List[int]:
    """Shard starts of an even split of [0, V) into S slices, as a
    tensor-parallel LM head with S ranks would hold them; the last entry is V."""
    step = -(-V // S)
    return [min(V, s * step) for s in range(S)] + [V]
