"""Helpers of the parity tests: move a generated batch to the GPU, run the CUDA
library through its C ABI, run the float64 oracle on the same inputs, and
compare them.

Tolerance (the benchmark spec): greedy and n-gram outputs bit-exact; in sampling mode
probabilities within 1e-6 absolute, and committed tokens and lengths identical
except on requests where the oracle's decision margin (|u - min(1, p/q)| or the
distance of u' to an edge of the chosen residual-CDF bucket) is below 1e-6 for
some row up to its stop row -- those are "flagged".

Budget: flagged rows may number at most FLAG_BUDGET (1e-4) of all rows. The
draw margin cannot meet that on flat rows over a large vocabulary, whatever
computes the draw: a bucket of width w catches u' within 1e-6 of an edge with
probability min(w, 2e-6), so a draw over 32000 near-uniform tokens is flagged
a few percent of the time. The full-configuration tests therefore assert the
budget on the accept-test flags and on the requests that actually differ on
every configuration, and on all flags where the rows are peaked or greedy.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

PROB_TOL = 1e-6
FLAG_BUDGET = 1e-4


def logits_to_device(a, device="cuda"):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)


@dataclass
class DeviceBatch:
    target: torch.Tensor
    draft: torch.Tensor | None
    draft_tokens: torch.Tensor
    cu_draft: torch.Tensor
    uniforms: torch.Tensor
    mode: torch.Tensor | None
    temperature: float


def to_device(batch, device="cuda") -> DeviceBatch:
    toks = batch.draft_tokens if batch.draft_tokens.size else np.zeros(1, np.int32)
    return DeviceBatch(
        logits_to_device(batch.target, device), logits_to_device(batch.draft, device),
        torch.from_numpy(np.ascontiguousarray(toks, np.int32)).to(device),
        torch.from_numpy(np.ascontiguousarray(batch.cu_draft, np.int32)).to(device),
        torch.from_numpy(np.ascontiguousarray(batch.uniforms, np.float32)).to(device),
        None if batch.mode is None else torch.from_numpy(np.ascontiguousarray(batch.mode, np.uint8)).to(device),
        float(batch.temperature))


def gpu_verify(db: DeviceBatch, workspace=None):
    from speculative_decoding_verification_27_gb300 import api
    tok, ln, pr = api.spec_verify(db.target, db.draft, db.draft_tokens, db.cu_draft, db.uniforms,
                                  db.temperature, db.mode, workspace=workspace)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), ln.cpu().numpy(), pr.cpu().numpy()


def oracle_verify(batch, nthreads=0):
    import oracle
    return oracle.spec_verify(batch.target, batch.draft, batch.draft_tokens, batch.cu_draft,
                              batch.uniforms, batch.temperature, batch.mode, nthreads)


@dataclass
class ParityReport:
    requests: int
    rows: int
    flagged_requests: int
    flagged_rows: int
    mismatched_requests: int
    max_prob_err: float
    accept_flagged_rows: int = 0   # rows flagged by their accept test alone


    def as_dict(self):
        return self.__dict__.copy()


def assert_flag_budget(flagged_rows: int, rows: int, budget: float = FLAG_BUDGET):
    """At most `budget` of all rows may be flagged (decision margin < 1e-6)."""
    assert flagged_rows <= budget * rows, f"{flagged_rows} flagged rows of {rows} (budget {budget})"


def accept_flags(batch, ora) -> np.ndarray:
    """Rows whose accept test was taken with |u - rho| < 1e-6."""
    u = batch.uniforms[:batch.R_t, 0].astype(np.float64)
    rho = ora.rho[:batch.R_t]
    tested = ~np.isnan(rho)
    return tested & (np.abs(u - np.where(tested, rho, 0.0)) < 1e-6)


def check_budget(rep: "ParityReport", budget: float = FLAG_BUDGET, draw_flags_in_budget: bool = True):
    """The flag budget (see the module docstring): accept-test flags and
    differing requests always; all flagged rows when draw_flags_in_budget."""
    assert_flag_budget(rep.accept_flagged_rows, rep.rows, budget)
    assert rep.mismatched_requests <= budget * rep.rows, \
        f"{rep.mismatched_requests} differing requests over {rep.rows} rows (budget {budget})"
    if draw_flags_in_budget:
        assert_flag_budget(rep.flagged_rows, rep.rows, budget)


def compare(batch, gpu, ora, prob_tol=PROB_TOL, flag_budget=None,
            draw_flags_in_budget=True) -> ParityReport:
    """Asserts parity of one call; returns its counts. With flag_budget, also
    checks the budget (check_budget)."""
    tok, ln, pr = gpu
    cu = batch.cu_draft.astype(np.int64)
    B = batch.B
    K = np.diff(cu)
    t0 = cu[:-1] + np.arange(B)
    greedy = batch.greedy_mask()
    flagged_rows = ora.flagged_rows()
    flagged = np.zeros(B, bool)
    mism = np.zeros(B, bool)
    for b in range(B):
        s = int(ora.stop[b])
        flagged[b] = bool(flagged_rows[t0[b]:t0[b] + s + 1].any())
        n = int(ora.out_len[b])
        if ln[b] != n or not np.array_equal(tok[t0[b]:t0[b] + n], ora.out_tokens[t0[b]:t0[b] + n]):
            mism[b] = True
    bad = np.nonzero(mism & ~flagged)[0]
    assert bad.size == 0, f"unflagged mismatches in requests {bad[:10]}"
    assert np.all(ln >= 1) and np.all(ln <= K + 1)
    # Greedy requests carry (-1, -1) on every row.
    req_of_row = np.repeat(np.arange(B), K + 1)
    g_rows = greedy[req_of_row]
    assert np.all(pr[g_rows] == -1.0)
    # Draft-slot rows of sampling requests: (p(x̂), q(x̂)) on every slot.
    slot = np.ones(batch.R_t, bool)
    slot[t0 + K] = False
    sel = slot & ~g_rows
    err = float(np.max(np.abs(pr[sel] - ora.out_probs[sel]), initial=0.0))
    # Bonus-slot rows: probabilities of the final token, where it matches.
    bsel = t0 + K
    ok = ~greedy & ~mism
    err_b = float(np.max(np.abs(pr[bsel[ok]] - ora.out_probs[bsel[ok]]), initial=0.0))
    max_err = max(err, err_b)
    assert max_err <= prob_tol, f"probability error {max_err}"
    rep = ParityReport(B, batch.R_t, int(flagged.sum()), int(flagged_rows.sum()), int(mism.sum()), max_err,
                       int(accept_flags(batch, ora).sum()))
    if flag_budget is not None:
        check_budget(rep, flag_budget, draw_flags_in_budget)
    return rep
