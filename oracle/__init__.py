"""Plain float64 CPU oracle for speculative-decoding verify-and-commit and the
n-gram proposer -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg import this package. The CUDA library never uses it and the
two share no code: the oracle is ``oracle.c`` (float64, one row at a time,
written from the pages' algorithm), compiled with gcc into ``liboracle.so``
beside it and called through ctypes with numpy arrays.

What each function follows is cited in ``oracle.c``. Every function here is
pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

FP32, BF16 = 0, 1
MODE_SAMPLE, MODE_GREEDY = 0, 1
MARGIN_EPS = 1e-6

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, IEEE float64: no fast-math,
    no FMA contraction, so x86 and Arm give the same results)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", "-o", tmp, _SRC, "-lm", "-lpthread",
        ])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_softmax.argtypes = [P, i32, i32, f64, P]
        lib.oracle_softmax.restype = f64
        lib.oracle_argmax.argtypes = [P, i32, i32]
        lib.oracle_argmax.restype = i32
        lib.oracle_inverse_cdf.argtypes = [P, i32, f64, P]
        lib.oracle_inverse_cdf.restype = i32
        lib.oracle_spec_verify.argtypes = [P, P, i32, i32, i32, P, P, P, P, f64,
                                           P, P, P, P, P, P, i32]
        lib.oracle_spec_verify.restype = i32
        lib.oracle_spec_verify_filtered.argtypes = [P, P, i32, i32, i32, P, P, P, P, f64, i32, f64,
                                                    P, P, P, P, P, P, i32]
        lib.oracle_spec_verify_filtered.restype = i32
        lib.oracle_filtered_softmax.argtypes = [P, i32, i32, f64, i32, f64, P, P]
        lib.oracle_filtered_softmax.restype = f64
        lib.oracle_ngram_propose.argtypes = [P, i64, P, i32, i32, i32, i32, P, P, P]
        lib.oracle_ngram_propose.restype = i32
        lib.oracle_default_threads.argtypes = []
        lib.oracle_default_threads.restype = i32
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(z):
    """float32 array -> (array, FP32); uint16 array of bf16 bit patterns -> (array, BF16)."""
    z = np.ascontiguousarray(z)
    if z.dtype == np.float32:
        return z, FP32
    if z.dtype == np.uint16:
        return z, BF16
    raise TypeError("logits must be float32 or uint16 (bf16 bit patterns)")


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def softmax(z, T: float = 1.0) -> np.ndarray:
    """Temperature softmax of one logit row, float64."""
    z, dt = _logits(z)
    out = np.empty(z.shape[-1], np.float64)
    _load().oracle_softmax(_ptr(z), dt, z.shape[-1], float(T), _ptr(out))
    return out


def argmax(z) -> int:
    """First index of the maximal logit."""
    z, dt = _logits(z)
    return int(_load().oracle_argmax(_ptr(z), dt, z.shape[-1]))


def inverse_cdf(r, u: float):
    """(index, margin) of the inverse-CDF draw from unnormalised weights r."""
    r = np.ascontiguousarray(r, np.float64)
    m = np.zeros(1, np.float64)
    k = _load().oracle_inverse_cdf(_ptr(r), r.shape[0], float(u), _ptr(m))
    return int(k), float(m[0])


@dataclass
class VerifyResult:
    out_tokens: np.ndarray  # [R_t] int32; request b's tokens at cu_draft[b]+b
    out_len: np.ndarray     # [B] int32
    out_probs: np.ndarray   # [R_t, 2] float64
    margin: np.ndarray      # [R_t] float64, smallest decision margin of the row (inf if none)
    rho: np.ndarray         # [R_t] float64, min(1, p/q) of tested sampling rows (nan otherwise)
    stop: np.ndarray        # [B] int32

    def flagged_rows(self) -> np.ndarray:
        return self.margin < MARGIN_EPS


def filtered_softmax(row, temperature: float, top_k: int = 0, top_p: float = 1.0):
    """(p, top-p decision margin) of one logit row under the top-k / top-p
    filters (oracle.c, oracle_filtered_softmax)."""
    row, dt = _logits(np.asarray(row)[None, :] if np.asarray(row).ndim == 1 else row)
    V = row.shape[-1]
    p = np.zeros(V, np.float64)
    m = ctypes.c_double(0.0)
    _load().oracle_filtered_softmax(_ptr(row), dt, V, float(temperature), int(top_k), float(top_p),
                                    _ptr(p), ctypes.byref(m))
    return p, m.value


def spec_verify(target, draft, draft_tokens, cu_draft, uniforms, temperature: float,
                mode=None, nthreads: int = 0, diagnostics: bool = True, top_k: int = 0,
                top_p: float = 1.0) -> VerifyResult:
    """Verify-and-commit for a packed batch (layout as the CUDA library's).

    target: [R_t, V] float32 or uint16(bf16); draft: [R_d, V] same dtype or None
    (one-hot q); draft_tokens: [R_d] int32; cu_draft: [B+1] int32; uniforms:
    [R_t, 2] float32; mode: [B] uint8 (0 sample, 1 greedy) or None. diagnostics=False skips the
    per-row (p(x̂), q(x̂)) outputs, leaving only the method's own work.
    top_k / top_p (0 / 1.0: off) filter the target and draft distributions
    alike before the step (oracle.c, oracle_filtered_softmax).
    """
    target, dt = _logits(target)
    V = target.shape[-1]
    if draft is not None:
        draft, dt2 = _logits(draft)
        assert dt2 == dt and draft.shape[-1] == V
    draft_tokens = np.ascontiguousarray(draft_tokens, np.int32)
    cu_draft = np.ascontiguousarray(cu_draft, np.int32)
    uniforms = np.ascontiguousarray(uniforms, np.float32)
    B = cu_draft.shape[0] - 1
    R_t = int(cu_draft[-1]) + B
    assert target.shape[0] >= R_t and uniforms.shape[0] >= R_t
    if mode is not None:
        mode = np.ascontiguousarray(mode, np.uint8)
    out_tokens = np.full(R_t, -1, np.int32)
    out_len = np.zeros(B, np.int32)
    out_probs = np.full((R_t, 2), np.nan, np.float64)
    margin = np.full(R_t, np.inf, np.float64)
    rho = np.full(R_t, np.nan, np.float64)
    stop = np.zeros(B, np.int32)
    st = _load().oracle_spec_verify_filtered(
        _ptr(target), _ptr(draft), dt, V, B, _ptr(draft_tokens), _ptr(cu_draft), _ptr(mode),
        _ptr(uniforms), float(temperature), int(top_k), float(top_p), _ptr(out_tokens), _ptr(out_len),
        _ptr(out_probs) if diagnostics else None, _ptr(margin), _ptr(rho), _ptr(stop), int(nthreads))
    if st != 0:
        raise ValueError(f"oracle_spec_verify: invalid request data (code {st})")
    return VerifyResult(out_tokens, out_len, out_probs, margin, rho, stop)


def ngram_propose(histories, hist_len, min_n: int, max_n: int, max_tokens: int):
    """(out_tokens [B, max_tokens], out_count [B], out_n [B]) for int32 histories [B, stride]."""
    histories = np.ascontiguousarray(histories, np.int32)
    if histories.ndim == 1:
        histories = histories[None, :]
    hist_len = np.ascontiguousarray(hist_len, np.int32)
    B, stride = histories.shape
    out = np.full((B, max(max_tokens, 0)), -1, np.int32)
    cnt = np.zeros(B, np.int32)
    nn = np.zeros(B, np.int32)
    st = _load().oracle_ngram_propose(_ptr(histories), stride, _ptr(hist_len), B, int(min_n),
                                      int(max_n), int(max_tokens), _ptr(out), _ptr(cnt), _ptr(nn))
    if st != 0:
        raise ValueError("oracle_ngram_propose: history length out of range")
    return out, cnt, nn


# ---------------------------------------------------------------------------
# Acceptance statistics and the draft-length controller (plain Python)
# ---------------------------------------------------------------------------
def acceptance_metrics(cu_draft, out_len, max_pos: int = 32) -> dict:
    """Counts of "5.2 Draft 模型与无模型方案", §7.1-7.2, over the rounds of one
    or more verify calls (each request is a round).

    D: proposed draft tokens; C: accepted draft tokens, i.e. the tokens
    committed from the draft before the first rejection (out_len - 1);
    R: rounds. Per slot i: offered (K_b > i), reached (slot i was tested, so
    every earlier slot was accepted) and accepted_at (slots 0..i accepted).
    """
    cu = [int(x) for x in cu_draft]
    lens = [int(x) for x in out_len]
    m = {"rounds": 0, "rounds_with_draft": 0, "drafted": 0, "accepted": 0, "committed": 0,
         "offered": [0] * max_pos, "reached": [0] * max_pos, "accepted_at": [0] * max_pos}
    for b in range(len(lens)):
        K = max(0, cu[b + 1] - cu[b])
        length = min(max(lens[b], 1), K + 1)
        stop = length - 1  # slots 0..stop-1 accepted; slot stop rejected, or the bonus slot
        m["rounds"] += 1
        if K > 0:
            m["rounds_with_draft"] += 1
        m["drafted"] += K
        m["accepted"] += stop
        m["committed"] += length
        for i in range(min(K, max_pos)):
            m["offered"][i] += 1
            if i <= stop:
                m["reached"][i] += 1
            if i < stop:
                m["accepted_at"][i] += 1
    return m


def derived_rates(m: dict) -> dict:
    """The page's quantities from the counts: C/D, 1 + C/R, coverage, and per
    slot the conditional rate and the rate through that slot."""
    R, D, C = m["rounds"], m["drafted"], m["accepted"]
    return {
        "draft_acceptance_rate": C / D if D else float("nan"),
        "mean_acceptance_length": 1 + C / R if R else float("nan"),
        "coverage": m["rounds_with_draft"] / R if R else float("nan"),
        "conditional": [a / r if r else float("nan") for a, r in zip(m["accepted_at"], m["reached"])],
        "through": [a / o if o else float("nan") for a, o in zip(m["accepted_at"], m["offered"])],
    }


class AdaptiveDraftLength:
    """Sliding-window draft-length rule of "投机解码从零实现" §5.2
    (动态草稿长度策略): keep the accepted fraction of the last `window`
    rounds; from 10 rounds on, after each round move the draft length one
    step up when the window's mean exceeds target + 0.1, one step down when
    it falls below target - 0.1, within [min_k, max_k]."""

    def __init__(self, window=100, min_k=1, max_k=10, target=0.7, initial_k=5):
        self.window, self.min_k, self.max_k, self.target = window, min_k, max_k, float(target)
        self.k = initial_k
        self.fractions = []

    def update(self, draft_len: int, accepted_len: int) -> int:
        self.fractions.append(accepted_len / max(draft_len, 1))
        if len(self.fractions) > self.window:
            self.fractions = self.fractions[1:]
        if len(self.fractions) >= 10:
            total = 0.0
            for f in self.fractions:  # oldest first
                total += f
            mean = total / len(self.fractions)
            if mean > self.target + 0.1:
                self.k = min(self.max_k, self.k + 1)
            elif mean < self.target - 0.1:
                self.k = max(self.min_k, self.k - 1)
        return self.k


# ---------------------------------------------------------------------------
# Multi-candidate verification: keep the candidate with the longest commit
# ---------------------------------------------------------------------------
def select_candidates(cu_cand, out_len, policy: str = "uniform", u_select=None):
    """Request b owns candidates cu_cand[b] .. cu_cand[b+1]-1, each verified as
    its own request ("投机解码从零实现" §5.1 批量验证: one pass verifies several
    drafts, each returning its accepted tokens and gain). The page does not
    say which result to keep; two rules:

    "uniform": candidate cu_cand[b] + min(n - 1, floor(u * n)) for n
      candidates and the request's selection uniform u = u_select[b] (a
      negative or NaN u picks the first). The choice does not depend on any
      verification outcome, so the kept commit is distributed as a single
      candidate's: lossless ("Draft Model（草稿模型）" §2).
    "longest": the longest committed length, the lowest index among ties.
      It raises the expected gain but looks at the outcomes, so the kept
      commit is no longer distributed as the target's.

    Returns (best [B] global candidate index, or -1 for a request without
    candidates; best_len [B], 0 then)."""
    cu = [int(x) for x in cu_cand]
    lens = [int(x) for x in out_len]
    if policy not in ("uniform", "longest"):
        raise ValueError(policy)
    if policy == "uniform" and u_select is None:
        raise ValueError("the uniform rule needs u_select")
    best, best_len = [], []
    for b in range(len(cu) - 1):
        n = cu[b + 1] - cu[b]
        bi, bl = -1, 0
        if n > 0 and policy == "uniform":
            u = float(u_select[b])
            j = int(np.floor(u * n)) if u >= 0.0 else 0
            bi = cu[b] + min(n - 1, j)
            bl = lens[bi]
        elif n > 0:
            for c in range(cu[b], cu[b + 1]):
                if bi < 0 or lens[c] > bl:
                    bi, bl = c, lens[c]
        best.append(bi)
        best_len.append(bl)
    return np.array(best, np.int32), np.array(best_len, np.int32)


# ---------------------------------------------------------------------------
# Suffix proposer: frequency-ranked continuation ("5.2 Draft 模型与无模型方案",
# §5.1-5.2 Suffix Decoding), plain Python
# ---------------------------------------------------------------------------
def suffix_propose(histories, hist_len, min_n: int, max_n: int, max_tokens: int,
                   min_share: float = 0.5, max_occ: int = 256):
    """For each history: the longest tail h[L-n, L) (n from min(max_n, L) down
    to min_n) that occurs earlier, with the same admissible starts as the
    n-gram proposer (0 <= s <= L-2n-1, so a continuation token precedes the
    tail); the max_occ most recent occurrences vote. Step j: every
    occurrence still in agreement whose continuation h[s+n+j] lies before the
    tail votes for that token; the most frequent token wins (ties: the token
    of the most recent voter). From the second step on, the proposal stops
    when the winner holds less than min_share of the votes (dispersed
    continuations); the occurrences that voted for the winner go on.
    Returns (out_tokens [B, max_tokens] (-1 padded), count [B], n [B])."""
    histories = np.asarray(histories)
    B = histories.shape[0]
    share = float(np.float32(min_share))
    out = np.full((B, max(max_tokens, 0)), -1, np.int32)
    cnt = np.zeros(B, np.int32)
    nn = np.zeros(B, np.int32)
    for b in range(B):
        L = int(hist_len[b])
        h = [int(x) for x in histories[b, :L]]
        occ, n = [], 0
        for m in range(min(max_n, L), min_n - 1, -1):
            tail = h[L - m:L]
            occ = [s for s in range(L - 2 * m - 1, -1, -1) if h[s:s + m] == tail]  # most recent first
            if occ:
                n = m
                break
        if not occ:
            continue
        active = occ[:max_occ]
        props = []
        for j in range(max_tokens):
            votes = [(s, h[s + n + j]) for s in active if s + n + j < L - n]
            if not votes:
                break
            count, recent = {}, {}
            for s, t in votes:
                count[t] = count.get(t, 0) + 1
                recent.setdefault(t, s)  # votes run most recent first
            win = max(count, key=lambda t: (count[t], recent[t]))
            if j > 0 and float(count[win]) < share * float(len(votes)):
                break
            props.append(win)
            active = [s for s, t in votes if t == win]
        out[b, :len(props)] = props
        cnt[b] = len(props)
        nn[b] = n
    return out, cnt, nn
