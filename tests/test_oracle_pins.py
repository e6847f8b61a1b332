"""Pins of the float64 oracle against what the pages and the mathematics fix.

None of these re-type the oracle's formulas: they measure the oracle as a black
box (its decisions on the 2**-24 lattice of uniforms, its emitted tokens) and
compare with closed forms computed by library routines (scipy's softmax), the
worked example printed on the pages, and statistics of the lossless property.

Sources:
  * "Draft Model（草稿模型）", §2 "接受-拒绝准则": accept with probability
    min(1, p/q), else re-draw from norm(max(0, p - q)); the emitted marginal
    equals p. Box "算法：Speculative Decoding (一步)": stop at the first
    rejection, bonus token from p_{K+1} when all K are accepted, 1..K+1
    tokens per round. "接受率分析": E[accept] >= 1 - TV(p, q) (equality for
    one position: sum_x min(p, q)).
  * "投机解码从零实现" (CSDN), §3.3: p = 0.4, q = 0.6 -> reject 1/3;
    §4.3: temperature divides both logit rows; q <= 0 rejects.
  * "Speculative Decoding在分布式推理中的应用", §二: strict verification
    accepts iff the draft equals the target's choice.
  * "5.2 Draft 模型与无模型方案", §4.3 one-hot q for copied proposals;
    §6 the n-gram proposer and its printed results.
"""
import json
import os

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

from speculative_decoding_verification_27_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LAT = 2 ** 24


def _logits(p):
    return np.log(np.asarray(p, np.float64)).astype(np.float32)


def _run1(oracle_mod, zt, zd, toks, us, T=1.0, mode=None):
    """One request: zt [K+1, V], zd [K, V] or None, toks [K], us [K+1, 2]."""
    toks = np.asarray(toks, np.int32)
    cu = np.array([0, toks.shape[0]], np.int32)
    return oracle_mod.spec_verify(np.asarray(zt, np.float32),
                                  None if zd is None else np.asarray(zd, np.float32),
                                  toks, cu, np.asarray(us, np.float32), T,
                                  None if mode is None else np.asarray(mode, np.uint8))


def _first_false(pred):
    """Smallest lattice index j in [0, LAT] with pred(j / LAT) False (pred monotone)."""
    lo, hi = 0, LAT
    if not pred(0.0):
        return 0
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if pred(mid / LAT):
            lo = mid
        else:
            hi = mid
    return hi


def _accept_measure(oracle_mod, zt, zd, toks, row, us_base, T=1.0):
    """Lattice measure of {u_row : the oracle accepts at `row`}."""
    def accepted(u):
        us = np.array(us_base, np.float64)
        us[row, 0] = u
        return _run1(oracle_mod, zt, zd, toks, us, T).out_len[0] > row + 1
    return _first_false(accepted) / LAT


def _draw_widths(oracle_mod, zt, zd, toks, row, us_base, T=1.0):
    """Lattice widths of each token's bucket in the draw made at `row`."""
    V = zt.shape[1]

    def token(u2):
        us = np.array(us_base, np.float64)
        us[row, 1] = u2
        r = _run1(oracle_mod, zt, zd, toks, us, T)
        assert r.out_len[0] == row + 1
        return r.out_tokens[row]
    edges = [0] + [_first_false(lambda u, k=k: token(u) <= k) for k in range(V)]
    edges[-1] = LAT
    return np.diff(np.array(edges, np.float64)) / LAT


# --------------------------------------------------------------------------
# Worked example: p = 0.4, q = 0.6 -> reject with probability 1/3
# --------------------------------------------------------------------------
def test_worked_example_reject_one_third(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    zt = np.stack([_logits(g["p"]), _logits([0.5, 0.5])])
    zd = _logits(g["q"])[None]
    x = g["draft_token"]
    acc = _accept_measure(oracle_mod, zt, zd, [x], 0, [[0, 0.5], [0.5, 0.5]])
    assert abs((1 - acc) - g["reject_probability"]) < 2.0 / LAT
    # Decisions right at the edge flip exactly there.
    r_in = _run1(oracle_mod, zt, zd, [x], [[2 / 3 - 4 / LAT, 0.5], [0.5, 0.5]])
    r_out = _run1(oracle_mod, zt, zd, [x], [[2 / 3 + 4 / LAT, 0.5], [0.5, 0.5]])
    assert r_in.out_len[0] == 2 and r_in.out_tokens[0] == x
    assert r_out.out_len[0] == 1
    # After a rejection the residual max(0, p - q) = [0, 0.2] puts all mass on token 1.
    w = _draw_widths(oracle_mod, zt, zd, [x], 0, [[0.999, 0.5], [0.5, 0.5]])
    assert np.allclose(w, g["residual"], atol=1.0 / LAT)


def test_worked_example_statistics(oracle_mod):
    """1e6 rounds of the worked example: reject frequency 1/3 within 5 sigma."""
    N = 1_000_000
    zt = np.tile(np.stack([_logits([0.4, 0.6]), _logits([0.5, 0.5])]), (N, 1))
    zd = np.tile(_logits([0.6, 0.4])[None], (N, 1))
    cu = np.arange(N + 1, dtype=np.int32)
    us = W.uniforms_for(cu, seed=11)
    r = oracle_mod.spec_verify(zt, zd, np.zeros(N, np.int32), cu, us, 1.0)
    rej = r.out_len == 1
    f = rej.mean()
    assert abs(f - 1 / 3) < 5 * np.sqrt((1 / 3) * (2 / 3) / N)
    first = r.out_tokens[cu[:-1] + np.arange(N)]
    assert np.all(first[rej] == 1)


# --------------------------------------------------------------------------
# Closed forms of the accept probability and the draws
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1.0, 0.7, 1.9])
def test_accept_probability_and_residual_closed_form(oracle_mod, T):
    rng = np.random.default_rng(5)
    V = 4
    zt = rng.normal(0, 1.5, (2, V)).astype(np.float32)
    zd = (zt[:1] + rng.normal(0, 1.0, (1, V))).astype(np.float32)
    p = sp_softmax(zt[0].astype(np.float64) / T)
    q = sp_softmax(zd[0].astype(np.float64) / T)
    res = np.maximum(p - q, 0)
    res /= res.sum()
    for x in range(V):
        acc = _accept_measure(oracle_mod, zt, zd, [x], 0, [[0, 0.5], [0.5, 0.5]], T)
        assert abs(acc - min(1.0, p[x] / q[x])) < 2.0 / LAT, (x, acc, p[x] / q[x])
        if p[x] < q[x]:
            w = _draw_widths(oracle_mod, zt, zd, [x], 0, [[1 - 1 / LAT, 0.5], [0.5, 0.5]], T)
            assert np.allclose(w, res, atol=2.0 / LAT)


def test_bonus_draw_is_target_distribution(oracle_mod):
    rng = np.random.default_rng(6)
    V = 4
    zt = rng.normal(0, 1.0, (2, V)).astype(np.float32)
    zd = zt[:1].copy()  # q == p: always accepted, the draw happens at the bonus row
    w = _draw_widths(oracle_mod, zt, zd, [2], 1, [[0, 0.5], [0.5, 0.5]], 0.8)
    assert np.allclose(w, sp_softmax(zt[1].astype(np.float64) / 0.8), atol=2.0 / LAT)


def test_one_hot_proposal(oracle_mod):
    """One-hot q: accept with probability p(x̂); the residual is p without x̂."""
    rng = np.random.default_rng(8)
    V = 4
    zt = rng.normal(0, 1.0, (2, V)).astype(np.float32)
    p = sp_softmax(zt[0].astype(np.float64))
    for x in range(V):
        acc = _accept_measure(oracle_mod, zt, None, [x], 0, [[0, 0.5], [0.5, 0.5]])
        assert abs(acc - p[x]) < 2.0 / LAT
        w = _draw_widths(oracle_mod, zt, None, [x], 0, [[1 - 1 / LAT, 0.5], [0.5, 0.5]])
        ref = p.copy()
        ref[x] = 0
        assert np.allclose(w, ref / ref.sum(), atol=2.0 / LAT)


def test_zero_draft_probability_rejects(oracle_mod):
    zt = np.stack([_logits([0.5, 0.5]), _logits([0.5, 0.5])])
    zd = np.array([[0.0, -np.inf]], np.float32)  # q(1) = 0
    r = _run1(oracle_mod, zt, zd, [1], [[0.0, 0.3], [0.5, 0.5]])
    assert r.out_len[0] == 1 and r.rho[0] == 0.0


# --------------------------------------------------------------------------
# Lossless: exact lattice integration of the emitted marginals (V=4, K<=2)
# --------------------------------------------------------------------------
def _position_marginal(oracle_mod, zt, zd, row, us_base, T):
    """P(emitted token at `row`) given rows before it accepted, integrating
    over x̂ ~ q_row and both uniforms of the row, from black-box measures."""
    V = zt.shape[1]
    q = sp_softmax(zd[row].astype(np.float64) / T)
    P = np.zeros(V)
    for x in range(V):
        toks = [0] * zd.shape[0]
        toks[row] = x
        for j in range(row):  # earlier slots: any token, accepted via u = 0 if rho > 0
            toks[j] = int(np.argmax(zt[j]))
        acc = _accept_measure(oracle_mod, zt, zd, toks, row, us_base, T)
        P[x] += q[x] * acc
        if acc < 1.0:
            us = np.array(us_base, np.float64)
            us[row, 0] = 1 - 1 / LAT
            P += q[x] * (1 - acc) * _draw_widths(oracle_mod, zt, zd, toks, row, us, T)
    return P


@pytest.mark.parametrize("K", [1, 2])
def test_lossless_lattice_integration(oracle_mod, K):
    rng = np.random.default_rng(10 + K)
    V, T = 4, 0.9
    zt = rng.normal(0, 1.2, (K + 1, V)).astype(np.float32)
    zd = (zt[:K] + rng.normal(0, 1.0, (K, V))).astype(np.float32)
    us = np.zeros((K + 1, 2))
    us[:, 1] = 0.5
    for row in range(K):
        P = _position_marginal(oracle_mod, zt, zd, row, us, T)
        p = sp_softmax(zt[row].astype(np.float64) / T)
        assert np.abs(P - p).max() < 1e-6, (row, P, p)
    # All K accepted (u = 0 accepts whenever rho > 0): the bonus token ~ p_{K+1}.
    toks = [int(np.argmax(zt[j])) for j in range(K)]
    w = _draw_widths(oracle_mod, zt, zd, toks, K, us, T)
    assert np.abs(w - sp_softmax(zt[K].astype(np.float64) / T)).max() < 2.0 / LAT


# --------------------------------------------------------------------------
# Lossless: chi-square of the emitted marginal over 1e6 rounds (V = 16)
# --------------------------------------------------------------------------
def _sample(q, n, rng):
    return np.searchsorted(np.cumsum(q), rng.random(n), side="right").clip(0, q.shape[0] - 1).astype(np.int32)


CHI2_15DOF_999 = 37.70  # chi-square quantile, 15 degrees of freedom, alpha = 0.001


def test_chi_square_first_token_and_acceptance(oracle_mod):
    rng = np.random.default_rng(12)
    V, N, T = 16, 1_000_000, 1.0
    zp = rng.normal(0, 1.5, V).astype(np.float32)
    zb = rng.normal(0, 1.5, V).astype(np.float32)
    zq = (zp + rng.normal(0, 1.0, V)).astype(np.float32)
    p = sp_softmax(zp.astype(np.float64))
    q = sp_softmax(zq.astype(np.float64))
    cu = np.arange(N + 1, dtype=np.int32)
    zt = np.tile(np.stack([zp, zb]), (N, 1))
    zd = np.tile(zq[None], (N, 1))
    toks = _sample(q, N, rng)
    r = oracle_mod.spec_verify(zt, zd, toks, cu, W.uniforms_for(cu, seed=13), T)
    first = r.out_tokens[cu[:-1] + np.arange(N)]
    hist = np.bincount(first, minlength=V)
    chi2 = float(((hist - N * p) ** 2 / (N * p)).sum())
    assert chi2 < CHI2_15DOF_999, chi2
    # One position: E[accept] = sum_x min(p, q) = 1 - TV(p, q).
    alpha = np.minimum(p, q).sum()
    acc = (r.out_len == 2).mean()
    assert abs(acc - alpha) < 5 * np.sqrt(alpha * (1 - alpha) / N)


def test_chi_square_second_token_given_acceptance(oracle_mod):
    rng = np.random.default_rng(14)
    V, N, T = 16, 1_000_000, 1.3
    zt1 = rng.normal(0, 1.5, (3, V)).astype(np.float32)
    zq1 = (zt1[:2] + rng.normal(0, 0.7, (2, V))).astype(np.float32)
    q = [sp_softmax(zq1[i].astype(np.float64) / T) for i in range(2)]
    p2 = sp_softmax(zt1[1].astype(np.float64) / T)
    cu = np.arange(0, 2 * N + 1, 2, dtype=np.int32)
    zt = np.tile(zt1, (N, 1))
    zd = np.tile(zq1, (N, 1))
    toks = np.stack([_sample(q[0], N, rng), _sample(q[1], N, rng)], 1).reshape(-1)
    r = oracle_mod.spec_verify(zt, zd, toks, cu, W.uniforms_for(cu, seed=15), T)
    base = cu[:-1] + np.arange(N)
    sel = r.out_len >= 2
    second = r.out_tokens[base[sel] + 1]
    n = second.shape[0]
    hist = np.bincount(second, minlength=V)
    chi2 = float(((hist - n * p2) ** 2 / (n * p2)).sum())
    assert n > 100_000 and chi2 < CHI2_15DOF_999, (n, chi2)


# --------------------------------------------------------------------------
# Softmax, argmax, strict mode
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_softmax_matches_library(oracle_mod, T):
    rng = np.random.default_rng(20)
    z = rng.normal(0, 3.0, 4099).astype(np.float32)
    p = oracle_mod.softmax(z, T)
    ref = sp_softmax(z.astype(np.float64) / T)
    assert np.allclose(p, ref, rtol=1e-12, atol=0)
    assert abs(p.sum() - 1.0) < 1e-12
    zb = W.to_bf16_bits(z)
    pb = oracle_mod.softmax(zb, T)
    assert np.allclose(pb, sp_softmax(W.bf16_bits_to_f32(zb).astype(np.float64) / T), rtol=1e-12, atol=0)


def test_softmax_masked_entries(oracle_mod):
    z = np.array([-np.inf, 1.0, -np.inf, 1.0], np.float32)
    assert np.allclose(oracle_mod.softmax(z), [0, 0.5, 0, 0.5])


def test_argmax_first_index(oracle_mod):
    rng = np.random.default_rng(21)
    for _ in range(50):
        z = rng.integers(-3, 3, 37).astype(np.float32)
        assert oracle_mod.argmax(z) == int(np.argmax(z))
        zb = W.to_bf16_bits(z)
        assert oracle_mod.argmax(zb) == int(np.argmax(W.bf16_bits_to_f32(zb)))


def test_strict_mode(oracle_mod):
    zt = np.array([[0, 3, 3, 1], [5, 0, 0, 0], [0, 0, 0, 9], [1, 1, 1, 1]], np.float32)
    cu = np.array([0, 3], np.int32)
    us = np.zeros((4, 2), np.float32)
    mode = np.array([1], np.uint8)
    # argmaxes: 1 (tie -> lowest), 0, 3, 0
    r = oracle_mod.spec_verify(zt, None, np.array([1, 0, 2], np.int32), cu, us, 1.0, mode)
    assert r.out_len[0] == 3 and list(r.out_tokens[:3]) == [1, 0, 3]
    r = oracle_mod.spec_verify(zt, None, np.array([1, 0, 3], np.int32), cu, us, 1.0, mode)
    assert r.out_len[0] == 4 and list(r.out_tokens) == [1, 0, 3, 0]
    r = oracle_mod.spec_verify(zt, None, np.array([2, 0, 3], np.int32), cu, us, 1.0, mode)
    assert r.out_len[0] == 1 and r.out_tokens[0] == 1


def test_output_length_invariant(oracle_mod):
    """1 <= out_len[b] <= K_b + 1; accepted prefix equals the drafts; tokens in range."""
    rng = np.random.default_rng(22)
    B, V = 200, 9
    Ks = rng.integers(0, 6, B).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(Ks)]).astype(np.int32)
    R_t = int(cu[-1]) + B
    zt = rng.normal(0, 1.0, (R_t, V)).astype(np.float32)
    zd = rng.normal(0, 1.0, (int(cu[-1]), V)).astype(np.float32)
    toks = rng.integers(0, V, int(cu[-1])).astype(np.int32)
    mode = (rng.random(B) < 0.3).astype(np.uint8)
    for d in (zd, None):
        r = oracle_mod.spec_verify(zt, d, toks, cu, W.uniforms_for(cu, 3), 0.8, mode)
        assert np.all(r.out_len >= 1) and np.all(r.out_len <= Ks + 1)
        for b in range(B):
            n = r.out_len[b]
            out = r.out_tokens[cu[b] + b: cu[b] + b + n]
            assert np.all(out[:-1] == toks[cu[b]:cu[b] + n - 1])
            assert 0 <= out[-1] < V


# --------------------------------------------------------------------------
# N-gram proposer
# --------------------------------------------------------------------------
def test_ngram_printed_cases(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "ngram_examples.json")))
    for c in g["cases"]:
        h = np.array(c["history"], np.int32)
        out, cnt, n = oracle_mod.ngram_propose(h, [h.shape[0]], c["min_n"], c["max_n"], c["max_tokens"])
        assert n[0] == c["n"] and list(out[0, :cnt[0]]) == c["draft"], c


def _ngram_naive(h, min_n, max_n, max_tokens):
    """All matching starts whose continuation is non-empty; the largest wins."""
    L = len(h)
    for n in range(min(max_n, L), min_n - 1, -1):
        tail = h[L - n:]
        cands = [s for s in range(L - n + 1) if h[s:s + n] == tail and s + n < L - n]
        if cands:
            s = max(cands)
            return n, h[s + n:L - n][:max_tokens]
    return 0, []


def test_ngram_bruteforce(oracle_mod):
    rng = np.random.default_rng(23)
    for trial in range(3000):
        L = int(rng.integers(0, 40))
        alpha = int(rng.integers(1, 5))
        h = rng.integers(0, alpha, L).astype(np.int32).tolist()
        min_n = int(rng.integers(1, 4))
        max_n = int(rng.integers(min_n, 7))
        mt = int(rng.integers(0, 6))
        stride = L + int(rng.integers(0, 3))
        hb = np.full((1, max(stride, 1)), -7, np.int32)
        hb[0, :L] = h
        out, cnt, n = oracle_mod.ngram_propose(hb, [L], min_n, max_n, mt)
        en, ed = _ngram_naive(h, min_n, max_n, mt)
        assert n[0] == en and list(out[0, :cnt[0]]) == ed, (h, min_n, max_n, mt)


# --------------------------------------------------------------------------
# Acceptance statistics ("5.2 Draft 模型与无模型方案", §7.1-7.2)
# --------------------------------------------------------------------------
def test_acceptance_metrics_worked_example(oracle_mod):
    import json
    g = json.load(open(os.path.join(GOLDEN, "acceptance_metrics.json")))
    m = oracle_mod.acceptance_metrics(g["cu_draft"], g["out_len"], max_pos=3)
    e = g["expect"]
    for k in ("rounds", "rounds_with_draft", "drafted", "accepted", "committed", "offered", "reached",
              "accepted_at"):
        assert m[k] == e[k], k
    r = oracle_mod.derived_rates(m)
    assert r["draft_acceptance_rate"] == e["draft_acceptance_rate"]
    assert r["mean_acceptance_length"] == e["mean_acceptance_length"]
    assert abs(r["coverage"] - e["coverage"]) < 1e-15
    for got, want in zip(r["conditional"], e["conditional"]):
        assert (want is None and got != got) or got == want
    assert r["through"] == e["through"]


def test_acceptance_metrics_identities(oracle_mod):
    """committed = C + R; fixed gamma (D = gamma R) gives 1 + C/R = 1 + gamma C/D
    (§7.2); the rate through slot i never exceeds the conditional rate, and
    reached[i+1] = accepted_at[i] for rounds that propose slot i+1."""
    rng = np.random.default_rng(3)
    gamma, B = 5, 400
    cu = np.arange(B + 1) * gamma
    lens = rng.integers(1, gamma + 2, size=B)
    m = oracle_mod.acceptance_metrics(cu, lens)
    r = oracle_mod.derived_rates(m)
    assert m["committed"] == m["accepted"] + m["rounds"]
    assert m["drafted"] == gamma * m["rounds"]
    assert abs(r["mean_acceptance_length"] - (1 + gamma * m["accepted"] / m["drafted"])) < 1e-12
    for i in range(gamma - 1):
        assert m["reached"][i + 1] == m["accepted_at"][i]
    for i in range(gamma):
        assert r["through"][i] <= r["conditional"][i] + 1e-15
    # accepted counts: sum over slots of accepted_at equals C
    assert sum(m["accepted_at"]) == m["accepted"]


# --------------------------------------------------------------------------
# Draft-length controller ("投机解码从零实现", §5.2 动态草稿长度策略)
# --------------------------------------------------------------------------
def test_controller_waits_for_ten_rounds_then_steps_to_the_bounds(oracle_mod):
    c = oracle_mod.AdaptiveDraftLength(window=100, min_k=1, max_k=10, target=0.7, initial_k=5)
    ks = [c.update(4, 4) for _ in range(15)]           # every proposal accepted
    assert ks == [5] * 9 + [6, 7, 8, 9, 10, 10]
    c = oracle_mod.AdaptiveDraftLength(window=100, min_k=2, max_k=10, target=0.7, initial_k=5)
    ks = [c.update(4, 0) for _ in range(14)]           # every proposal rejected
    assert ks == [5] * 9 + [4, 3, 2, 2, 2]
    c = oracle_mod.AdaptiveDraftLength(window=100, min_k=1, max_k=10, target=0.7, initial_k=5)
    assert [c.update(10, 7) for _ in range(30)] == [5] * 30   # on target: no move
    c = oracle_mod.AdaptiveDraftLength(window=100, min_k=1, max_k=10, target=0.7, initial_k=5)
    assert [c.update(0, 0) for _ in range(12)] == [5] * 9 + [4, 3, 2]  # no proposal counts as 0


def test_controller_window_forgets_old_rounds(oracle_mod):
    """window 10, target 0.65 (band 0.55..0.75): ten all-accepted rounds, then
    all-rejected ones; after n of those the window mean is (10 - n) / 10."""
    c = oracle_mod.AdaptiveDraftLength(window=10, min_k=1, max_k=10, target=0.65, initial_k=5)
    ks = [c.update(3, 3) for _ in range(10)] + [c.update(3, 0) for _ in range(10)]
    # means 0.9, 0.8 raise; 0.7, 0.6 hold; 0.5 .. 0.0 lower
    assert ks == [5] * 9 + [6] + [7, 8, 8, 8, 7, 6, 5, 4, 3, 2]


# --------------------------------------------------------------------------
# Top-k / top-p filtered verify ("投机解码从零实现" §5.4: top-k and nucleus
# rejection sampling keep the distribution; the same filter on p and q)
# --------------------------------------------------------------------------
LN2_T = 1.0 / np.log(2.0)  # with T = 1/ln 2, exp(z / T) = 2^z exactly for these logits


def test_filters_closed_forms(oracle_mod):
    z = np.array([2, 1, 0, -1, -3], np.float32)  # weights 4, 2, 1, 1/2, 1/8
    w = np.array([4, 2, 1, 0.5, 0.125])
    cases = [  # (top_k, top_p, kept)
        (0, 1.0, 5), (5, 1.0, 5), (2, 1.0, 2), (1, 1.0, 1),
        (0, 0.5, 1),     # 4/7.625 = 0.5246 >= 0.5
        (0, 0.53, 2),    # 0.5246 < 0.53 <= 6/7.625
        (0, 0.90, 3),    # 6/7.625 = 0.787 < 0.90 <= 7/7.625 = 0.918
        (3, 0.90, 3),    # on the top-3 renormalised: 4/7, 6/7 < 0.9 <= 1
        (4, 0.80, 3),    # top-4 total 7.5: 6/7.5 = 0.8 reaches 0.80 exactly? see margin test
    ]
    for k, pp, kept in cases[:-1]:
        p, m = oracle_mod.filtered_softmax(z, LN2_T, k, pp)
        want = np.where(np.arange(5) < kept, w, 0.0)
        want = want / want.sum()
        assert np.allclose(p, want, rtol=0, atol=1e-14), (k, pp, p)
        assert (m == np.inf) == (pp >= 1.0)


def test_filters_keep_tie_groups_whole(oracle_mod):
    p, _ = oracle_mod.filtered_softmax(np.array([1, 1, 1, 0], np.float32), LN2_T, 2, 1.0)
    assert np.allclose(p, [1 / 3, 1 / 3, 1 / 3, 0], atol=1e-15)      # k-th largest is tied
    p, _ = oracle_mod.filtered_softmax(np.array([1, 0, 1, -1], np.float32), LN2_T, 0, 0.3)
    assert np.allclose(p, [0.5, 0, 0.5, 0], atol=1e-15)              # first group already > 0.3
    p, _ = oracle_mod.filtered_softmax(np.array([-np.inf, 3, -np.inf, 2], np.float32), LN2_T, 3, 1.0)
    assert np.allclose(p, [0, 2 / 3, 0, 1 / 3], atol=1e-15)          # -inf never kept in mass


def test_filters_margin_flags_near_equal_boundary(oracle_mod):
    z = np.array([2, 1, 0, -1, -3], np.float32)
    # top-4 mass 7.5; the first two values carry 6/7.5 = 0.8 exactly
    _, m = oracle_mod.filtered_softmax(z, LN2_T, 4, 0.8)
    assert m < 1e-12
    _, m = oracle_mod.filtered_softmax(z, LN2_T, 4, 0.75)
    assert abs(m - 0.05) < 1e-12     # 4/7.5 = 0.5333 < 0.75 <= 0.8


def test_filters_off_is_the_unfiltered_oracle(oracle_mod):
    b = W.gaussian_sampling(seed=41, B=20, K=4, V=300, sigma=2.0, draft_sigma=0.7, T=0.8)
    r0 = oracle_mod.spec_verify(b.target, b.draft, b.draft_tokens, b.cu_draft, b.uniforms, b.temperature)
    r1 = oracle_mod.spec_verify(b.target, b.draft, b.draft_tokens, b.cu_draft, b.uniforms, b.temperature,
                                top_k=300, top_p=1.0)
    assert np.array_equal(r0.out_tokens, r1.out_tokens) and np.array_equal(r0.out_len, r1.out_len)
    assert np.array_equal(r0.out_probs, r1.out_probs, equal_nan=True)


def test_filtered_verify_is_lossless_for_the_filtered_target(oracle_mod):
    """V=16, K=1, top-k 9 then top-p 0.85 on both rows; x̂ ~ q' (the filtered
    draft); over 1e6 rounds the first emitted token follows p' (chi-square)."""
    rng = np.random.default_rng(17)
    V, N, k, pp = 16, 1_000_000, 9, 0.85
    zp = rng.normal(0, 1.5, V).astype(np.float32)
    zq = (zp + rng.normal(0, 1.0, V)).astype(np.float32)
    zb = rng.normal(0, 1.5, V).astype(np.float32)
    p1, _ = oracle_mod.filtered_softmax(zp, 1.0, k, pp)
    q1, _ = oracle_mod.filtered_softmax(zq, 1.0, k, pp)
    cu = np.arange(N + 1, dtype=np.int32)
    x = np.searchsorted(np.cumsum(q1), rng.random(N), side="right").clip(0, V - 1).astype(np.int32)
    target = np.tile(np.stack([zp, zb]), (N, 1))
    draft = np.tile(zq[None], (N, 1))
    r = oracle_mod.spec_verify(target, draft, x, cu, W.uniforms_for(cu, seed=23), 1.0, diagnostics=False,
                               top_k=k, top_p=pp)
    first = r.out_tokens.reshape(N, 2)[:, 0]
    hist = np.bincount(first, minlength=V)
    keep = p1 > 0
    assert hist[~keep].sum() == 0
    chi2 = float(((hist[keep] - N * p1[keep]) ** 2 / (N * p1[keep])).sum())
    dof = int(keep.sum()) - 1
    from scipy.stats import chi2 as chi2_dist
    assert chi2 < chi2_dist.ppf(0.999, dof), (chi2, dof)


def test_select_candidates_worked_example(oracle_mod):
    """Three requests: candidates (2, 5, 5) keep the first 5; (1) keeps it;
    none gives -1."""
    best, best_len = oracle_mod.select_candidates([0, 3, 4, 4], [2, 5, 5, 1], "longest")
    assert best.tolist() == [1, 3, -1] and best_len.tolist() == [5, 1, 0]


def test_select_candidates_uniform_worked_example(oracle_mod):
    """floor(u * n): u = 0.5 of 3 candidates keeps the second, u just below 1
    the last, u = 0 the first; one candidate is always kept; a negative u
    keeps the first."""
    cu, lens = [0, 3, 4, 4, 6], [2, 5, 5, 1, 3, 4]
    best, best_len = oracle_mod.select_candidates(cu, lens, "uniform", [0.5, 0.9, 0.3, 1 - 2 ** -24])
    assert best.tolist() == [1, 3, -1, 5] and best_len.tolist() == [5, 1, 0, 4]
    best, _ = oracle_mod.select_candidates(cu, lens, "uniform", [0.0, 0.0, 0.0, 0.0])
    assert best.tolist() == [0, 3, -1, 4]
    best, _ = oracle_mod.select_candidates(cu, lens, "uniform", [1 - 2 ** -24, -0.5, 0.5, 0.5])
    assert best.tolist() == [2, 3, -1, 5]
    # Each of n candidates is kept for exactly 1/n of the uniform's lattice.
    n = 3
    u = np.arange(0, 2 ** 24, 4099, dtype=np.float64) / 2 ** 24
    picks = [oracle_mod.select_candidates([0, n], [1] * n, "uniform", [x])[0][0] for x in u]
    frac = np.bincount(picks, minlength=n) / len(picks)
    assert np.abs(frac - 1 / n).max() < 2e-3


def _two_candidate_rounds(oracle_mod, N, seed):
    """N requests of two candidates; each candidate proposes one token drawn
    from q (K = 1) and is verified as its own request."""
    rng = np.random.default_rng(seed)
    V, T = 16, 1.0
    zp = rng.normal(0, 1.5, V).astype(np.float32)
    zb = rng.normal(0, 1.5, V).astype(np.float32)
    zq = (zp + rng.normal(0, 1.0, V)).astype(np.float32)
    p = sp_softmax(zp.astype(np.float64))
    q = sp_softmax(zq.astype(np.float64))
    C = 2 * N
    cu = np.arange(C + 1, dtype=np.int32)
    toks = _sample(q, C, rng)
    r = oracle_mod.spec_verify(np.tile(np.stack([zp, zb]), (C, 1)), np.tile(zq[None], (C, 1)), toks, cu,
                               W.uniforms_for(cu, seed=seed + 1), T, diagnostics=False)
    cu_cand = np.arange(0, C + 1, 2, dtype=np.int32)
    return p, r, cu_cand


def test_select_uniform_is_lossless_and_longest_is_not(oracle_mod):
    """Two candidates per request, each drawn from q and verified alone. The
    uniform rule's kept first token follows p (chi-square, 15 dof); the
    longest rule's, which prefers the candidate that was accepted, does not."""
    N = 500_000
    p, r, cu_cand = _two_candidate_rounds(oracle_mod, N, 31)
    first = r.out_tokens.reshape(-1, 2)[:, 0]   # each candidate: target rows (slot 0, bonus)
    u = W.selection_uniforms(N, seed=33)
    for policy, lossless in (("uniform", True), ("longest", False)):
        best, _ = oracle_mod.select_candidates(cu_cand, r.out_len, policy, u)
        hist = np.bincount(first[best], minlength=16)
        chi2 = float(((hist - N * p) ** 2 / (N * p)).sum())
        if lossless:
            assert chi2 < CHI2_15DOF_999, chi2
        else:
            assert chi2 > 50 * CHI2_15DOF_999, chi2


# --------------------------------------------------------------------------
# Suffix proposer ("5.2 Draft 模型与无模型方案", §5.1-5.2)
# --------------------------------------------------------------------------
def test_suffix_prefers_the_frequent_continuation(oracle_mod):
    """The page's case: after a suffix, "return" 20 times and "raise" twice."""
    rng = np.random.default_rng(80)
    S, RET, RAISE = [7, 8, 9], 100, 101
    h = []
    conts = [RET] * 20 + [RAISE] * 2
    rng.shuffle(conts)
    conts[-1] = RAISE  # the most recent occurrence says "raise"
    for t in conts:
        h += list(rng.integers(1000, 2000, size=5)) + S + [t]
    h += S
    out, cnt, n = oracle_mod.suffix_propose(np.array([h], np.int32), [len(h)], 3, 3, 4)
    assert n[0] == 3 and out[0, 0] == RET
    o2, c2, _ = oracle_mod.ngram_propose(np.array([h], np.int32), [len(h)], 3, 3, 4)
    assert o2[0, 0] == RAISE  # the n-gram proposer copies the most recent match


def test_suffix_length_follows_the_agreement(oracle_mod):
    """Four occurrences continue S 100 50, S 100 50, S 100 60, S 100 70: the
    second step has 2 of 4 votes."""
    S = [7, 8, 9]
    h = []
    for tail in ([100, 50], [100, 50], [100, 60], [100, 70]):
        h += [300, 301] + S + tail
    h += S
    H = np.array([h], np.int32)
    out, cnt, _ = oracle_mod.suffix_propose(H, [len(h)], 3, 3, 5, min_share=0.5)
    assert out[0, :2].tolist() == [100, 50]       # 2/4 >= 0.5 goes on
    out, cnt, _ = oracle_mod.suffix_propose(H, [len(h)], 3, 3, 5, min_share=0.6)
    assert cnt[0] == 1 and out[0, 0] == 100        # 2/4 < 0.6 stops
    # ties: 60 and 70 once each after 100 -> among [100, 60] / [100, 70] the most recent
    h2 = []
    for tail in ([100, 60], [100, 70]):
        h2 += [300, 301] + S + tail
    h2 += S
    out, cnt, _ = oracle_mod.suffix_propose(np.array([h2], np.int32), [len(h2)], 3, 3, 5, min_share=0.5)
    assert out[0, :2].tolist() == [100, 70]


def test_suffix_with_one_occurrence_is_the_ngram_proposer(oracle_mod):
    """max_occ = 1 and min_share = 0: only the most recent match votes, so the
    proposal is the n-gram proposer's (pinned to the page's printed cases)."""
    rng = np.random.default_rng(81)
    B, stride = 200, 60
    hist = rng.integers(0, 4, size=(B, stride)).astype(np.int32)
    hl = rng.integers(0, 61, size=B).astype(np.int32)
    for mn, mx, mt in [(1, 3, 5), (2, 4, 2), (3, 3, 6)]:
        a = oracle_mod.suffix_propose(hist, hl, mn, mx, mt, min_share=0.0, max_occ=1)
        g = oracle_mod.ngram_propose(hist, hl, mn, mx, mt)
        assert np.array_equal(a[1], g[1]) and np.array_equal(a[2], g[2])
        for b in range(B):
            assert np.array_equal(a[0][b, :a[1][b]], g[0][b, :g[1][b]])
