"""Pins of the oracle's decision margins: the numbers that decide which rows
are "flagged", i.e. which rows a GPU result may legitimately differ on.

A row's margin is the smallest distance between one of its random numbers and
the value that decides it:
  * accept test ("Draft Model（草稿模型）" §2 "接受-拒绝准则": accept with
    probability min(1, p/q); "投机解码从零实现" §4.3: q = 0 rejects):
    |u - rho| with rho = min(1, p(x̂)/q(x̂)), rho = 0 when q(x̂) = 0;
  * draw (same page: re-draw from norm(max(0, p - q)); the algorithm box's
    bonus draw from p_{K+1}; "5.2 Draft 模型与无模型方案" §4.3 one-hot q): the
    distance from u' to the nearer edge of the chosen bucket of the
    normalised CDF, min(u' - C_{k-1}/Z, C_k/Z - u').
The tests treat the oracle as a black box. Every expected value is computed
here from scipy's softmax and the uniform actually passed (an exact float32),
on vocabularies of at most 4 where the residual CDF is a closed form. A
dropped normaliser, a wrong sign, the wrong bucket edge, rho without its
min(1, .) or a max where the row takes the min of its margins each fail one
of them.
"""
import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

LAT = 2.0 ** -24  # spacing of the float32 uniforms just below 1
TOL = 1e-12


def _logits(p):
    return np.log(np.asarray(p, np.float64)).astype(np.float32)


def _run(oracle_mod, zt, zd, toks, us, T=1.0):
    toks = np.asarray(toks, np.int32)
    cu = np.array([0, toks.shape[0]], np.int32)
    return oracle_mod.spec_verify(np.asarray(zt, np.float32),
                                  None if zd is None else np.asarray(zd, np.float32),
                                  toks, cu, np.asarray(us, np.float32), T)


def _sm(z, T=1.0):
    return sp_softmax(np.asarray(z, np.float64) / T)


def _f32(x):
    return float(np.float32(x))


def _buckets(r):
    """Edges of the normalised CDF of r: (lower, upper) per token."""
    C = np.cumsum(r)
    Z = C[-1]
    up = C / Z
    lo = np.concatenate([[0.0], up[:-1]])
    return lo, up


def _bucket_mid(r):
    """A u' in the middle of r's widest bucket, and that bucket's half width."""
    lo, up = _buckets(r)
    k = int(np.argmax(up - lo))
    return _f32((lo[k] + up[k]) / 2), (up[k] - lo[k]) / 2


# --------------------------------------------------------------------------
# Accept margin |u - rho|
# --------------------------------------------------------------------------
P3 = [0.5, 0.3, 0.2]
Q3 = [0.2, 0.3, 0.5]   # token 2: rho = 0.4; token 0: p > q, rho = 1


@pytest.mark.parametrize("T", [1.0, 0.7])
@pytest.mark.parametrize("steps", [-700, -3, -1, 0, 1, 2, 5, 900])
def test_accept_margin_is_distance_to_rho(oracle_mod, T, steps):
    zt = np.stack([_logits(P3), _logits([0.2, 0.3, 0.5])])
    zd = _logits(Q3)[None]
    p, q = _sm(zt[0], T), _sm(zd[0], T)
    rho = min(1.0, p[2] / q[2])
    u = _f32(rho + steps * LAT)
    u2, half = _bucket_mid(np.maximum(p - q, 0.0))
    r = _run(oracle_mod, zt, zd, [2], [[u, u2], [0.5, 0.5]], T)
    assert abs(r.rho[0] - rho) < TOL
    accepted = u < rho
    assert (r.out_len[0] == 2) == accepted
    # Row 0's draw (after a rejection) sits mid-bucket, far from its edges,
    # so the row's margin is the accept margin alone.
    assert half > 0.05
    assert abs(r.margin[0] - abs(u - rho)) < TOL, (u, rho, r.margin[0])
    assert bool(r.flagged_rows()[0]) == (abs(u - rho) < 1e-6)


@pytest.mark.parametrize("steps", [1, 2, 40, 5000])
def test_accept_margin_caps_rho_at_one(oracle_mod, steps):
    """p(x̂) > q(x̂): rho = 1, so the margin is 1 - u, not |u - p/q|."""
    zt = np.stack([_logits(P3), _logits([0.25, 0.25, 0.5])])
    zd = _logits(Q3)[None]
    u = _f32(1.0 - steps * LAT)
    r = _run(oracle_mod, zt, zd, [0], [[u, 0.5], [0.5, 0.5]])
    assert r.rho[0] == 1.0 and r.out_len[0] == 2  # always accepted
    assert abs(r.margin[0] - (1.0 - u)) < TOL
    assert bool(r.flagged_rows()[0]) == (1.0 - u < 1e-6)


@pytest.mark.parametrize("steps", [1, 3, 100])
def test_accept_margin_with_zero_draft_probability(oracle_mod, steps):
    """q(x̂) = 0: rho = 0 and every u rejects; the margin is u itself."""
    zt = np.stack([_logits([0.6, 0.4]), _logits([0.5, 0.5])])
    zd = np.array([[0.0, -np.inf]], np.float32)
    u = _f32(steps * LAT)
    r = _run(oracle_mod, zt, zd, [1], [[u, 0.3], [0.5, 0.5]])
    assert r.rho[0] == 0.0 and r.out_len[0] == 1
    # Residual = p where q = 0 (token 1 only): u' = 0.3 lies 0.3 / 0.7 from its edges.
    assert abs(r.margin[0] - u) < TOL


def test_accept_margin_one_hot(oracle_mod):
    """One-hot q: rho = p(x̂)."""
    zt = np.stack([_logits([0.1, 0.6, 0.3]), _logits([0.5, 0.25, 0.25])])
    p = _sm(zt[0])
    r = p.copy()
    r[1] = 0.0
    u2, half = _bucket_mid(r)   # after a rejection: mid of token 2's bucket [0.25, 1]
    assert half > 0.3
    for steps in (-2, 0, 3, 10000):
        u = _f32(p[1] + steps * LAT)
        res = _run(oracle_mod, zt, None, [1], [[u, u2], [0.5, 0.5]])
        assert abs(res.rho[0] - p[1]) < TOL
        assert (res.out_len[0] == 2) == (u < p[1])
        assert abs(res.margin[0] - abs(u - p[1])) < TOL


# --------------------------------------------------------------------------
# Draw margin: distance of u' to the chosen bucket's edges
# --------------------------------------------------------------------------
PR = [0.3, 0.25, 0.25, 0.2]
QR = [0.1, 0.15, 0.2, 0.55]   # r = max(0, p - q) = [0.2, 0.1, 0.05, 0], Z = 0.35


def _residual_case():
    zt = np.stack([_logits(PR), _logits([0.25] * 4)])
    zd = _logits(QR)[None]
    p, q = _sm(zt[0]), _sm(zd[0])
    return zt, zd, np.maximum(p - q, 0.0)


@pytest.mark.parametrize("steps", [-5, -1, 1, 2, 30])
def test_residual_draw_margin_at_inner_edges(oracle_mod, steps):
    zt, zd, r = _residual_case()
    lo, up = _buckets(r)
    u = 0.999  # far above rho = 0.2/0.55: rejected, accept margin ~0.64
    for k in (0, 1):  # the edges between tokens 0|1 and 1|2
        e = up[k]
        u2 = _f32(e + steps * LAT)
        res = _run(oracle_mod, zt, zd, [3], [[u, u2], [0.5, 0.5]])
        assert res.out_len[0] == 1
        want_tok = k if u2 < e else k + 1
        assert res.out_tokens[0] == want_tok
        assert abs(res.margin[0] - abs(u2 - e)) < TOL, (k, steps, res.margin[0], abs(u2 - e))


@pytest.mark.parametrize("steps", [1, 4, 77])
def test_residual_draw_margin_at_outer_edges(oracle_mod, steps):
    """u' near 0 measures from the first bucket's lower edge; u' near 1 from
    the last positive bucket's upper edge (1, after normalising by Z)."""
    zt, zd, r = _residual_case()
    u_low = _f32(steps * LAT)
    res = _run(oracle_mod, zt, zd, [3], [[0.999, u_low], [0.5, 0.5]])
    assert res.out_tokens[0] == 0 and abs(res.margin[0] - u_low) < TOL
    u_high = _f32(1.0 - steps * LAT)
    res = _run(oracle_mod, zt, zd, [3], [[0.999, u_high], [0.5, 0.5]])
    assert res.out_tokens[0] == 2 and abs(res.margin[0] - (1.0 - u_high)) < TOL


def test_residual_draw_margin_mid_bucket_uses_the_nearer_edge(oracle_mod):
    zt, zd, r = _residual_case()
    lo, up = _buckets(r)
    for k in range(3):
        for frac in (0.2, 0.5, 0.9):
            u2 = _f32(lo[k] + frac * (up[k] - lo[k]))
            res = _run(oracle_mod, zt, zd, [3], [[0.999, u2], [0.5, 0.5]])
            assert res.out_tokens[0] == k
            want = min(u2 - lo[k], up[k] - u2)  # the accept margin is ~0.64
            assert abs(res.margin[0] - want) < TOL, (k, frac)


def test_one_hot_draw_margin(oracle_mod):
    """Rejected one-hot proposal: r = p without x̂, Z = 1 - p(x̂)."""
    zt = np.stack([_logits([0.1, 0.6, 0.3]), _logits([0.5, 0.25, 0.25])])
    p = _sm(zt[0])
    r = p.copy()
    r[1] = 0.0
    lo, up = _buckets(r)   # edge between tokens 0 and 2 at 0.1 / 0.4 = 0.25
    for steps in (-3, 1, 8):
        u2 = _f32(up[0] + steps * LAT)
        res = _run(oracle_mod, zt, None, [1], [[0.999, u2], [0.5, 0.5]])
        assert res.out_len[0] == 1 and res.out_tokens[0] == (0 if u2 < up[0] else 2)
        assert abs(res.margin[0] - abs(u2 - up[0])) < TOL


@pytest.mark.parametrize("T", [1.0, 1.6])
def test_bonus_draw_margin(oracle_mod, T):
    """No proposal (K = 0): the draw is from p itself, Z = 1; edges C_k."""
    pb = [0.15, 0.35, 0.3, 0.2]
    zt = _logits(pb)[None]
    p = _sm(zt[0], T)
    lo, up = _buckets(p)
    for k in range(3):
        for steps in (-2, 3):
            u2 = _f32(up[k] + steps * LAT)
            res = _run(oracle_mod, zt, None, [], [[0.5, u2]], T)
            assert res.out_len[0] == 1 and res.out_tokens[0] == (k if u2 < up[k] else k + 1)
            assert abs(res.margin[0] - abs(u2 - up[k])) < TOL
    # The bonus row after K accepted drafts carries the same margin.
    zt2 = np.stack([_logits([0.5, 0.5, 1e-9, 1e-9]), zt[0]])
    u2 = _f32(up[1] + 6 * LAT)
    res = _run(oracle_mod, zt2, zt2[:1], [0], [[0.0, 0.5], [0.5, u2]], T)
    assert res.out_len[0] == 2 and res.out_tokens[1] == 2
    assert abs(res.margin[1] - abs(u2 - up[1])) < TOL
    assert res.margin[0] > 0.1  # u = 0 against rho = 1


def test_row_margin_is_the_smaller_of_its_decisions(oracle_mod):
    """A rejected row holds two decisions; its margin is the smaller one."""
    zt, zd, r = _residual_case()
    lo, up = _buckets(r)
    rho = _sm(zt[0])[3] / _sm(zd[0])[3]
    u = _f32(rho + 3 * LAT)           # accept margin ~1.8e-7 (rejected)
    u2 = _f32(up[0] - 40 * LAT)       # draw margin ~2.4e-6
    res = _run(oracle_mod, zt, zd, [3], [[u, u2], [0.5, 0.5]])
    assert abs(res.margin[0] - (u - rho)) < TOL
    u = _f32(rho + 400 * LAT)         # accept margin ~2.4e-5
    res = _run(oracle_mod, zt, zd, [3], [[u, u2], [0.5, 0.5]])
    assert abs(res.margin[0] - (up[0] - u2)) < TOL


def test_rows_after_the_stop_carry_no_margin(oracle_mod):
    """Only decisions that were taken count: rows after the first rejection
    (never tested, never drawn from) are never flagged."""
    zt = np.stack([_logits(PR)] * 3)
    zd = np.stack([_logits(QR)] * 2)
    rho = _sm(zt[0])[3] / _sm(zd[0])[3]
    res = _run(oracle_mod, zt, zd, [3, 3], [[0.999, 0.5], [_f32(rho), 0.5], [0.5, _f32(0.5)]])
    assert res.out_len[0] == 1
    assert np.isinf(res.margin[1]) and np.isinf(res.margin[2])
    assert not res.flagged_rows()[1:].any()


def test_accept_flags_of_the_parity_report(oracle_mod):
    """parity.accept_flags counts the rows whose accept test was taken within
    1e-6 of rho, and no others (rows after the stop, bonus rows)."""
    import parity
    from speculative_decoding_verification_27_gb300 import workloads as W
    zt = np.stack([_logits(PR)] * 3)
    zd = np.stack([_logits(QR)] * 2)
    rho = _sm(zt[0])[3] / _sm(zd[0])[3]
    cu = np.array([0, 2], np.int32)
    for u0, want in ((_f32(rho - 2 * LAT), [True, False, False]),   # accepted, then row 1 tested
                     (_f32(rho + 2 * LAT), [True, False, False]),   # rejected at row 0
                     (0.999, [False, False, False])):
        us = np.array([[u0, 0.5], [_f32(0.2), 0.5], [0.5, 0.5]], np.float32)
        b = W.VerifyBatch("margins", zt, zd, np.array([3, 3], np.int32), cu, us, 1.0, None)
        o = oracle_mod.spec_verify(zt, zd, b.draft_tokens, cu, us, 1.0)
        assert parity.accept_flags(b, o).tolist() == want
