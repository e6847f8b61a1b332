"""Acceptance statistics (device kernel) and the draft-length controller (host
code in the library) against the oracle's plain-Python versions."""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_verification_27_gb300 import api, build
from speculative_decoding_verification_27_gb300 import workloads as W

FAKE = ctypes.c_void_p(0x10000)


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return api.load()


@pytest.mark.parametrize("window,min_k,max_k,target", [(100, 1, 10, 0.7), (10, 2, 8, 0.5), (1, 0, 3, 0.9),
                                                        (37, 1, 16, 0.62)])
def test_controller_matches_oracle(lib, oracle_mod, window, min_k, max_k, target):
    rng = np.random.default_rng(window * 7 + max_k)
    c = api.AdaptiveDraftLength(window, min_k, max_k, target, (min_k + max_k) // 2)
    o = oracle_mod.AdaptiveDraftLength(window, min_k, max_k, target, (min_k + max_k) // 2)
    # phases of high, low and mixed acceptance
    for phase in range(6):
        p = [0.95, 0.2, 0.6, 0.0, 1.0, 0.75][phase]
        for _ in range(int(rng.integers(5, 60))):
            k = int(rng.integers(0, 9))
            acc = int(rng.binomial(k, p))
            assert c.update(k, acc) == o.update(k, acc)


def test_controller_rejects_bad_arguments(lib):
    s = api._Adapt()
    E = api.SV_ERR_INVALID_ARG
    assert lib.sv_adapt_init(ctypes.byref(s), 0, 1, 10, ctypes.c_double(0.7), 5) == E       # window
    assert lib.sv_adapt_init(ctypes.byref(s), 2000, 1, 10, ctypes.c_double(0.7), 5) == E    # window
    assert lib.sv_adapt_init(ctypes.byref(s), 10, 5, 4, ctypes.c_double(0.7), 5) == E       # bounds
    assert lib.sv_adapt_init(ctypes.byref(s), 10, 1, 4, ctypes.c_double(0.7), 5) == E       # initial
    assert lib.sv_adapt_init(None, 10, 1, 4, ctypes.c_double(0.7), 2) == E
    assert lib.sv_adapt_init(ctypes.byref(s), 10, 1, 4, ctypes.c_double(0.7), 2) == api.SV_OK
    assert lib.sv_adapt_update(ctypes.byref(s), 3, 4) == E   # more accepted than proposed
    assert lib.sv_adapt_update(ctypes.byref(s), -1, 0) == E


def test_metrics_host_validation(lib):
    fn = lib.sv_accumulate_metrics
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    E = api.SV_ERR_INVALID_ARG
    assert fn(FAKE, FAKE, -1, FAKE, None) == E
    assert fn(FAKE, FAKE, 4, None, None) == E
    assert fn(FAKE, FAKE, 4, ctypes.c_void_p(0x10004), None) == E   # not 8-byte aligned
    assert fn(None, FAKE, 4, FAKE, None) == E
    assert fn(FAKE, FAKE, 0, FAKE, None) == api.SV_OK                  # nothing to add


def _check_same(got: dict, want: dict):
    for k in ("rounds", "rounds_with_draft", "drafted", "accepted", "committed", "offered", "reached",
              "accepted_at"):
        assert got[k] == want[k], k


@pytest.mark.gpu
def test_metrics_kernel_matches_oracle_over_two_calls(cuda_lib, oracle_mod):
    """Counts from the GPU's own verify outputs, accumulated over two calls
    (config-5 style ragged batch, then a batch with K_b up to 40)."""
    import parity
    m = api.new_metrics()
    cus, lens = [], []
    b1 = W.config5(seed=61, B=96, V=3000)
    K2 = np.random.default_rng(62).integers(0, 41, size=20).astype(np.int32)
    b2 = W.gaussian_sampling(seed=63, B=20, K=K2, V=700, sigma=0.3, draft_sigma=0.05, T=1.0)
    for b in (b1, b2):
        db = parity.to_device(b)
        tok, ln, _ = api.spec_verify(db.target, db.draft, db.draft_tokens, db.cu_draft, db.uniforms,
                                     db.temperature, db.mode)
        api.sv_accumulate_metrics(db.cu_draft, ln, m)
        torch.cuda.synchronize()
        cus.append(b.cu_draft)
        lens.append(ln.cpu().numpy())
    want = oracle_mod.acceptance_metrics(cus[0], lens[0])
    w2 = oracle_mod.acceptance_metrics(cus[1], lens[1])
    for k in ("rounds", "rounds_with_draft", "drafted", "accepted", "committed"):
        want[k] += w2[k]
    for k in ("offered", "reached", "accepted_at"):
        want[k] = [a + c for a, c in zip(want[k], w2[k])]
    got = api.metrics_dict(m)
    _check_same(got, want)
    assert got["drafted"] == int(K2.sum()) + int(np.diff(b1.cu_draft).sum())


@pytest.mark.gpu
def test_metrics_kernel_large_batch_and_clamping(cuda_lib, oracle_mod):
    """100k rounds on several CTAs; out-of-range lengths are clamped alike."""
    rng = np.random.default_rng(64)
    B = 100_000
    K = rng.integers(0, 12, size=B).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(K)]).astype(np.int32)
    lens = rng.integers(-1, 14, size=B).astype(np.int32)
    m = api.new_metrics()
    api.sv_accumulate_metrics(torch.from_numpy(cu).cuda(), torch.from_numpy(lens).cuda(), m)
    torch.cuda.synchronize()
    _check_same(api.metrics_dict(m), oracle_mod.acceptance_metrics(cu, lens))


@pytest.mark.gpu
@pytest.mark.parametrize("policy", ["uniform", "longest"])
def test_select_candidates_after_a_flattened_verify(cuda_lib, oracle_mod, policy):
    """Requests with 0..5 candidates, each candidate verified as its own
    request; the kept candidate matches the oracle's rule on the GPU's own
    lengths, and the flattened verify matches the oracle."""
    import parity
    rng = np.random.default_rng(70)
    B = 40
    M = rng.integers(0, 6, size=B)
    cu_cand = np.concatenate([[0], np.cumsum(M)]).astype(np.int32)
    C = int(cu_cand[-1])
    flat = W.gaussian_sampling(seed=71, B=C, K=rng.integers(1, 7, size=C).astype(np.int32), V=5000,
                               sigma=1.0, draft_sigma=0.3, T=1.0, dtype="bf16")
    u = W.selection_uniforms(B, seed=72)
    u[:3] = [0.0, 1 - 2 ** -24, -0.25]  # the ends of the range, and a negative u
    db = parity.to_device(flat)
    tok, ln, pr = api.spec_verify(db.target, db.draft, db.draft_tokens, db.cu_draft, db.uniforms,
                                  db.temperature)
    pol = api.SV_SELECT_UNIFORM if policy == "uniform" else api.SV_SELECT_LONGEST_BIASED
    best, best_len = api.sv_select_candidates(torch.from_numpy(cu_cand).cuda(), ln, pol,
                                              torch.from_numpy(u).cuda() if policy == "uniform" else None)
    torch.cuda.synchronize()
    parity.compare(flat, (tok.cpu().numpy(), ln.cpu().numpy(), pr.cpu().numpy()), parity.oracle_verify(flat))
    want_b, want_l = oracle_mod.select_candidates(cu_cand, ln.cpu().numpy(), policy, u)
    assert np.array_equal(best.cpu().numpy(), want_b) and np.array_equal(best_len.cpu().numpy(), want_l)
    assert (want_b == -1).sum() == (M == 0).sum()


@pytest.mark.gpu
def test_select_candidates_rejects_an_unknown_policy_or_a_missing_uniform(cuda_lib):
    cu = torch.zeros(2, dtype=torch.int32, device="cuda")
    ln = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(api.SpecVerifyError):
        api.sv_select_candidates(cu, ln, 7)
    with pytest.raises(api.SpecVerifyError):
        api.sv_select_candidates(cu, ln, api.SV_SELECT_UNIFORM, None)
