"""Frequency-ranked suffix proposer on the GPU against the oracle, bit-exact
("5.2 Draft 模型与无模型方案", §5 Suffix Decoding). Tiny vocabularies give
hundreds of occurrences per tail, so the voter cap, the ordered collection of
occurrences and the vote ties are all exercised."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_27_gb300 import api
from speculative_decoding_verification_27_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(hist, hl, *args, **kw):
    out, cnt, nn = api.suffix_propose(torch.from_numpy(hist).cuda(), torch.from_numpy(hl).cuda(), *args, **kw)
    torch.cuda.synchronize()
    return out.cpu().numpy(), cnt.cpu().numpy(), nn.cpu().numpy()


def _assert_same(g, o):
    g_out, g_cnt, g_n = g
    o_out, o_cnt, o_n = o
    assert np.array_equal(g_cnt, o_cnt)
    assert np.array_equal(g_n, o_n)
    assert np.array_equal(g_out, o_out)  # the oracle pads with -1 as the kernel does


@pytest.mark.parametrize("V,stride,min_n,max_n,max_tokens,share,occ", [
    (2, 300, 1, 4, 6, 0.5, 256),
    (3, 300, 2, 3, 5, 0.6, 7),
    (4, 120, 1, 3, 5, 0.0, 1),
    (4, 120, 1, 3, 8, 1.0, 256),
    (8, 500, 2, 5, 4, 0.34, 64),
])
def test_small_random_histories(cuda_lib, oracle_mod, V, stride, min_n, max_n, max_tokens, share, occ):
    rng = np.random.default_rng(1000 + V * 7 + stride)
    B = 200
    hist = rng.integers(0, V, size=(B, stride)).astype(np.int32)
    hl = rng.integers(0, stride + 1, size=B).astype(np.int32)
    hl[:4] = [0, 1, 2, stride]
    g = _run(hist, hl, min_n, max_n, max_tokens, share, occ)
    o = oracle_mod.suffix_propose(hist, hl, min_n, max_n, max_tokens, min_share=share, max_occ=occ)
    _assert_same(g, o)
    assert (g[1] > 0).any()


def test_voter_cap_on_long_binary_histories(cuda_lib, oracle_mod):
    """V = 2 and L = 3000: a 3-token tail recurs ~370 times, above the cap."""
    rng = np.random.default_rng(1101)
    B, L = 24, 3000
    hist = rng.integers(0, 2, size=(B, L)).astype(np.int32)
    hl = np.full(B, L, np.int32)
    for occ in (256, 100):
        g = _run(hist, hl, 3, 3, 10, 0.4, occ)
        o = oracle_mod.suffix_propose(hist, hl, 3, 3, 10, min_share=0.4, max_occ=occ)
        _assert_same(g, o)


def test_frequent_continuation_beats_the_most_recent(cuda_lib, oracle_mod):
    """The page's case: a suffix followed by one token 20 times, another twice
    (the most recent of them); the n-gram proposer copies the most recent."""
    rng = np.random.default_rng(80)
    S, RET, RAISE = [7, 8, 9], 100, 101
    h, conts = [], [RET] * 20 + [RAISE] * 2
    rng.shuffle(conts)
    conts[-1] = RAISE
    for t in conts:
        h += list(rng.integers(1000, 2000, size=5)) + S + [t]
    h += S
    hist, hl = np.array([h], np.int32), np.array([len(h)], np.int32)
    g = _run(hist, hl, 3, 3, 4)
    assert g[2][0] == 3 and g[0][0, 0] == RET
    _assert_same(g, oracle_mod.suffix_propose(hist, hl, 3, 3, 4))
    ng = api.ngram_propose(torch.from_numpy(hist).cuda(), torch.from_numpy(hl).cuda(), 3, 3, 4)
    assert ng[0].cpu().numpy()[0, 0] == RAISE


def test_one_voter_is_the_ngram_proposer(cuda_lib):
    """max_occ = 1, min_share = 0: the GPU suffix proposer equals the GPU
    n-gram proposer."""
    nb = W.config4_histories(seed=4, B=64, L=4096, ragged=True)
    h = torch.from_numpy(nb.histories).cuda()
    hl = torch.from_numpy(nb.hist_len).cuda()
    a = api.suffix_propose(h, hl, 2, 4, 5, 0.0, 1)
    b = api.ngram_propose(h, hl, 2, 4, 5)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_config4_histories_full(cuda_lib, oracle_mod):
    """The n-gram workload: 128 histories x 8192 tokens, n = 3, 5 tokens."""
    nb = W.config4_histories(seed=4)
    g = _run(nb.histories, nb.hist_len, nb.min_n, nb.max_n, nb.max_tokens)
    o = oracle_mod.suffix_propose(nb.histories, nb.hist_len, nb.min_n, nb.max_n, nb.max_tokens)
    _assert_same(g, o)
    assert 0.15 < (g[1] > 0).mean() < 0.5


@pytest.mark.parametrize("stride", [16384, 16385, 20000])
def test_staging_limit_and_global_reads(cuda_lib, oracle_mod, stride):
    """At the 16384-token staging limit (64 KB of shared memory, opted in)
    and above it, where the history is read from global memory."""
    rng = np.random.default_rng(stride)
    B = 6
    hist = rng.integers(0, 50, size=(B, stride)).astype(np.int32)
    hist[0, 100:140] = hist[0, stride - 40:stride]
    hist[1, 9000:9010] = hist[1, stride - 10:stride]
    hl = np.full(B, stride, np.int32)
    hl[5] = 3
    g = _run(hist, hl, 2, 4, 6, 0.5, 256)
    o = oracle_mod.suffix_propose(hist, hl, 2, 4, 6, min_share=0.5, max_occ=256)
    _assert_same(g, o)


def test_zero_tokens_and_empty_batch(cuda_lib, oracle_mod):
    rng = np.random.default_rng(5)
    hist = rng.integers(0, 3, size=(10, 40)).astype(np.int32)
    hl = np.full(10, 40, np.int32)
    g = _run(hist, hl, 1, 3, 0)
    o = oracle_mod.suffix_propose(hist, hl, 1, 3, 0)
    assert np.array_equal(g[1], o[1]) and np.array_equal(g[2], o[2])
    assert g[0].shape == (10, 0)
    e = torch.empty((0, 16), dtype=torch.int32, device="cuda")
    out, cnt, nn = api.suffix_propose(e, torch.empty(0, dtype=torch.int32, device="cuda"), 1, 3, 5)
    assert out.shape == (0, 5) and cnt.numel() == 0


@pytest.mark.parametrize("stride", [12288, 12289])
def test_ngram_at_its_staging_limit(cuda_lib, oracle_mod, stride):
    """The n-gram proposer at its 12288-token staging limit (48 KB of dynamic
    shared memory plus the static words) and one token above it."""
    rng = np.random.default_rng(stride)
    hist = rng.integers(0, 32000, size=(3, stride)).astype(np.int32)
    hist[0, 500:530] = hist[0, stride - 30:stride]
    hl = np.full(3, stride, np.int32)
    out, cnt, nn = api.ngram_propose(torch.from_numpy(hist).cuda(), torch.from_numpy(hl).cuda(), 2, 4, 6)
    torch.cuda.synchronize()
    o_out, o_cnt, o_n = oracle_mod.ngram_propose(hist, hl, 2, 4, 6)
    assert np.array_equal(cnt.cpu().numpy(), o_cnt) and np.array_equal(nn.cpu().numpy(), o_n)
    assert o_cnt[0] > 0
    g = out.cpu().numpy()
    for b in range(3):
        assert np.array_equal(g[b, :o_cnt[b]], o_out[b, :o_cnt[b]])


def test_suffix_proposals_then_one_hot_verify(cuda_lib, oracle_mod):
    """The proposer's pipeline: suffix proposals packed by sv_pack_drafts and
    verified with one-hot q against fp32 target logits (V = 32000), against
    the oracle's proposals and verify. Repetitive histories (8 distinct
    tokens) make the votes matter."""
    import parity
    rng = np.random.default_rng(1200)
    B, L, mt = 64, 2000, 5
    hist = rng.integers(0, 8, size=(B, L)).astype(np.int32)
    hl = rng.integers(L // 2, L + 1, size=B).astype(np.int32)
    h, dl = torch.from_numpy(hist).cuda(), torch.from_numpy(hl).cuda()
    out, cnt, nn = api.suffix_propose(h, dl, 2, 3, mt, 0.6, 256)
    cu, packed = api.sv_pack_drafts(out, cnt, mt)
    torch.cuda.synchronize()
    o_out, o_cnt, o_n = oracle_mod.suffix_propose(hist, hl, 2, 3, mt, min_share=0.6, max_occ=256)
    assert np.array_equal(cnt.cpu().numpy(), o_cnt) and np.array_equal(nn.cpu().numpy(), o_n)
    assert np.array_equal(out.cpu().numpy(), o_out)
    assert ((o_cnt > 0) & (o_cnt < mt)).sum() > 10  # many proposals end early on split votes
    vb = W.config4_verify(seed=1201, proposals=o_out, counts=o_cnt)
    assert np.array_equal(cu.cpu().numpy(), vb.cu_draft)
    assert np.array_equal(packed.cpu().numpy()[:vb.R_d], vb.draft_tokens)
    db = parity.to_device(vb)
    rep = parity.compare(vb, parity.gpu_verify(db), parity.oracle_verify(vb))
    assert rep.mismatched_requests <= max(1, 1e-4 * rep.rows)
