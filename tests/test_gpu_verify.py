"""GPU parity of spec_verify / spec_verify_greedy against the float64 oracle,
through the C ABI, on the five benchmark configurations (full sizes where the
oracle finishes in seconds) and on edge cases."""
import numpy as np
import pytest
import torch

import parity
from speculative_decoding_verification_27_gb300 import api
from speculative_decoding_verification_27_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(batch, workspace=None, flag_budget=None, draw_flags_in_budget=True):
    db = parity.to_device(batch)
    gpu = parity.gpu_verify(db, workspace)
    ora = parity.oracle_verify(batch)
    return parity.compare(batch, gpu, ora, flag_budget=flag_budget,
                          draw_flags_in_budget=draw_flags_in_budget), gpu, ora


# --------------------------------------------------------------------------
# The five configurations
# --------------------------------------------------------------------------
def test_config1_sampling_1000_rounds(cuda_lib, kernel_path):
    """B=1, K=4, V=32000 fp32, T=1: 1000 rounds of fresh logits, one workspace."""
    ws = api.new_workspace(1, 5, 32000)
    total = parity.ParityReport(0, 0, 0, 0, 0, 0.0, 0)
    for r in range(1000):
        rep, _, _ = _run(W.config1(seed=101, round_index=r), ws)
        for f in ("requests", "rows", "flagged_requests", "flagged_rows", "mismatched_requests",
                  "accept_flagged_rows"):
            setattr(total, f, getattr(total, f) + getattr(rep, f))
        total.max_prob_err = max(total.max_prob_err, rep.max_prob_err)
    print("config1:", total.as_dict())
    # Flat rows over 32000 tokens: draw flags exceed the budget by construction.
    parity.check_budget(total, draw_flags_in_budget=False)
    assert api.sv_check_status(ws) == 0


def test_config2_greedy_full_bit_exact(cuda_lib, kernel_path):
    b = W.config2(seed=102)
    db = parity.to_device(b)
    tok, ln = api.spec_verify_greedy(db.target, db.draft_tokens, db.cu_draft)
    torch.cuda.synchronize()
    ora = parity.oracle_verify(b)
    tok, ln = tok.cpu().numpy(), ln.cpu().numpy()
    assert np.array_equal(ln, ora.out_len)
    t0 = b.cu_draft[:-1] + np.arange(b.B)
    for i in range(b.B):
        n = ln[i]
        assert np.array_equal(tok[t0[i]:t0[i] + n], ora.out_tokens[t0[i]:t0[i] + n])
    # The same through spec_verify with every request in GREEDY mode.
    gpu = parity.gpu_verify(db)
    rep = parity.compare(b, gpu, ora, flag_budget=parity.FLAG_BUDGET)
    print("config2:", rep.as_dict())
    assert rep.mismatched_requests == 0 and rep.flagged_requests == 0


def test_config3_sampling_full(cuda_lib, kernel_path):
    """B=256, K=7, V=151936 bf16, T=0.7 (the benchmark's workload), every request."""
    rep, _, _ = _run(W.config3(seed=103), flag_budget=parity.FLAG_BUDGET)
    print("config3:", rep.as_dict())
    assert rep.mismatched_requests <= 1e-4 * rep.rows


def test_config3_literal_zipf_reading(cuda_lib):
    # The literal reading gives near-flat rows: draw flags exceed the budget by construction.
    rep, _, _ = _run(W.config3(seed=113, B=24, literal_zipf=True), flag_budget=parity.FLAG_BUDGET,
                     draw_flags_in_budget=False)
    assert rep.mismatched_requests <= max(1, 1e-4 * rep.rows)


def test_config4_ngram_then_one_hot_verify(cuda_lib, kernel_path):
    import oracle
    nb = W.config4_histories(seed=104)
    h = torch.from_numpy(nb.histories).cuda()
    hl = torch.from_numpy(nb.hist_len).cuda()
    out, cnt, nn = api.ngram_propose(h, hl, nb.min_n, nb.max_n, nb.max_tokens)
    cu, packed = api.sv_pack_drafts(out, cnt, nb.max_tokens)
    torch.cuda.synchronize()
    o_out, o_cnt, o_n = oracle.ngram_propose(nb.histories, nb.hist_len, nb.min_n, nb.max_n, nb.max_tokens)
    assert np.array_equal(cnt.cpu().numpy(), o_cnt) and np.array_equal(nn.cpu().numpy(), o_n)
    g_out = out.cpu().numpy()
    for b in range(nb.histories.shape[0]):
        assert np.array_equal(g_out[b, :o_cnt[b]], o_out[b, :o_cnt[b]])
        assert np.all(g_out[b, o_cnt[b]:] == -1)
    assert o_cnt.sum() > 0
    vb = W.config4_verify(seed=104, proposals=o_out, counts=o_cnt)
    assert np.array_equal(cu.cpu().numpy(), vb.cu_draft)
    assert np.array_equal(packed.cpu().numpy()[:vb.R_d], vb.draft_tokens)
    rep, _, _ = _run(vb, flag_budget=parity.FLAG_BUDGET, draw_flags_in_budget=False)  # flat rows
    print("config4:", rep.as_dict())
    assert rep.mismatched_requests <= max(1, 1e-4 * rep.rows)


def test_config5_ragged_mixed_full(cuda_lib, kernel_path):
    """B=512, K_b in 1..8, V=256000 bf16, half greedy requests."""
    rep, _, _ = _run(W.config5(seed=105), flag_budget=parity.FLAG_BUDGET, draw_flags_in_budget=False)  # flat rows
    print("config5:", rep.as_dict())
    assert rep.mismatched_requests <= max(1, 1e-4 * rep.rows)


# --------------------------------------------------------------------------
# Edge cases
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("V", [1, 2, 3, 7, 33, 1000, 4097, 8200])
def test_small_and_ragged_vocab(cuda_lib, kernel_path, dtype, V):
    """V not a multiple of the vector width takes the scalar-load path."""
    Ks = np.array([0, 1, 3, 5, 2, 0, 4], np.int32)
    b = W.gaussian_sampling(seed=200 + V, B=Ks.size, K=Ks, V=V, sigma=2.0, draft_sigma=0.7,
                            T=0.9, dtype=dtype)
    b.mode = np.array([0, 1, 0, 0, 1, 0, 0], np.uint8)
    rep, _, _ = _run(b)
    assert rep.mismatched_requests <= 1


@pytest.mark.parametrize("T", [0.3, 1.0, 2.5])
def test_temperatures(cuda_lib, kernel_path, T):
    b = W.gaussian_sampling(seed=300, B=40, K=5, V=5000, sigma=3.0, draft_sigma=1.0, T=T, dtype="bf16")
    rep, _, _ = _run(b)
    assert rep.mismatched_requests <= 1


def test_one_hot_proposals(cuda_lib, kernel_path):
    b = W.gaussian_sampling(seed=301, B=64, K=4, V=3000, sigma=1.0, draft_sigma=0.5, T=1.0)
    b.draft = None
    rep, _, _ = _run(b)
    assert rep.mismatched_requests <= 1


def test_unaligned_rows_take_scalar_path(cuda_lib):
    """Logit base pointer not 16-byte aligned (element aligned only)."""
    b = W.gaussian_sampling(seed=302, B=16, K=3, V=4096, sigma=2.0, draft_sigma=0.5, T=1.0, dtype="bf16")
    db = parity.to_device(b)
    flat = torch.empty(db.target.numel() + 1, dtype=torch.bfloat16, device="cuda")
    flat[1:].copy_(db.target.reshape(-1))
    db.target = flat[1:].view(db.target.shape)
    assert db.target.data_ptr() % 16 != 0
    gpu = parity.gpu_verify(db)
    parity.compare(b, gpu, parity.oracle_verify(b))


def test_masked_logits_and_ties(cuda_lib, kernel_path):
    V = 64
    zt = np.full((6, V), -np.inf, np.float32)
    zt[:, 5] = 1.0
    zt[:, 9] = 1.0   # tie with 5: greedy argmax is 5
    zt[:, 40] = 0.5
    zd = np.full((4, V), -np.inf, np.float32)
    zd[:, 9] = 0.0
    zd[:, 40] = 0.0
    cu = np.array([0, 2, 4], np.int32)
    toks = np.array([9, 40, 5, 9], np.int32)
    for mode in (np.array([0, 1], np.uint8), np.array([1, 0], np.uint8)):
        b = W.VerifyBatch("masked", zt, zd, toks, cu, W.uniforms_for(cu, 7), 1.0, mode)
        rep, gpu, ora = _run(b)
        assert rep.mismatched_requests == 0


def test_empty_batch_is_a_noop(cuda_lib):
    z = torch.zeros((1, 8), device="cuda")
    cu = torch.zeros(1, dtype=torch.int32, device="cuda")
    tok, ln, _ = api.spec_verify(z, None, torch.zeros(1, dtype=torch.int32, device="cuda"), cu,
                                 torch.zeros((1, 2), device="cuda"), 1.0)
    torch.cuda.synchronize()
    assert ln.numel() == 0


def test_rerun_is_bit_identical(cuda_lib, kernel_path):
    b = W.config5(seed=303, B=48, V=20000)
    db = parity.to_device(b)
    a = parity.gpu_verify(db)
    c = parity.gpu_verify(db)
    for x, y in zip(a, c):
        assert np.array_equal(x, y)


def test_data_errors_set_status_and_leave_workspace_usable(cuda_lib, kernel_path):
    b = W.gaussian_sampling(seed=304, B=8, K=3, V=512, sigma=1.0, draft_sigma=0.5, T=1.0)
    ws = api.new_workspace(b.B, b.R_t, b.V)
    db = parity.to_device(b)
    bad = db.draft_tokens.clone()
    bad[2] = 512  # out of range
    api.spec_verify(db.target, db.draft, bad, db.cu_draft, db.uniforms, 1.0, workspace=ws)
    assert api.sv_check_status(ws) & api.SV_DATA_BAD_TOKEN
    cu_bad = db.cu_draft.clone()
    cu_bad[3] = 1  # decreasing offsets
    api.spec_verify(db.target, db.draft, db.draft_tokens, cu_bad, db.uniforms, 1.0, workspace=ws)
    assert api.sv_check_status(ws) & api.SV_DATA_BAD_OFFSETS
    gpu = parity.gpu_verify(db, ws)
    parity.compare(b, gpu, parity.oracle_verify(b))
    assert api.sv_check_status(ws) == 0


# --------------------------------------------------------------------------
# Statistics of the GPU path itself
# --------------------------------------------------------------------------
def test_chi_square_through_the_gpu(cuda_lib, kernel_path):
    """1e6 rounds, V=16, K=1: the first emitted token follows p (lossless)."""
    from scipy.special import softmax
    rng = np.random.default_rng(12)
    V, N = 16, 1_000_000
    zp = rng.normal(0, 1.5, V).astype(np.float32)
    zb = rng.normal(0, 1.5, V).astype(np.float32)
    zq = (zp + rng.normal(0, 1.0, V)).astype(np.float32)
    p = softmax(zp.astype(np.float64))
    q = softmax(zq.astype(np.float64))
    cu = np.arange(N + 1, dtype=np.int32)
    toks = np.searchsorted(np.cumsum(q), rng.random(N), side="right").clip(0, V - 1).astype(np.int32)
    target = torch.from_numpy(np.stack([zp, zb])).cuda().repeat(N, 1)
    draft = torch.from_numpy(zq[None]).cuda().repeat(N, 1)
    tok, ln, _ = api.spec_verify(target, draft, torch.from_numpy(toks).cuda(),
                                 torch.from_numpy(cu).cuda(),
                                 torch.from_numpy(W.uniforms_for(cu, seed=21)).cuda(), 1.0,
                                 want_probs=False)
    first = tok.view(N, 2)[:, 0].cpu().numpy()
    hist = np.bincount(first, minlength=V)
    chi2 = float(((hist - N * p) ** 2 / (N * p)).sum())
    assert chi2 < 37.70, chi2
    alpha = np.minimum(p, q).sum()
    acc = (ln.cpu().numpy() == 2).mean()
    assert abs(acc - alpha) < 5 * np.sqrt(alpha * (1 - alpha) / N)


# --------------------------------------------------------------------------
# n-gram proposer edge cases
# --------------------------------------------------------------------------
@pytest.mark.parametrize("min_n,max_n,max_tokens", [(1, 1, 4), (1, 3, 5), (2, 4, 1), (3, 3, 0), (2, 6, 9)])
def test_ngram_small_random_histories_bit_exact(cuda_lib, min_n, max_n, max_tokens):
    """Tiny vocabulary (many matches), lengths 0..64 in rows of stride 80."""
    import oracle
    rng = np.random.default_rng(1000 + 10 * min_n + max_n)
    B, stride = 300, 80
    hist = rng.integers(0, 4, size=(B, stride)).astype(np.int32)
    hl = rng.integers(0, 65, size=B).astype(np.int32)
    hl[:4] = [0, 1, 2, 64]
    out, cnt, nn = api.ngram_propose(torch.from_numpy(hist).cuda(), torch.from_numpy(hl).cuda(),
                                     min_n, max_n, max_tokens)
    torch.cuda.synchronize()
    o_out, o_cnt, o_n = oracle.ngram_propose(hist, hl, min_n, max_n, max_tokens)
    assert np.array_equal(cnt.cpu().numpy(), o_cnt)
    assert np.array_equal(nn.cpu().numpy(), o_n)
    g = out.cpu().numpy()
    for b in range(B):
        assert np.array_equal(g[b, :o_cnt[b]], o_out[b, :o_cnt[b]])
        assert np.all(g[b, o_cnt[b]:] == -1)


def test_ngram_long_history_read_from_global(cuda_lib):
    """Histories longer than the shared-memory staging limit (12288 tokens)."""
    import oracle
    rng = np.random.default_rng(77)
    B, L = 6, 20000
    hist = rng.integers(0, 32000, size=(B, L)).astype(np.int32)
    hist[0, 100:140] = hist[0, L - 40:L]      # early copy of the tail
    hist[1, 15000:15010] = hist[1, L - 10:L]  # late copy
    hl = np.full(B, L, np.int32)
    hl[5] = 3
    out, cnt, nn = api.ngram_propose(torch.from_numpy(hist).cuda(), torch.from_numpy(hl).cuda(), 2, 4, 6)
    torch.cuda.synchronize()
    o_out, o_cnt, o_n = oracle.ngram_propose(hist, hl, 2, 4, 6)
    assert np.array_equal(cnt.cpu().numpy(), o_cnt) and np.array_equal(nn.cpu().numpy(), o_n)
    assert o_cnt[0] > 0 and o_cnt[1] > 0
    g = out.cpu().numpy()
    for b in range(B):
        assert np.array_equal(g[b, :o_cnt[b]], o_out[b, :o_cnt[b]])


# --------------------------------------------------------------------------
# The binding's default workspace
# --------------------------------------------------------------------------
def test_default_workspace_is_reused_without_clearing(cuda_lib):
    """Calls that pass no workspace share one cached block per stream: after
    the first call of a layout, calls allocate nothing and clear nothing; a
    new layout clears the block once; results stay equal to the oracle's."""
    a = W.gaussian_sampling(seed=320, B=24, K=4, V=5000, sigma=2.0, draft_sigma=0.7, T=0.9, dtype="bf16")
    c = W.gaussian_sampling(seed=321, B=40, K=3, V=5000, sigma=2.0, draft_sigma=0.7, T=0.9, dtype="bf16")
    da, dc = parity.to_device(a), parity.to_device(c)
    out = (torch.empty(max(a.R_t, c.R_t), dtype=torch.int32, device="cuda"),
           torch.empty(max(a.B, c.B), dtype=torch.int32, device="cuda"),
           torch.empty((max(a.R_t, c.R_t), 2), dtype=torch.float32, device="cuda"))

    def call(b, db):
        n = b.R_t
        api.spec_verify(db.target, db.draft, db.draft_tokens, db.cu_draft, db.uniforms, db.temperature,
                        db.mode, out_tokens=out[0][:n], out_len=out[1][:b.B], out_probs=out[2][:n])
        torch.cuda.synchronize()
        parity.compare(b, (out[0][:n].cpu().numpy(), out[1][:b.B].cpu().numpy(), out[2][:n].cpu().numpy()),
                       parity.oracle_verify(b))

    call(a, da)   # first call of this layout: the block is made and cleared
    clears, mem = api.default_workspace_clears, torch.cuda.memory_allocated()
    ws = api.default_workspace(0, "cuda", layout=("verify", a.B, a.V))
    for _ in range(3):
        call(a, da)
    assert api.default_workspace_clears == clears and torch.cuda.memory_allocated() == mem
    call(c, dc)   # another B: cleared once, then reused
    call(c, dc)
    assert api.default_workspace_clears == clears + 1
    call(a, da)
    assert api.default_workspace_clears == clears + 2
    assert api.default_workspace(0, "cuda", layout=("verify", a.B, a.V)).data_ptr() == ws.data_ptr()
    assert api.sv_check_status(ws) == 0


# --------------------------------------------------------------------------
# Kernel choice
# --------------------------------------------------------------------------
def test_cluster_threshold_default_and_dispatch(cuda_lib):
    """spec_verify takes the one-cluster-per-row kernel when the workspace
    holds at most SV_CLUSTER_ROWS_DEFAULT = 64 target rows; both kernels give
    the oracle's commits on a batch right at the threshold and past it."""
    assert api.sv_set_cluster_rows(-1) == 64
    for B in (16, 17):  # K = 3: 64 and 68 target rows
        b = W.gaussian_sampling(seed=700 + B, B=B, K=3, V=4096, sigma=2.0, draft_sigma=0.7, T=0.9, dtype="bf16")
        rep, _, _ = _run(b)
        assert rep.mismatched_requests <= 1


def test_cluster_rows_beyond_the_workspace_are_reported(cuda_lib):
    """Offsets that claim more rows than the workspace holds: the cluster
    kernel sets SV_DATA_BAD_OFFSETS and writes no output."""
    prev = api.sv_set_cluster_rows(1 << 20)
    try:
        b = W.gaussian_sampling(seed=720, B=4, K=3, V=512, sigma=1.0, draft_sigma=0.5, T=1.0)
        db = parity.to_device(b)
        ws = api.new_workspace(b.B, b.R_t, b.V)
        cu_bad = db.cu_draft.clone()
        cu_bad[-1] += 3  # R_t beyond the workspace (and beyond the caller's rows: nothing may read them)
        ln = torch.full((b.B,), -7, dtype=torch.int32, device="cuda")
        api.spec_verify(db.target, db.draft, db.draft_tokens, cu_bad, db.uniforms, 1.0, out_len=ln, workspace=ws)
        torch.cuda.synchronize()
        assert api.sv_check_status(ws) & api.SV_DATA_BAD_OFFSETS
        assert (ln.cpu().numpy() == -7).all()
        gpu = parity.gpu_verify(db, ws)
        parity.compare(b, gpu, parity.oracle_verify(b))
        assert api.sv_check_status(ws) == 0
    finally:
        api.sv_set_cluster_rows(prev)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_greedy_entry_ties_empty_rows_and_two_lookup_rounds(cuda_lib, dtype):
    """spec_verify_greedy on 16-byte vector rows runs the one-CTA-per-row
    greedy kernel: logits on a coarse grid (ties: the lowest index wins),
    rows of -inf only (index 0), requests with K = 0, an out-of-range token,
    and B = 300 > 256 requests (two rounds of the request lookup)."""
    rng = np.random.default_rng(730)
    B, V = 300, 1024
    Ks = rng.integers(0, 6, B).astype(np.int32)
    cu = np.concatenate([[0], np.cumsum(Ks)]).astype(np.int32)
    R_t = int(cu[-1]) + B
    zt = (np.round(rng.normal(0, 1.5, (R_t, V)) * 2) / 2).astype(np.float32)
    zt[rng.choice(R_t, 7, replace=False)] = -np.inf
    am = np.argmax(zt, axis=1)  # first index of the maximum (0 for -inf rows)
    toks = np.empty(int(cu[-1]), np.int32)
    for b_ in range(B):
        for i in range(Ks[b_]):
            row = cu[b_] + b_ + i
            toks[cu[b_] + i] = am[row] if rng.random() < 0.75 else rng.integers(V)
    bad = toks.size // 2
    b_bad = int(np.searchsorted(cu, bad, side="right") - 1)
    toks_ora = toks.copy()  # the oracle refuses an out-of-range token: any mismatch stands in
    toks_ora[bad] = (am[bad + b_bad] + 1) % V
    toks[bad] = V + 5  # out of range: a mismatch, and a status bit
    mode = np.full(B, 1, np.uint8)
    zstore = W.to_bf16_bits(zt) if dtype == "bf16" else zt
    b = W.VerifyBatch("greedy_edges", zstore, None, toks, cu, W.uniforms_for(cu, 11), 1.0, mode)
    db = parity.to_device(b)
    ws = api.new_workspace(b.B, b.R_t, b.V)
    tok, ln = api.spec_verify_greedy(db.target, db.draft_tokens, db.cu_draft, workspace=ws)
    torch.cuda.synchronize()
    assert api.sv_check_status(ws) == api.SV_DATA_BAD_TOKEN
    ora = parity.oracle_verify(W.VerifyBatch("greedy_edges", zstore, None, toks_ora, cu, b.uniforms, 1.0, mode))
    tok, ln = tok.cpu().numpy(), ln.cpu().numpy()
    assert np.array_equal(ln, ora.out_len)
    t0 = b.cu_draft[:-1] + np.arange(b.B)
    for i in range(b.B):
        n = ln[i]
        want = ora.out_tokens[t0[i]:t0[i] + n].copy()
        if cu[i] <= bad < cu[i + 1] and bad - cu[i] < n - 1:
            want[bad - cu[i]] = V + 5  # not reached: the bad slot rejects, so it is never committed
        assert np.array_equal(tok[t0[i]:t0[i] + n], want), i
    tok2, ln2 = api.spec_verify_greedy(db.target, db.draft_tokens, db.cu_draft, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(ln2.cpu(), torch.from_numpy(ln)) and api.sv_check_status(ws) == api.SV_DATA_BAD_TOKEN


# --------------------------------------------------------------------------
# The one-CTA-per-row kernel for one-hot batches
# --------------------------------------------------------------------------
@pytest.fixture
def onehot_kernel(cuda_lib):
    """Routes one-hot batches of short rows to the one-CTA-per-row kernel
    (no cluster kernel); restores the thresholds afterwards."""
    prev = api.sv_set_cluster_rows(0)
    prev_oh = api.sv_set_onehot_row_bytes(api.SV_ONEHOT_ROW_BYTES_DEFAULT)
    yield
    api.sv_set_cluster_rows(prev)
    api.sv_set_onehot_row_bytes(prev_oh)


@pytest.mark.parametrize("dtype,V", [("fp32", 3000), ("fp32", 32000), ("bf16", 8200), ("bf16", 65536)])
def test_one_hot_kernel_ragged_mixed(onehot_kernel, dtype, V):
    """Ragged K (0, 1, 31 and beyond 31, whose rows count their progress
    instead of tracking per-slot bits), half the requests greedy, one-hot
    proposals: every output equals the oracle's."""
    Ks = [0, 1, 3, 31, 32, 40, 7, 2, 5, 0, 4, 6]
    b = W.gaussian_sampling(seed=310 + V, B=len(Ks), K=Ks, V=V, sigma=2.0, draft_sigma=0.5, T=0.8, dtype=dtype)
    b.draft = None
    b.mode = np.array([0, 1] * (len(Ks) // 2), np.uint8)
    rep, _, _ = _run(b)
    assert rep.mismatched_requests == 0, rep.as_dict()


def test_one_hot_kernel_config4(onehot_kernel):
    """Config 4's verify (n-gram proposals, fp32 V=32000) on the one-hot
    kernel, the path spec_verify takes for it by default."""
    import oracle
    nb = W.config4_histories(seed=104)
    o_out, o_cnt, _ = oracle.ngram_propose(nb.histories, nb.hist_len, nb.min_n, nb.max_n, nb.max_tokens)
    vb = W.config4_verify(seed=104, proposals=o_out, counts=o_cnt)
    rep, _, _ = _run(vb, flag_budget=parity.FLAG_BUDGET, draw_flags_in_budget=False)  # flat rows
    assert rep.mismatched_requests <= max(1, 1e-4 * rep.rows)


def test_one_hot_kernel_data_errors_and_rerun(onehot_kernel):
    """A token out of range and decreasing offsets set their status bits;
    the workspace stays usable and a rerun is bit-identical."""
    b = W.gaussian_sampling(seed=320, B=8, K=3, V=512, sigma=1.0, draft_sigma=0.5, T=1.0)
    b.draft = None
    ws = api.new_workspace(b.B, b.R_t, b.V)
    db = parity.to_device(b)
    bad = db.draft_tokens.clone()
    bad[2] = 512
    api.spec_verify(db.target, None, bad, db.cu_draft, db.uniforms, 1.0, workspace=ws)
    assert api.sv_check_status(ws) & api.SV_DATA_BAD_TOKEN
    cu_bad = db.cu_draft.clone()
    cu_bad[3] = 1
    api.spec_verify(db.target, None, db.draft_tokens, cu_bad, db.uniforms, 1.0, workspace=ws)
    assert api.sv_check_status(ws) & api.SV_DATA_BAD_OFFSETS
    g1 = parity.gpu_verify(db, ws)
    g2 = parity.gpu_verify(db, ws)
    rep = parity.compare(b, g1, parity.oracle_verify(b))
    assert rep.mismatched_requests == 0, rep.as_dict()
    assert np.array_equal(g1[1], g2[1]) and np.array_equal(g1[2], g2[2])
    t0 = b.cu_draft[:-1] + np.arange(b.B)
    for i in range(b.B):
        assert np.array_equal(g1[0][t0[i]:t0[i] + g1[1][i]], g2[0][t0[i]:t0[i] + g2[1][i]])
    assert api.sv_check_status(ws) == 0


def test_one_hot_kernel_chi_square(onehot_kernel):
    """1e6 rounds, V=16, K=1, one-hot proposals drawn from some q: accepting
    x̂ with probability p(x̂) and otherwise drawing from p without x̂ emits a
    first token that follows p, and accepts with probability sum q p."""
    from scipy.special import softmax
    rng = np.random.default_rng(13)
    V, N = 16, 1_000_000
    zp = rng.normal(0, 1.5, V).astype(np.float32)
    zb = rng.normal(0, 1.5, V).astype(np.float32)
    p = softmax(zp.astype(np.float64))
    q = softmax(rng.normal(0, 1.0, V))
    cu = np.arange(N + 1, dtype=np.int32)
    toks = np.searchsorted(np.cumsum(q), rng.random(N), side="right").clip(0, V - 1).astype(np.int32)
    target = torch.from_numpy(np.stack([zp, zb])).cuda().repeat(N, 1)
    tok, ln, _ = api.spec_verify(target, None, torch.from_numpy(toks).cuda(), torch.from_numpy(cu).cuda(),
                                 torch.from_numpy(W.uniforms_for(cu, seed=22)).cuda(), 1.0, want_probs=False)
    first = tok.view(N, 2)[:, 0].cpu().numpy()
    hist = np.bincount(first, minlength=V)
    chi2 = float(((hist - N * p) ** 2 / (N * p)).sum())
    assert chi2 < 37.70, chi2
    alpha = float((q * p).sum())
    acc = (ln.cpu().numpy() == 2).mean()
    assert abs(acc - alpha) < 5 * np.sqrt(alpha * (1 - alpha) / N)
