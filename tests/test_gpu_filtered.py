"""GPU parity of spec_verify_filtered (top-k / top-p on target and draft rows)
against the float64 oracle's filtered verify, through the C ABI."""
import numpy as np
import pytest
import torch

import parity
from speculative_decoding_verification_27_gb300 import api
from speculative_decoding_verification_27_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(batch, top_k, top_p, flag_budget=None):
    import oracle
    db = parity.to_device(batch)
    tok, ln, pr = api.spec_verify_filtered(db.target, db.draft, db.draft_tokens, db.cu_draft, db.uniforms,
                                           db.temperature, top_k, top_p, db.mode)
    torch.cuda.synchronize()
    ora = oracle.spec_verify(batch.target, batch.draft, batch.draft_tokens, batch.cu_draft, batch.uniforms,
                             batch.temperature, batch.mode, top_k=top_k, top_p=top_p)
    return parity.compare(batch, (tok.cpu().numpy(), ln.cpu().numpy(), pr.cpu().numpy()), ora,
                          flag_budget=flag_budget)


def _proposals_from_filtered_draft(batch, top_k, top_p, seed):
    """x̂ ~ q', the filtered draft distribution, as a draft model sampling
    under the same filter proposes (the case in which the filtered step is
    lossless). q' comes from the oracle; a proposal outside q' would be
    rejected with certainty and leave an empty residual when p' = q'."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    u = np.random.default_rng(seed).random(batch.R_d)

    def one(j):
        q, _ = oracle.filtered_softmax(batch.draft[j], batch.temperature, top_k, top_p)
        c = np.cumsum(q)
        return min(int(np.searchsorted(c, u[j] * c[-1], side="right")), q.shape[0] - 1)
    with ThreadPoolExecutor(max_workers=oracle.default_threads()) as ex:
        return np.array(list(ex.map(one, range(batch.R_d))), np.int32)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("V", [33, 1000, 4097, 8200])
@pytest.mark.parametrize("top_k,top_p", [(5, 1.0), (0, 0.8), (20, 0.9), (1, 1.0), (0, 0.3)])
def test_filtered_small_vocab(cuda_lib, dtype, V, top_k, top_p):
    Ks = np.array([0, 1, 3, 5, 2, 0, 4, 6], np.int32)
    b = W.gaussian_sampling(seed=500 + V + top_k, B=Ks.size, K=Ks, V=V, sigma=2.0, draft_sigma=0.7,
                            T=0.9, dtype=dtype)
    b.mode = np.array([0, 1, 0, 0, 1, 0, 0, 0], np.uint8)
    rep = _run(b, top_k, top_p)
    assert rep.mismatched_requests <= 1


@pytest.mark.parametrize("top_k,top_p", [(50, 0.9), (0, 0.95), (1000, 1.0)])
def test_filtered_large_vocab_peaked_rows(cuda_lib, top_k, top_p):
    """Rows of the benchmark's shape (V=151936 bf16, T=0.7, peaked rank
    scores), 24 requests."""
    b = W.config3(seed=510 + top_k, B=24)
    rep = _run(b, top_k, top_p)
    print(rep.as_dict())
    assert rep.mismatched_requests <= 1


def test_filtered_config3_full_batch(cuda_lib):
    """The benchmark batch (B=256, K=7, V=151936 bf16, T=0.7, peaked rows)
    under top-k 50 / top-p 0.9, every request, proposals drawn from the
    filtered draft; flagged rows within the 1e-4 budget."""
    b = W.config3(seed=515)
    b.draft_tokens = _proposals_from_filtered_draft(b, 50, 0.9, seed=516)
    rep = _run(b, 50, 0.9, flag_budget=parity.FLAG_BUDGET)
    print("filtered config3:", rep.as_dict())
    assert rep.mismatched_requests <= 1e-4 * rep.rows


def test_filtered_one_hot_and_ties(cuda_lib):
    """One-hot proposals filter the target only; logits on a coarse grid make
    long tie groups at every threshold."""
    rng = np.random.default_rng(520)
    b = W.gaussian_sampling(seed=521, B=40, K=4, V=3000, sigma=1.0, draft_sigma=0.5, T=1.0)
    b.draft = None
    rep = _run(b, 40, 0.85)
    assert rep.mismatched_requests <= 1
    b = W.gaussian_sampling(seed=522, B=40, K=4, V=2048, sigma=2.0, draft_sigma=1.0, T=1.0)
    b.target = (np.round(b.target * 2) / 2).astype(np.float32)   # values on a 0.5 grid
    b.draft = (np.round(b.draft * 2) / 2).astype(np.float32)
    for k, p in [(7, 1.0), (0, 0.6), (30, 0.75)]:
        rep = _run(b, k, p)
        assert rep.mismatched_requests <= 1


def test_filters_off_equal_the_plain_step(cuda_lib):
    b = W.config5(seed=530, B=48, V=20000)
    db = parity.to_device(b)
    a = api.spec_verify(db.target, db.draft, db.draft_tokens, db.cu_draft, db.uniforms, db.temperature, db.mode)
    f = api.spec_verify_filtered(db.target, db.draft, db.draft_tokens, db.cu_draft, db.uniforms,
                                 db.temperature, 0, 1.0, db.mode)
    torch.cuda.synchronize()
    assert torch.equal(a[1], f[1]) and torch.equal(a[2], f[2])
    t0 = b.cu_draft[:-1] + np.arange(b.B)
    ta, tf, ln = a[0].cpu().numpy(), f[0].cpu().numpy(), a[1].cpu().numpy()
    for i in range(b.B):
        assert np.array_equal(ta[t0[i]:t0[i] + ln[i]], tf[t0[i]:t0[i] + ln[i]])


def test_filtered_bad_offsets_stay_in_bounds(cuda_lib):
    """Offsets that claim more rows than the caller holds: the thresholds
    stop at the caller's rows and the step reports the offsets."""
    b = W.gaussian_sampling(seed=540, B=6, K=3, V=512, sigma=1.0, draft_sigma=0.5, T=1.0)
    db = parity.to_device(b)
    cu_bad = db.cu_draft.clone()
    cu_bad[-1] += 50
    ws = torch.zeros(api.spec_verify_filtered_workspace_size(b.B, b.R_t, b.V), dtype=torch.uint8,
                     device="cuda")
    api.spec_verify_filtered(db.target, db.draft, db.draft_tokens, cu_bad, db.uniforms, 1.0, 10, 0.9,
                             workspace=ws)
    torch.cuda.synchronize()
    fb = api.spec_verify_filtered_workspace_size(b.B, b.R_t, b.V) - api.spec_verify_workspace_size(b.B, b.R_t, b.V)
    assert api.sv_check_status(ws[fb:]) & api.SV_DATA_BAD_OFFSETS


def _shaped_rows(shape, R, V, rng):
    """Rows that push the threshold kernel's one-pass collection to its
    edges: rising values pass every chunk's floor (a compaction per chunk),
    falling values pass almost nothing after the first chunk, and constant or
    two-valued rows leave a tie group at the floor that does not fit (the
    passes over the row take over)."""
    x = np.arange(V, dtype=np.float64)
    if shape == "ascending":
        z = np.tile(-6.0 + 12.0 * x / V, (R, 1)) + rng.normal(0, 0.01, (R, V))
    elif shape == "descending":
        z = np.tile(6.0 - 12.0 * x / V, (R, 1)) + rng.normal(0, 0.01, (R, V))
    elif shape == "constant":
        z = np.zeros((R, V))
    else:  # two levels, the high one in the second half
        z = np.where(x[None, :] >= V // 2, 1.0, 0.0) + np.zeros((R, 1))
    return z.astype(np.float32)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("shape", ["ascending", "descending", "constant", "two_levels"])
@pytest.mark.parametrize("top_k,top_p", [(50, 1.0), (256, 0.9), (257, 0.8), (1, 0.5), (0, 0.9), (0, 0.5)])
def test_one_pass_collection_edges(cuda_lib, dtype, shape, top_k, top_p):
    rng = np.random.default_rng(560 + top_k)
    V = 40000
    b = W.gaussian_sampling(seed=561 + top_k, B=6, K=2, V=V, sigma=2.0, draft_sigma=0.5, T=1.0)
    zt = _shaped_rows(shape, b.R_t, V, rng)
    zd = zt[np.concatenate([np.arange(b.cu_draft[i] + i, b.cu_draft[i] + i + 2) for i in range(b.B)])]
    zd = zd + rng.normal(0, 0.3, zd.shape).astype(np.float32)
    if dtype == "bf16":
        b.target, b.draft = W.to_bf16_bits(zt), W.to_bf16_bits(zd)
    else:
        b.target, b.draft = zt, zd.astype(np.float32)
    rep = _run(b, top_k, top_p)
    assert rep.mismatched_requests <= 1


@pytest.mark.parametrize("top_k,top_p", [(50, 0.9), (0, 0.9)])
def test_filtered_rerun_is_bit_identical(cuda_lib, top_k, top_p):
    """The threshold kernel appends candidates in whatever order the atomics
    give, but its counts and fixed-point mass sums are exact, so a repeated
    call returns the same tokens, lengths and probabilities bit for bit (on
    peaked rows, and on flat rows that take the passes over the row)."""
    for b in (W.config3(seed=550, B=16),
              W.gaussian_sampling(seed=551, B=16, K=5, V=60000, sigma=2.0, draft_sigma=0.75, T=1.0,
                                  dtype="bf16")):
        db = parity.to_device(b)
        runs = []
        for _ in range(3):
            tok, ln, pr = api.spec_verify_filtered(db.target, db.draft, db.draft_tokens, db.cu_draft,
                                                   db.uniforms, db.temperature, top_k, top_p, db.mode)
            torch.cuda.synchronize()
            runs.append((tok.clone(), ln.clone(), pr.clone()))
        for r in runs[1:]:
            assert all(torch.equal(x, y) for x, y in zip(runs[0], r))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("top_k,top_p", [(50, 1.0), (128, 0.9), (129, 0.9), (8, 0.6)])
def test_warp_rows_and_fallback_rows_in_one_batch(cuda_lib, dtype, top_k, top_p):
    """Top-k up to 128 goes to the one-warp-per-row kernel first; rows it
    cannot finish (here: rising rows whose values all pass the floor, and
    rows of one value) go to the CTA kernel, which skips the rest. Peaked,
    rising and constant rows alternate in one batch; k = 129 takes the CTA
    kernel alone."""
    rng = np.random.default_rng(570 + top_k)
    V = 40000
    b = W.gaussian_sampling(seed=571 + top_k, B=8, K=3, V=V, sigma=2.0, draft_sigma=0.5, T=1.0)
    R = b.R_t
    x = np.arange(V, dtype=np.float64)
    zt = np.empty((R, V))
    for r in range(R):
        kind = r % 3
        if kind == 0:   # peaked: a random permutation of rank scores
            zt[r, rng.permutation(V)] = -4.4 * np.log(np.arange(1, V + 1)) + rng.normal(0, 1, V)
        elif kind == 1:  # rising: every chunk beats the floor
            zt[r] = -6.0 + 12.0 * x / V + rng.normal(0, 0.01, V)
        else:            # one value: a tie group of the whole row
            zt[r] = 0.5
    zt = zt.astype(np.float32)
    rows_d = np.concatenate([np.arange(b.cu_draft[i] + i, b.cu_draft[i] + i + 3) for i in range(b.B)])
    zd = (zt[rows_d] + rng.normal(0, 0.3, (rows_d.size, V))).astype(np.float32)
    if dtype == "bf16":
        b.target, b.draft = W.to_bf16_bits(zt), W.to_bf16_bits(zd)
    else:
        b.target, b.draft = zt, zd
    rep = _run(b, top_k, top_p)
    assert rep.mismatched_requests <= 1


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_listed_rows_degenerate_residual_and_one_hot(cuda_lib, dtype):
    """Top-k rows the one-warp kernel lists: their draws read the kept list.
    The draft rows equal the target rows and the proposals are tokens of
    no mass under q' (outside the top k), so every request rejects its first
    proposal with certainty and the residual max(0, p' - q') is empty: the
    draw falls back to p' and the status word says so. The same batch with
    one-hot proposals removes x̂ from p' instead."""
    rng = np.random.default_rng(580)
    V, k = 32000, 40
    b = W.gaussian_sampling(seed=581, B=24, K=4, V=V, sigma=2.0, draft_sigma=0.5, T=0.8, dtype=dtype)
    rows_d = np.concatenate([np.arange(b.cu_draft[i] + i, b.cu_draft[i + 1] + i) for i in range(b.B)])
    b.draft = b.target[rows_d].copy()
    zt = W.bf16_bits_to_f32(b.target) if dtype == "bf16" else b.target
    zd = zt[rows_d]
    # Proposals below every row's k-th largest logit: q'(x̂) = 0.
    kth = -np.sort(-zd, axis=1)[:, k - 1]
    prop = np.empty(rows_d.size, np.int32)
    for j in range(rows_d.size):
        cand = np.nonzero(zd[j] < kth[j])[0]
        prop[j] = cand[rng.integers(cand.size)]
    b.draft_tokens = prop
    db = parity.to_device(b)
    nbytes = api.spec_verify_filtered_workspace_size(b.B, b.R_t, b.V)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    tok, ln, pr = api.spec_verify_filtered(db.target, db.draft, db.draft_tokens, db.cu_draft, db.uniforms,
                                           db.temperature, k, 1.0, db.mode, workspace=ws)
    torch.cuda.synchronize()
    fb = nbytes - api.spec_verify_workspace_size(b.B, b.R_t, b.V)
    assert api.sv_check_status(ws[fb:]) == api.SV_DATA_DEGENERATE_RESIDUAL
    assert (ln.cpu().numpy() == 1).all()
    import oracle
    ora = oracle.spec_verify(b.target, b.draft, b.draft_tokens, b.cu_draft, b.uniforms, b.temperature, b.mode,
                             top_k=k, top_p=1.0)
    rep = parity.compare(b, (tok.cpu().numpy(), ln.cpu().numpy(), pr.cpu().numpy()), ora)
    assert rep.mismatched_requests == 0, rep.as_dict()
    b.draft = None
    rep = _run(b, k, 1.0)
    assert rep.mismatched_requests == 0, rep.as_dict()


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("one_hot", [False, True])
def test_filtered_commit_and_verify_share_a_batch(cuda_lib, dtype, one_hot):
    """With the one-warp thresholds, requests whose rows all carry their
    statistics commit in one CTA each; greedy requests and those with more
    than 31 drafts go to the verify kernel, which skips the others. A mixed
    batch, then one the commit takes whole (the verify kernel leaves at
    once), then the mixed one again, all on one workspace: every call
    matches the oracle and the two mixed calls are bit-identical."""
    import oracle
    V, k, p = 8200, 20, 0.9
    Ks = [0, 1, 7, 31, 32, 40, 3, 5, 2, 33, 6, 4]
    mixed = W.gaussian_sampling(seed=590, B=len(Ks), K=Ks, V=V, sigma=2.0, draft_sigma=0.5, T=0.9, dtype=dtype)
    mixed.mode = np.array([0, 0, 1, 0, 0, 0, 1, 0, 0, 0, 0, 1], np.uint8)
    # Same B and R_t (one workspace layout), every request sampled with K <= 31.
    whole = W.gaussian_sampling(seed=591, B=len(Ks), K=[31, 31, 31, 31, 20, 5, 5, 3, 3, 2, 1, 1], V=V,
                                sigma=2.0, draft_sigma=0.5, T=0.9, dtype=dtype)
    assert whole.R_t == mixed.R_t
    if one_hot:
        mixed.draft = whole.draft = None
    ws = torch.zeros(api.spec_verify_filtered_workspace_size(mixed.B, mixed.R_t, V), dtype=torch.uint8,
                     device="cuda")
    outs = []
    for b in (mixed, whole, mixed):
        db = parity.to_device(b)
        tok, ln, pr = api.spec_verify_filtered(db.target, db.draft, db.draft_tokens, db.cu_draft, db.uniforms,
                                               db.temperature, k, p, db.mode, workspace=ws)
        torch.cuda.synchronize()
        ora = oracle.spec_verify(b.target, b.draft, b.draft_tokens, b.cu_draft, b.uniforms, b.temperature,
                                 b.mode, top_k=k, top_p=p)
        rep = parity.compare(b, (tok.cpu().numpy(), ln.cpu().numpy(), pr.cpu().numpy()), ora)
        assert rep.mismatched_requests == 0, rep.as_dict()
        outs.append((tok, ln, pr))
    assert all(torch.equal(x, y) for x, y in zip(outs[0], outs[2]))
