"""spec_verify_noalloc (scratch in the library's fixed device block) against
spec_verify (caller workspace) and the float64 oracle, through the C ABI, on
two calls in a row; its limits (batches beyond the block) and its argument
checks. Named to be collected last; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import parity
from speculative_decoding_verification_27_gb300 import api
from speculative_decoding_verification_27_gb300 import workloads as W

FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation rejects first


def _committed(batch, tok, ln):
    t0 = batch.cu_draft[:-1].astype(np.int64) + np.arange(batch.B)
    return [tok[t0[b]:t0[b] + ln[b]].tolist() for b in range(batch.B)]


def _noalloc_call(lib, db, out_tokens, out_len, out_probs, status):
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    fn = lib.spec_verify_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    dtype = api.SV_BF16 if db.target.dtype == torch.bfloat16 else api.SV_FP32
    return fn(P(db.target), P(db.draft), dtype, int(db.target.shape[1]), int(db.cu_draft.numel() - 1),
              P(db.draft_tokens), P(db.cu_draft), P(db.mode), P(db.uniforms),
              float(db.temperature), P(out_tokens), P(out_len), P(out_probs), P(status),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _batches():
    mixed = W.config5(seed=901, B=48, V=20000)              # bf16, ragged, half greedy
    fp32 = W.gaussian_sampling(seed=902, B=9, K=np.array([0, 1, 3, 5, 2, 0, 4, 6, 1], np.int32),
                               V=4097, sigma=2.0, draft_sigma=0.7, T=0.9)  # scalar-load path
    onehot = W.gaussian_sampling(seed=903, B=20, K=4, V=3000, sigma=1.0, draft_sigma=0.5, T=1.0)
    onehot.draft = None
    return [mixed, fp32, onehot]


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_two_calls_in_a_row(cuda_lib):
    lib = api.load()
    for batch in _batches():
        ora = parity.oracle_verify(batch)
        db = parity.to_device(batch)
        ref_tok, ref_len, ref_pr = api.spec_verify(db.target, db.draft, db.draft_tokens, db.cu_draft,
                                                   db.uniforms, db.temperature, db.mode)
        torch.cuda.synchronize()
        ref_tok, ref_len, ref_pr = ref_tok.cpu().numpy(), ref_len.cpu().numpy(), ref_pr.cpu().numpy()
        R_t = batch.R_t
        out_tokens = torch.full((R_t,), -1, dtype=torch.int32, device="cuda")
        out_len = torch.zeros(batch.B, dtype=torch.int32, device="cuda")
        out_probs = torch.zeros((R_t, 2), dtype=torch.float32, device="cuda")
        status = torch.full((1,), 0x7fffffff, dtype=torch.int32, device="cuda")
        for call in range(2):
            assert _noalloc_call(lib, db, out_tokens, out_len, out_probs, status) == api.SV_OK
            torch.cuda.synchronize()
            assert int(status.item()) == 0, (batch.name, call)
            ln = out_len.cpu().numpy()
            assert np.array_equal(ln, ref_len), (batch.name, call)
            assert _committed(batch, out_tokens.cpu().numpy(), ln) == _committed(batch, ref_tok, ref_len)
            err = float(np.max(np.abs(out_probs.cpu().numpy() - ref_pr)))
            assert err <= parity.PROB_TOL, (batch.name, call, err)
            # And against the oracle, as every other entry point is.
            parity.compare(batch, (out_tokens.cpu().numpy(), ln, out_probs.cpu().numpy()), ora)
            out_len.zero_()
            out_probs.zero_()
            status.fill_(0x7fffffff)


@pytest.mark.gpu
def test_noalloc_reports_data_errors_per_call(cuda_lib):
    lib = api.load()
    b = W.gaussian_sampling(seed=904, B=8, K=3, V=512, sigma=1.0, draft_sigma=0.5, T=1.0)
    db = parity.to_device(b)
    out_tokens = torch.full((b.R_t,), -1, dtype=torch.int32, device="cuda")
    out_len = torch.zeros(b.B, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    good = db.draft_tokens
    db.draft_tokens = good.clone()
    db.draft_tokens[2] = 512  # out of range
    assert _noalloc_call(lib, db, out_tokens, out_len, None, status) == api.SV_OK
    torch.cuda.synchronize()
    assert int(status.item()) & api.SV_DATA_BAD_TOKEN
    # The next call starts clean: the bit does not carry over.
    db.draft_tokens = good
    assert _noalloc_call(lib, db, out_tokens, out_len, None, status) == api.SV_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.gpu
def test_noalloc_flags_rows_beyond_the_block_and_writes_nothing(cuda_lib):
    """B and V pass the host check, but cu_draft[B] + B target rows do not fit
    the block's row records: the kernel sets SV_DATA_BAD_OFFSETS and writes no
    output; the next call that fits is clean. Every array is allocated at the
    full row count, so nothing is out of bounds even if the check failed."""
    lib = api.load()
    B, V = 2, 8
    rows_fit = (api.SV_NOALLOC_SCRATCH_BYTES - 600 * 1024) // 32   # well under the block's row records
    K = np.array([70000, 70000], np.int32)                          # R_t = 140002 rows, 4.5 MB of records
    assert int(K.sum()) + B > api.SV_NOALLOC_SCRATCH_BYTES // 32 > rows_fit
    big = W.gaussian_sampling(seed=905, B=B, K=K, V=V, sigma=1.0, draft_sigma=0.5, T=1.0)
    db = parity.to_device(big)
    out_tokens = torch.full((big.R_t,), -7, dtype=torch.int32, device="cuda")
    out_len = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    out_probs = torch.full((big.R_t, 2), -7.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc_call(lib, db, out_tokens, out_len, out_probs, status) == api.SV_OK
    torch.cuda.synchronize()
    assert int(status.item()) & api.SV_DATA_BAD_OFFSETS
    assert bool((out_len == -7).all()) and bool((out_tokens == -7).all()) and bool((out_probs == -7.0).all())
    small = W.gaussian_sampling(seed=906, B=B, K=np.array([3, 5], np.int32), V=V, sigma=1.0,
                                draft_sigma=0.5, T=1.0)
    ds = parity.to_device(small)
    assert _noalloc_call(lib, ds, out_tokens, out_len, out_probs, status) == api.SV_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    parity.compare(small, (out_tokens.cpu().numpy()[:small.R_t], out_len.cpu().numpy(),
                           out_probs.cpu().numpy()[:small.R_t]), parity.oracle_verify(small))


def test_noalloc_rejects_batches_beyond_the_block_on_the_host():
    from speculative_decoding_verification_27_gb300 import build
    build.build_library()
    lib = api.load()
    fn = lib.spec_verify_noalloc
    fn.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int, ctypes.c_int32, ctypes.c_int32] + \
        [ctypes.c_void_p] * 4 + [ctypes.c_float] + [ctypes.c_void_p] * 5
    fn.restype = ctypes.c_int
    call = lambda B, V: fn(FAKE, None, api.SV_BF16, V, B, FAKE, FAKE, None, FAKE, 1.0, FAKE, FAKE,
                           None, None, None)
    assert api.spec_verify_workspace_size(4096, 4096 * 8, 151936) > api.SV_NOALLOC_SCRATCH_BYTES
    assert call(4096, 151936) == api.SV_ERR_INVALID_ARG
    assert call(-1, 1000) == api.SV_ERR_INVALID_ARG
    assert call(0, 1000) == api.SV_OK  # empty batch: nothing enqueued


def test_noalloc_checks_arguments_before_any_cuda_call():
    """Bad arguments return SV_ERR_INVALID_ARG without touching CUDA (so a
    rejected call enqueues nothing). Without a GPU, a call with valid
    arguments fails in its first CUDA call instead, which shows that the
    rejected ones never got that far."""
    from speculative_decoding_verification_27_gb300 import build
    build.build_library()
    fn = api._noalloc_fn()
    ALIGNED = ctypes.c_void_p(0x10000)
    ODD = ctypes.c_void_p(0x10002)

    def call(dtype=api.SV_BF16, T=1.0, target=ALIGNED, uniforms=ALIGNED, status=None, V=1000, B=4):
        return fn(target, None, dtype, V, B, ALIGNED, ALIGNED, None, uniforms, T, ALIGNED, ALIGNED,
                  None, status, None)
    assert call(dtype=7) == api.SV_ERR_INVALID_ARG
    assert call(T=0.0) == api.SV_ERR_INVALID_ARG
    assert call(T=float("nan")) == api.SV_ERR_INVALID_ARG
    assert call(T=float("inf")) == api.SV_ERR_INVALID_ARG
    assert call(uniforms=None) == api.SV_ERR_INVALID_ARG
    assert call(target=ctypes.c_void_p(0x10001)) == api.SV_ERR_INVALID_ARG   # bf16 needs 2-byte alignment
    assert call(status=ODD) == api.SV_ERR_INVALID_ARG
    assert call(V=0) == api.SV_ERR_INVALID_ARG
    assert call(V=600000) == api.SV_ERR_INVALID_ARG
    if not torch.cuda.is_available():
        assert call() == api.SV_ERR_CUDA
