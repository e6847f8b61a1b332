"""Vocabulary-sharded verify-and-commit on the GPU against the float64 oracle
on the whole vocabulary, through the C ABI (the sv_vshard_* kernels and the
exchanges of vshard.py).

All shards in one process: the exchanges stack and take maxima of the
shards' parts. Two processes, one shard each, on the same GPU with a gloo
group: the kernels never wait on one another (every exchange goes through
the host), so the two ranks need not run at the same time."""
import os

import numpy as np
import pytest
import torch

import parity
from speculative_decoding_verification_27_gb300 import api, vshard
from speculative_decoding_verification_27_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _shards(db, bounds):
    return [vshard.Shard(db.target[:, a:b].contiguous(),
                         None if db.draft is None else db.draft[:, a:b].contiguous(), a)
            for a, b in zip(bounds[:-1], bounds[1:])]


def _run(batch, bounds, flag_budget=None, draw_flags_in_budget=True):
    db = parity.to_device(batch)
    out_probs = torch.empty((batch.R_t, 2), dtype=torch.float32, device="cuda")
    tok, ln, pr, status = vshard.spec_verify_vsharded(
        _shards(db, bounds), batch.V, db.draft_tokens, db.cu_draft, db.uniforms, db.temperature, db.mode,
        out_probs=out_probs)
    torch.cuda.synchronize()
    assert int(status.item()) & ~api.SV_DATA_DEGENERATE_RESIDUAL == 0, int(status.item())
    return parity.compare(batch, (tok.cpu().numpy(), ln.cpu().numpy(), pr.cpu().numpy()),
                          parity.oracle_verify(batch), flag_budget=flag_budget,
                          draw_flags_in_budget=draw_flags_in_budget)


@pytest.mark.parametrize("S", [2, 3, 4])
def test_vsharded_peaked_bf16_even_split(cuda_lib, S):
    """The benchmark's row shape (V=151936 bf16, T=0.7, peaked rows), 32
    requests, split evenly over S shards."""
    b = W.config3(seed=600 + S, B=32)
    rep = _run(b, vshard.split_vocab(b.V, S), flag_budget=parity.FLAG_BUDGET)
    print(S, rep.as_dict())


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("bounds", [[0, 1000, 1001, 4097], [0, 7, 2050, 4097], [0, 4097]])
def test_vsharded_uneven_slices_mixed_modes(cuda_lib, dtype, bounds):
    """Uneven slices (one of a single token, widths not a multiple of the
    vector width: the scalar-load path), ragged K, greedy and sampled
    requests together."""
    Ks = np.array([0, 1, 3, 5, 2, 0, 4, 6, 1, 2], np.int32)
    b = W.gaussian_sampling(seed=610 + len(bounds), B=Ks.size, K=Ks, V=4097, sigma=2.0, draft_sigma=0.7, T=0.9,
                            dtype=dtype)
    b.mode = np.array([0, 1, 0, 0, 1, 0, 0, 1, 0, 0], np.uint8)
    rep = _run(b, bounds)
    assert rep.mismatched_requests <= 1


def test_vsharded_one_hot_proposals(cuda_lib):
    """One-hot q (draft NULL): the residual is p without x̂ in the shard that
    holds x̂."""
    b = W.gaussian_sampling(seed=620, B=64, K=4, V=32000, sigma=2.0, draft_sigma=0.5, T=1.0)
    b.draft = None
    rep = _run(b, vshard.split_vocab(b.V, 4), flag_budget=parity.FLAG_BUDGET, draw_flags_in_budget=False)
    print(rep.as_dict())


def test_vsharded_ragged_mixed_config5_shape(cuda_lib):
    """Config 5's shape (V=256000 bf16, K_b in 1..8, half greedy), 64 requests, 2 shards."""
    b = W.config5(seed=630, B=64)
    rep = _run(b, vshard.split_vocab(b.V, 2), flag_budget=parity.FLAG_BUDGET, draw_flags_in_budget=False)
    print(rep.as_dict())


def test_vsharded_equals_the_one_launch_kernel(cuda_lib):
    """Same batch through spec_verify and through 3 shards: identical commits
    (no request of this batch is flagged) and probabilities within 1e-6."""
    b = W.config3(seed=640, B=24)
    db = parity.to_device(b)
    tok1, ln1, pr1 = api.spec_verify(db.target, db.draft, db.draft_tokens, db.cu_draft, db.uniforms,
                                     db.temperature, db.mode)
    out_probs = torch.empty_like(pr1)
    tok2, ln2, pr2, _ = vshard.spec_verify_vsharded(_shards(db, vshard.split_vocab(b.V, 3)), b.V, db.draft_tokens,
                                                    db.cu_draft, db.uniforms, db.temperature, db.mode,
                                                    out_probs=out_probs)
    torch.cuda.synchronize()
    ora = parity.oracle_verify(b)
    assert not ora.flagged_rows().any()
    assert torch.equal(ln1, ln2)
    t0 = b.cu_draft[:-1] + np.arange(b.B)
    a, c, n = tok1.cpu().numpy(), tok2.cpu().numpy(), ln1.cpu().numpy()
    for i in range(b.B):
        assert np.array_equal(a[t0[i]:t0[i] + n[i]], c[t0[i]:t0[i] + n[i]])
    assert float((pr1 - pr2).abs().max()) <= parity.PROB_TOL


def test_vsharded_bad_offsets_are_reported(cuda_lib):
    b = W.gaussian_sampling(seed=650, B=6, K=3, V=512, sigma=1.0, draft_sigma=0.5, T=1.0)
    db = parity.to_device(b)
    cu_bad = db.cu_draft.clone()
    cu_bad[2] = 100  # decreasing afterwards, and past the draft rows
    _, _, _, status = vshard.spec_verify_vsharded(_shards(db, [0, 200, 512]), b.V, db.draft_tokens, cu_bad,
                                                  db.uniforms, 1.0, out_probs=None)
    torch.cuda.synchronize()
    assert int(status.item()) & api.SV_DATA_BAD_OFFSETS


def _rank_main(rank, world, port, seed, result_path):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import datetime
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=120))
    try:
        torch.cuda.set_device(0)
        b = W.config3(seed=seed, B=16)
        db = parity.to_device(b)
        bounds = vshard.split_vocab(b.V, world)
        sh = _shards(db, bounds)[rank]
        out_probs = torch.empty((b.R_t, 2), dtype=torch.float32, device="cuda")
        tok, ln, pr, status = vshard.spec_verify_vsharded(
            [sh], b.V, db.draft_tokens, db.cu_draft, db.uniforms, db.temperature, db.mode,
            exchange=vshard.GroupShards(), out_probs=out_probs)
        torch.cuda.synchronize()
        np.savez(f"{result_path}.{rank}.npz", tok=tok.cpu().numpy(), ln=ln.cpu().numpy(), pr=pr.cpu().numpy(),
                 status=status.cpu().numpy())
    finally:
        dist.destroy_process_group()


def test_vsharded_two_ranks_gloo_one_shard_each(cuda_lib, tmp_path):
    """Two processes, one vocabulary shard each (both on cuda:0), exchanges
    over a gloo group: both ranks end with the oracle's commit."""
    import socket

    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    path = str(tmp_path / "vs")
    mp.start_processes(_rank_main, args=(2, port, 660, path), nprocs=2, join=True, start_method="spawn")
    b = W.config3(seed=660, B=16)
    ora = parity.oracle_verify(b)
    outs = [np.load(f"{path}.{r}.npz") for r in range(2)]
    for o in outs:
        assert int(o["status"][0]) == 0
        parity.compare(b, (o["tok"], o["ln"], o["pr"]), ora, flag_budget=parity.FLAG_BUDGET)
    assert np.array_equal(outs[0]["ln"], outs[1]["ln"])
