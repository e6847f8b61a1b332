"""Request sharding over ranks, on the CPU: the partition, and two gloo ranks
whose shard outputs (float64 oracle) gathered in rank order equal the
single-process output; plus the benchmark's slowest-rank reduction."""
import json
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

from speculative_decoding_verification_27_gb300 import sharding
from speculative_decoding_verification_27_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _batch():
    b = W.config5(seed=77, B=37, V=700)
    return b


def test_partition_is_contiguous_and_balanced():
    rng = np.random.default_rng(5)
    for world in (1, 2, 3, 4, 8):
        K = rng.integers(0, 9, size=200)
        cu = np.concatenate([[0], np.cumsum(K)]).astype(np.int32)
        greedy = rng.random(200) < 0.5
        bounds = sharding.partition_requests(cu, world, greedy)
        assert bounds[0] == 0 and bounds[-1] == 200 and np.all(np.diff(bounds) >= 0)
        w = sharding.request_weights(cu, greedy, True)
        share = w.sum() / world
        for r in range(world):
            got = w[bounds[r]:bounds[r + 1]].sum()
            assert abs(got - share) <= w.max() + 1e-9


def test_partition_with_fewer_requests_than_ranks():
    cu = np.array([0, 3, 5], np.int32)
    bounds = sharding.partition_requests(cu, 4)
    assert bounds[0] == 0 and bounds[-1] == 2 and np.all(np.diff(bounds) >= 0)


def test_shard_slices_cover_the_packed_layout():
    b = _batch()
    bounds = sharding.partition_requests(b.cu_draft, 3, b.greedy_mask(), b.draft is not None)
    shards = [sharding.shard_of(b.cu_draft, bounds[r], bounds[r + 1]) for r in range(3)]
    assert shards[0].t0 == 0 and shards[-1].t1 == b.R_t
    assert shards[0].d0 == 0 and shards[-1].d1 == b.R_d
    for a, c in zip(shards, shards[1:]):
        assert a.t1 == c.t0 and a.d1 == c.d0 and a.hi == c.lo
    for s in shards:
        lb = sharding.local_batch(b, s)
        assert lb.B == s.B and lb.R_t == s.t1 - s.t0 and lb.R_d == s.d1 - s.d0
        assert np.array_equal(lb.target, b.target[s.t0:s.t1])


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist

    import bench
    import parity
    from speculative_decoding_verification_27_gb300 import sharding as S

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _batch()
        bounds = S.partition_requests(b.cu_draft, world, b.greedy_mask(), b.draft is not None)
        shard = S.shard_of(b.cu_draft, int(bounds[rank]), int(bounds[rank + 1]))
        res = parity.oracle_verify(S.local_batch(b, shard), nthreads=1)
        merged = S.gather_outputs(res.out_tokens, res.out_len, res.out_probs)
        sizes = [None] * world
        dist.all_gather_object(sizes, int(shard.B))
        slowest = bench.max_over_ranks(1.5 + rank, "cpu")
        seeds = [None] * world
        dist.all_gather_object(seeds, bench.rank_seed(3, rank))
        if rank == 0:
            whole = parity.oracle_verify(b, nthreads=1)
            ok = (np.array_equal(merged[0], whole.out_tokens) and np.array_equal(merged[1], whole.out_len)
                  and np.array_equal(merged[2], whole.out_probs))
            with open(out_path, "w") as f:
                json.dump({"equal": bool(ok), "slowest": slowest, "seeds": seeds, "sizes": sizes}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_outputs_equal_whole(oracle_mod, tmp_path):
    out = tmp_path / "result.json"
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, str(out))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("a rank did not finish")
        assert p.exitcode == 0
    r = json.loads(out.read_text())
    assert r["equal"]
    assert r["slowest"] == 2.5
    assert r["seeds"] == [3, 4]
    assert sum(r["sizes"]) == 37 and min(r["sizes"]) > 0
