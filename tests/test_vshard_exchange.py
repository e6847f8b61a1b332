"""The exchanges of the vocabulary-sharded verify (vshard.py) on the CPU:
two gloo ranks gather in rank order (= vocabulary order), take element-wise
maxima and OR the status bits, exactly as one process holding both shards
does. (The kernels between the exchanges need a GPU: tests/test_gpu_vshard.py.)"""
import datetime
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_verification_27_gb300 import vshard


def _parts(rank):
    g = torch.Generator().manual_seed(100 + rank)
    stats = torch.randint(-50, 50, (7, vshard.STAT_WORDS), generator=g, dtype=torch.int32)
    masses = torch.rand(5, generator=g, dtype=torch.float64)
    tok = torch.full((5,), -1, dtype=torch.int32)
    tok[rank::2] = torch.arange(rank, 5, 2, dtype=torch.int32) * 10 + rank
    prob = torch.where(tok[:, None] >= 0, torch.rand(5, 2, generator=g), torch.full((5, 2), -1.0))
    status = torch.tensor([1 << rank], dtype=torch.int32)
    return stats, masses, tok, prob, status


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    try:
        ex = vshard.GroupShards()
        assert ex.count(1) == world and ex.first_index(1) == rank
        stats, masses, tok, prob, status = _parts(rank)
        torch.save({"stats": ex.gather([stats]), "masses": ex.gather([masses]), "tok": ex.max([tok]),
                    "prob": ex.max([prob]), "status": ex.bit_or(status)}, f"{out}.{rank}.pt")
    finally:
        dist.destroy_process_group()


def test_group_exchanges_match_one_process_holding_both_shards(tmp_path):
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    out = str(tmp_path / "ex")
    mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    local = vshard.LocalShards()
    p0, p1 = _parts(0), _parts(1)
    want = {"stats": local.gather([p0[0], p1[0]]), "masses": local.gather([p0[1], p1[1]]),
            "tok": local.max([p0[2], p1[2]]), "prob": local.max([p0[3], p1[3]])}
    for r in range(2):
        got = torch.load(f"{out}.{r}.pt")
        for k, v in want.items():
            assert torch.equal(got[k], v), (r, k)
        assert int(got["status"][0]) == 3  # both ranks' bits
    # The token of every request comes from the one rank that drew it.
    assert want["tok"].tolist() == [0, 11, 20, 31, 40]


def test_split_vocab_covers_the_vocabulary_in_order():
    for V, S in [(151936, 2), (151936, 3), (32000, 4), (7, 4), (5, 8)]:
        b = vshard.split_vocab(V, S)
        assert b[0] == 0 and b[-1] == V and len(b) == S + 1
        assert all(x <= y for x, y in zip(b[:-1], b[1:]))
        assert max(np.diff(b)) - min(np.diff(b)[np.diff(b) > 0]) <= -(-V // S)
