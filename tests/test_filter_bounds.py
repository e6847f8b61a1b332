"""The floors of the threshold kernel's one-pass collection, checked against
the oracle's filtered softmax ("投机解码从零实现" §5.4 top-k / top-p) on the
CPU. The kernel keeps every logit at or above a floor and selects the row's
threshold among those alone, so each floor must be at most the oracle's
threshold (the smallest kept logit):

  top-k: the k-th largest of the 256 threads' running maxima over the chunks
    seen so far (k of those maxima lie at or above it);
  top-p alone: (R + log2((1 - p) S / V) - 0.05) / c with S the mass seen so
    far relative to 2^R (a logit of mass below (1 - p) S_total / V cannot be
    in the nucleus, since all of them together weigh less than (1 - p)
    S_total, and S only grows).

The chunk layout is the kernel's: thread t holds the 16-byte words
(chunk * 4 + u) * 256 + t, u < 4, of the row."""
import math

import numpy as np
import pytest

from speculative_decoding_verification_27_gb300 import workloads as W

THREADS, WORDS = 256, 4


def _thread_of(V: int, ev: int) -> np.ndarray:
    """(chunk, thread) of every logit under the kernel's layout."""
    j = np.arange(V) // ev                   # 16-byte word
    chunk = j // (WORDS * THREADS)
    thread = j % THREADS
    return chunk, thread


def _kept_min(row, T, k, p, oracle_mod):
    probs, _ = oracle_mod.filtered_softmax(row, T, top_k=k, top_p=p)
    z = W.logits_as_f32(row).astype(np.float64)
    return z[probs > 0].min()


def _rows(seed):
    rng = np.random.default_rng(seed)
    peaked = W.config3(seed=seed, B=2)       # bf16 rank-score rows, V = 151936
    flat = rng.normal(0, 2.0, size=(2, 40000)).astype(np.float32)
    return [(peaked.target[i], 2, 0.7) for i in range(2)] + [(flat[i], 4, 1.0) for i in range(2)]


@pytest.mark.parametrize("k", [1, 50, 256])
def test_top_k_floors_never_exceed_the_threshold(oracle_mod, k):
    for row, bytes_per, T in _rows(300 + k):
        z = W.logits_as_f32(row).astype(np.float64)
        V = z.size
        chunk, thread = _thread_of(V, 16 // bytes_per)
        tau = _kept_min(row, T, k, 1.0, oracle_mod)
        rmax = np.full(THREADS, -np.inf)
        for c in range(int(chunk.max()) + 1):
            sel = chunk == c
            np.maximum.at(rmax, thread[sel], z[sel])
            if c in (0, 1, 3, 7, 15):
                floor = np.sort(rmax)[::-1][k - 1]
                assert floor <= tau
                assert (z >= floor).sum() >= k


@pytest.mark.parametrize("p", [0.5, 0.9, 0.99])
def test_top_p_floors_never_exceed_the_nucleus(oracle_mod, p):
    for row, bytes_per, T in _rows(400 + int(100 * p)):
        z = W.logits_as_f32(row).astype(np.float64)
        V = z.size
        c = math.log2(math.e) / T
        chunk, _ = _thread_of(V, 16 // bytes_per)
        tau = _kept_min(row, T, 0, p, oracle_mod)
        for last in range(int(chunk.max()) + 1):
            seen = z[chunk <= last]
            R = math.ceil(seen.max() * c)
            S = np.exp2(seen * c - R).sum()
            floor = (R + math.log2((1 - p) * S / V) - 0.05) / c
            assert floor <= tau, (last, floor, tau)


@pytest.mark.parametrize("k", [2, 50, 256])
def test_top_k_floor_is_tight_when_the_top_k_sit_in_distinct_threads(oracle_mod, k):
    """The k largest logits placed in k different threads of the first chunk:
    the k-th largest of the threads' maxima is then exactly the row's k-th
    largest logit, the threshold (a floor one place higher would drop it)."""
    rng = np.random.default_rng(500 + k)
    V, ev = 40000, 4                               # fp32: 4 logits per 16-byte word
    z = rng.uniform(-5.0, 5.0, V).astype(np.float32)
    top = 10.0 + np.arange(k, dtype=np.float32)    # distinct, all above the rest
    z[np.arange(k) * ev] = top                     # word t (thread t, chunk 0) for t < k
    chunk, thread = _thread_of(V, ev)
    tau = _kept_min(z, 1.0, k, 1.0, oracle_mod)
    assert tau == 10.0
    rmax = np.full(THREADS, -np.inf)
    sel = chunk == 0
    np.maximum.at(rmax, thread[sel], z[sel].astype(np.float64))
    floor = np.sort(rmax)[::-1][k - 1]
    assert floor == tau
