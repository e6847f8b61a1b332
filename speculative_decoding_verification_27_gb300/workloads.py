"""Seeded synthetic inputs for the verify-and-commit step and the n-gram proposer.

This module is the only code that both the CUDA path's callers (tests, bench)
and the float64 oracle's callers share. It holds none of the method's
arithmetic: no softmax, no accept test, no residual, no inverse-CDF draw.

* Uniforms are Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
  Numbers: As Easy as 1, 2, 3", SC'11), implemented here from that published
  definition: key = the 64-bit seed, counter = (request b, slot i, round, 0);
  word 0 gives the accept uniform u, word 1 the draw uniform u', each as
  (w >> 8) * 2**-24, so every uniform is an exact float32 in [0, 1).
* Logit noise comes from torch's seeded CPU generator; permutations, choices
  and Gumbel uniforms from numpy's PCG64, both seeded from (seed, stream).
* Draft tokens "sampled from q" use the Gumbel-max identity:
  argmax_x (z_x / T + G_x), G_x = -log(-log U_x), is an exact sample of
  softmax(z / T) without computing that softmax.
* bf16 logits are float32 values rounded to nearest-even and stored as their
  16-bit patterns (uint16).

Recipes (shapes and distributions of the five benchmark configurations):
  1. B=1, K=4, V=32000 fp32; z_t ~ N(0, 2^2); z_d = z_t + N(0, 0.5^2);
     x̂ ~ q; T = 1.0; rounds r = 0..999 with fresh logits and uniforms.
  2. B=64, K=5, V=128256 bf16 greedy; z ~ N(0, 3^2); one random token per
     row set to max(others) + 2.0 after rounding (unique argmax); x̂ = the
     argmax with probability 0.7, else uniform over V.
  3. B=256, K=7, V=151936 bf16, T=0.7; z_t[pi(r)] = -4.4 ln r + N(0,1) with
     a fresh random permutation pi per row (4x the log of Zipf s=1.1 rank
     weights: peaked rows); z_d = z_t + N(0,1); x̂ ~ q.
  4. B=128 histories of 8192 int32 tokens uniform over V=32000; spans of
     U[16,64] tokens copied from earlier positions until 30% of each history
     is covered. Proposals (n=3, max 5 tokens) are verified with one-hot q
     against fp32 target logits z ~ N(0, 2^2), T = 1.0.
  5. B=512, K_b ~ U{1..8}, V=256000 bf16, T=1.0; z_t ~ N(0, 2^2);
     z_d = z_t + N(0, 0.75^2); request b is greedy with probability 0.5
     (x̂ as in 2), else sampling with x̂ ~ q. Draft rows of greedy requests
     are never read and are left zero.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# ----------------------------------------------------------------------------
# Philox4x32-10
# ----------------------------------------------------------------------------
_PHILOX_M0 = np.uint64(0xD2511F53)
_PHILOX_M1 = np.uint64(0xCD9E8D57)
_PHILOX_W0 = 0x9E3779B9
_PHILOX_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(counter: np.ndarray, key) -> np.ndarray:
    """Philox4x32 with 10 rounds. counter: [N, 4] uint32, key: (k0, k1).

    Each round multiplies words 0 and 2 by the two Philox multipliers (64-bit
    products split into hi/lo halves), mixes the high halves with words 1 and
    3 and the key, and the key is bumped by the two Weyl constants between
    rounds.
    """
    c = np.asarray(counter, dtype=np.uint32).reshape(-1, 4).astype(np.uint64)
    c0, c1, c2, c3 = c[:, 0], c[:, 1], c[:, 2], c[:, 3]
    k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
    for rnd in range(10):
        if rnd:
            k0 = (k0 + _PHILOX_W0) & 0xFFFFFFFF
            k1 = (k1 + _PHILOX_W1) & 0xFFFFFFFF
        p0 = _PHILOX_M0 * c0
        p1 = _PHILOX_M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK32
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1, hi0 ^ c3 ^ np.uint64(k1), lo0)
    return np.stack([c0, c1, c2, c3], axis=1).astype(np.uint32)


def _seed_key(seed: int):
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & 0xFFFFFFFF, seed >> 32


def uniforms_for(cu_draft: np.ndarray, seed: int, round_index: int = 0) -> np.ndarray:
    """[R_t, 2] float32: (u, u') for target row (b, i), counter (b, i, round, 0)."""
    cu = np.asarray(cu_draft, np.int64)
    B = cu.shape[0] - 1
    k = np.diff(cu) + 1
    b = np.repeat(np.arange(B, dtype=np.int64), k)
    i = np.arange(int(k.sum()), dtype=np.int64) - np.repeat(cu[:-1] + np.arange(B), k)
    ctr = np.zeros((b.shape[0], 4), np.uint32)
    ctr[:, 0] = b
    ctr[:, 1] = i
    ctr[:, 2] = round_index
    w = philox4x32_10(ctr, _seed_key(seed))
    return ((w[:, :2] >> np.uint32(8)).astype(np.float32) * np.float32(2.0 ** -24)).astype(np.float32)


def selection_uniforms(B: int, seed: int, round_index: int = 0) -> np.ndarray:
    """[B] float32 in [0, 1): one uniform per request for choosing among its
    draft candidates, drawn apart from the verify uniforms: Philox counter
    (b, 0, round, 1); u = (w0 >> 8) * 2^-24."""
    ctr = np.zeros((int(B), 4), np.uint32)
    ctr[:, 0] = np.arange(int(B), dtype=np.uint32)
    ctr[:, 2] = round_index
    ctr[:, 3] = 1
    w = philox4x32_10(ctr, _seed_key(seed))
    return ((w[:, 0] >> np.uint32(8)).astype(np.float32) * np.float32(2.0 ** -24)).astype(np.float32)


# ----------------------------------------------------------------------------
# bf16 storage
# ----------------------------------------------------------------------------
def to_bf16_bits(x) -> np.ndarray:
    """Round float32 to bf16 (nearest-even) and return the 16-bit patterns
    (torch's conversion, multi-threaded; checked bit for bit against the
    round-to-nearest-even formula in the tests)."""
    import torch
    t = x if isinstance(x, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(x, np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def logits_as_f32(z: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(z) if z.dtype == np.uint16 else np.asarray(z, np.float32)


# ----------------------------------------------------------------------------
# Batches
# ----------------------------------------------------------------------------
@dataclass
class VerifyBatch:
    """Packed inputs of one spec_verify call.

    target: [R_t, V] float32 or uint16 (bf16 patterns); row (b, i) at
    cu_draft[b] + b + i. draft: [R_d, V] same dtype, row (b, i) at
    cu_draft[b] + i, or None for one-hot proposals. draft_tokens: [R_d] int32.
    cu_draft: [B+1] int32. mode: [B] uint8 (0 sample, 1 greedy) or None.
    uniforms: [R_t, 2] float32.
    """
    name: str
    target: np.ndarray
    draft: Optional[np.ndarray]
    draft_tokens: np.ndarray
    cu_draft: np.ndarray
    uniforms: np.ndarray
    temperature: float
    mode: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.cu_draft.shape[0] - 1)

    @property
    def V(self) -> int:
        return int(self.target.shape[1])

    @property
    def R_t(self) -> int:
        return int(self.cu_draft[-1]) + self.B

    @property
    def R_d(self) -> int:
        return int(self.cu_draft[-1])

    @property
    def elem_bytes(self) -> int:
        return 2 if self.target.dtype == np.uint16 else 4

    def greedy_mask(self) -> np.ndarray:
        if self.mode is None:
            return np.zeros(self.B, bool)
        return self.mode.astype(bool)

    def draft_rows_read(self) -> int:
        """Draft rows the step must read: sampling requests with a draft row set."""
        if self.draft is None:
            return 0
        k = np.diff(self.cu_draft.astype(np.int64))
        return int(k[~self.greedy_mask()].sum())

    def algorithmic_bytes(self) -> int:
        """Every needed logit read once: V * s * (R_t + sampling draft rows)."""
        return self.V * self.elem_bytes * (self.R_t + self.draft_rows_read())


@dataclass
class NgramBatch:
    histories: np.ndarray  # [B, stride] int32
    hist_len: np.ndarray   # [B] int32
    min_n: int
    max_n: int
    max_tokens: int


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed) & 0xFFFFFFFF, *stream])))


class _Normal:
    """Seeded float32 Gaussian noise from torch's CPU generator (multi-threaded;
    numpy's sampler is several times slower at these sizes)."""

    def __init__(self, rng: np.random.Generator):
        import torch
        self._torch = torch
        self._g = torch.Generator().manual_seed(int(rng.integers(0, 2 ** 62)))

    def __call__(self, shape, sigma: float = 1.0) -> np.ndarray:
        z = self._torch.randn(shape, generator=self._g, dtype=self._torch.float32)
        if sigma != 1.0:
            z.mul_(float(sigma))
        return z.numpy()


def _gumbel_argmax(z: np.ndarray, T: float, rng: np.random.Generator, chunk: int = 64) -> np.ndarray:
    """x̂ ~ softmax(z / T) per row via argmax(z / T + Gumbel noise), float64."""
    import torch
    g = torch.Generator().manual_seed(int(rng.integers(0, 2 ** 62)))
    out = np.empty(z.shape[0], np.int32)
    for r0 in range(0, z.shape[0], chunk):
        zz = torch.from_numpy(logits_as_f32(z[r0:r0 + chunk])).double().div_(T)
        u = torch.rand(zz.shape, generator=g, dtype=torch.float64).clamp_(min=1e-300)
        zz.sub_(u.log_().neg_().log_())
        out[r0:r0 + chunk] = zz.argmax(dim=1).numpy()
    return out


def _greedy_draft_tokens(target: np.ndarray, rows: np.ndarray, V: int, rng, p_match: float = 0.7):
    """x̂ = argmax of the target row with probability p_match, else uniform over V."""
    zt = logits_as_f32(target[rows])
    am = np.argmax(zt, axis=1).astype(np.int32)
    hit = rng.random(rows.shape[0]) < p_match
    return np.where(hit, am, rng.integers(0, V, rows.shape[0])).astype(np.int32)


def _ragged_cu(K: np.ndarray) -> np.ndarray:
    cu = np.zeros(K.shape[0] + 1, np.int32)
    cu[1:] = np.cumsum(K)
    return cu


def _target_rows_of_draft_slots(cu: np.ndarray) -> np.ndarray:
    """Target-row index (cu[b] + b + i) for every draft slot (b, i)."""
    B = cu.shape[0] - 1
    K = np.diff(cu.astype(np.int64))
    return (np.arange(int(cu[-1]), dtype=np.int64) + np.repeat(np.arange(B), K)).astype(np.int64)


# ----------------------------------------------------------------------------
# Configurations
# ----------------------------------------------------------------------------
def gaussian_sampling(seed: int, B: int, K, V: int, sigma: float, draft_sigma: float,
                      T: float, dtype: str = "fp32", round_index: int = 0,
                      name: str = "gaussian") -> VerifyBatch:
    """Sampling batch with z_t ~ N(0, sigma^2), z_d = z_t + N(0, draft_sigma^2), x̂ ~ q."""
    rng = _rng(seed, 1, round_index)
    normal = _Normal(rng)
    Ks = np.full(B, K, np.int32) if np.isscalar(K) else np.asarray(K, np.int32)
    cu = _ragged_cu(Ks)
    R_t, R_d = int(cu[-1]) + B, int(cu[-1])
    zt = normal((R_t, V), sigma)
    if dtype == "bf16":
        zt = bf16_bits_to_f32(to_bf16_bits(zt))
    rows = _target_rows_of_draft_slots(cu)
    zd = zt[rows] + normal((R_d, V), draft_sigma)
    if dtype == "bf16":
        zt_s, zd_s = to_bf16_bits(zt), to_bf16_bits(zd)
    else:
        zt_s, zd_s = zt, zd.astype(np.float32)
    toks = _gumbel_argmax(zd_s, T, rng)
    return VerifyBatch(name, zt_s, zd_s, toks, cu, uniforms_for(cu, seed, round_index), T,
                       None, {"seed": seed, "round": round_index})


def config1(seed: int = 1, round_index: int = 0, V: int = 32000, K: int = 4) -> VerifyBatch:
    """Sampling, B=1, K=4, V=32000 fp32, T=1.0 (one of its 1000 rounds)."""
    return gaussian_sampling(seed, 1, K, V, 2.0, 0.5, 1.0, "fp32", round_index, "config1")


def config2(seed: int = 2, B: int = 64, K: int = 5, V: int = 128256,
            margin: float = 2.0, p_match: float = 0.7) -> VerifyBatch:
    """Greedy/strict, B=64, K=5, V=128256 bf16 with a planted argmax margin."""
    rng = _rng(seed, 2)
    cu = _ragged_cu(np.full(B, K, np.int32))
    R_t = int(cu[-1]) + B
    z = bf16_bits_to_f32(to_bf16_bits(_Normal(rng)((R_t, V), 3.0)))
    win = rng.integers(0, V, R_t)
    others = z.copy()
    others[np.arange(R_t), win] = -np.inf
    z[np.arange(R_t), win] = others.max(axis=1) + np.float32(margin)
    zb = to_bf16_bits(z)
    zf = bf16_bits_to_f32(zb)
    top = zf.max(axis=1)
    assert np.all((zf == top[:, None]).sum(axis=1) == 1), "planted argmax must be unique"
    rows = _target_rows_of_draft_slots(cu)
    toks = _greedy_draft_tokens(zb, rows, V, rng, p_match)
    mode = np.ones(B, np.uint8)
    return VerifyBatch("config2", zb, None, toks, cu, uniforms_for(cu, seed), 1.0, mode,
                       {"seed": seed})


def config3(seed: int = 3, B: int = 256, K: int = 7, V: int = 151936, T: float = 0.7,
            zipf_scale: float = 4.0, zipf_s: float = 1.1, literal_zipf: bool = False) -> VerifyBatch:
    """Sampling, B=256, K=7, V=151936 bf16, T=0.7, peaked rank-score rows.

    Peaked reading (default): z_t[pi(r)] = zipf_scale * ln(r**-zipf_s) + N(0,1).
    literal_zipf=True uses zipf_scale * r**-zipf_s + N(0,1) instead (near-flat
    rows at this V). The bytes read are the same either way.
    """
    rng = _rng(seed, 3)
    cu = _ragged_cu(np.full(B, K, np.int32))
    R_t, R_d = int(cu[-1]) + B, int(cu[-1])
    r = np.arange(1, V + 1, dtype=np.float64)
    base = (zipf_scale * r ** -zipf_s if literal_zipf else -zipf_scale * zipf_s * np.log(r)).astype(np.float32)
    import torch
    base_t = torch.from_numpy(base)
    normal = _Normal(rng)
    zt = np.empty((R_t, V), np.uint16)
    chunk = 128
    for r0 in range(0, R_t, chunk):
        n = min(chunk, R_t - r0)
        # z[j] = base[sigma(j)] for a uniformly random permutation sigma of the
        # ranks (sigma is the inverse of pi, and is itself uniform).
        sig = np.empty((n, V), np.int64)
        for k in range(n):
            sig[k] = rng.permutation(V)
        zt[r0:r0 + n] = to_bf16_bits(base_t[torch.from_numpy(sig)].add_(torch.from_numpy(normal((n, V)))))
    rows = _target_rows_of_draft_slots(cu)
    zd = np.empty((R_d, V), np.uint16)
    for r0 in range(0, R_d, chunk):
        n = min(chunk, R_d - r0)
        zd[r0:r0 + n] = to_bf16_bits(bf16_bits_to_f32(zt[rows[r0:r0 + n]]) + normal((n, V)))
    toks = _gumbel_argmax(zd, T, rng)
    return VerifyBatch("config3", zt, zd, toks, cu, uniforms_for(cu, seed), T, None,
                       {"seed": seed, "literal_zipf": literal_zipf})


def config4_histories(seed: int = 4, B: int = 128, L: int = 8192, V: int = 32000,
                      coverage: float = 0.3, span=(16, 64), n: int = 3,
                      max_tokens: int = 5, ragged: bool = False) -> NgramBatch:
    """Token histories with planted copied spans (the n-gram proposer's input)."""
    rng = _rng(seed, 4)
    h = rng.integers(0, V, (B, L), dtype=np.int64).astype(np.int32)
    lens = np.full(B, L, np.int32)
    if ragged:
        lens = rng.integers(1, L + 1, B).astype(np.int32)
    for b in range(B):
        Lb = int(lens[b])
        covered = np.zeros(Lb, bool)
        if Lb < 2 * span[0]:
            continue
        while covered.sum() < coverage * Lb:
            ln = int(rng.integers(span[0], min(span[1], Lb // 2) + 1))
            # Destinations start anywhere after one span length and are clipped
            # at the end, so every position (the tail included) is equally
            # likely to lie in a copy; the source lies wholly before it.
            d = int(rng.integers(ln, Lb))
            m = min(ln, Lb - d)
            s = int(rng.integers(0, d - ln + 1))
            h[b, d:d + m] = h[b, s:s + m]
            covered[d:d + m] = True
    return NgramBatch(h, lens, n, n, max_tokens)


def config4_verify(seed: int, proposals: np.ndarray, counts: np.ndarray, V: int = 32000,
                   sigma: float = 2.0) -> VerifyBatch:
    """Verify batch for n-gram proposals: K_b = counts[b], one-hot q, fp32 z ~ N(0, sigma^2)."""
    rng = _rng(seed, 41)
    counts = np.asarray(counts, np.int32)
    cu = _ragged_cu(counts)
    B = counts.shape[0]
    R_t = int(cu[-1]) + B
    toks = np.concatenate([proposals[b, :counts[b]] for b in range(B)]).astype(np.int32) \
        if int(cu[-1]) else np.zeros(0, np.int32)
    zt = _Normal(rng)((R_t, V), sigma)
    return VerifyBatch("config4", zt, None, toks, cu, uniforms_for(cu, seed), 1.0, None,
                       {"seed": seed})


def config5(seed: int = 5, B: int = 512, V: int = 256000, Kmax: int = 8, T: float = 1.0,
            sigma: float = 2.0, draft_sigma: float = 0.75, p_greedy: float = 0.5) -> VerifyBatch:
    """Ragged mixed batch: K_b ~ U{1..Kmax}, V=256000 bf16, half greedy requests."""
    rng = _rng(seed, 5)
    Ks = rng.integers(1, Kmax + 1, B).astype(np.int32)
    mode = (rng.random(B) < p_greedy).astype(np.uint8)
    cu = _ragged_cu(Ks)
    R_t, R_d = int(cu[-1]) + B, int(cu[-1])
    normal = _Normal(rng)
    zt = np.empty((R_t, V), np.uint16)
    chunk = 128
    for r0 in range(0, R_t, chunk):
        n = min(chunk, R_t - r0)
        zt[r0:r0 + n] = to_bf16_bits(normal((n, V), sigma))
    rows = _target_rows_of_draft_slots(cu)
    req_of_slot = np.repeat(np.arange(B), Ks)
    samp_slots = np.nonzero(mode[req_of_slot] == 0)[0]
    greedy_slots = np.nonzero(mode[req_of_slot] == 1)[0]
    zd = np.zeros((R_d, V), np.uint16)
    for s0 in range(0, samp_slots.shape[0], chunk):
        sl = samp_slots[s0:s0 + chunk]
        zd[sl] = to_bf16_bits(bf16_bits_to_f32(zt[rows[sl]]) + normal((sl.shape[0], V), draft_sigma))
    toks = np.zeros(R_d, np.int32)
    if samp_slots.size:
        toks[samp_slots] = _gumbel_argmax(zd[samp_slots], T, rng)
    if greedy_slots.size:
        toks[greedy_slots] = _greedy_draft_tokens(zt, rows[greedy_slots], V, rng)
    return VerifyBatch("config5", zt, zd, toks, cu, uniforms_for(cu, seed), T, mode,
                       {"seed": seed})
