"""The seeded input generators: Philox4x32-10 against its published
known-answer vectors, bf16 rounding against torch, and the recipe properties of
the five benchmark configurations (at reduced sizes)."""
import numpy as np
import torch

from speculative_decoding_verification_27_gb300 import workloads as W

# Known-answer vectors of Philox4x32-10 from the Random123 distribution
# (Salmon et al., SC'11): (counter, key) -> output words.
PHILOX_KAT = [
    ((0x00000000, 0x00000000, 0x00000000, 0x00000000), (0x00000000, 0x00000000),
     (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF), (0xFFFFFFFF, 0xFFFFFFFF),
     (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


def test_philox_known_answers():
    for ctr, key, want in PHILOX_KAT:
        got = W.philox4x32_10(np.array([ctr], np.uint64).astype(np.uint32), key)[0]
        assert tuple(int(w) for w in got) == want


def test_uniforms_exact_and_layout_independent():
    cu = np.array([0, 3, 3, 7], np.int32)
    u = W.uniforms_for(cu, seed=99)
    assert u.shape == (7 + 3, 2) and u.dtype == np.float32
    assert np.all(u >= 0) and np.all(u < 1)
    assert np.all((u * 2 ** 24) == np.floor(u * 2 ** 24))  # on the 2^-24 lattice
    # Request 2's rows do not depend on how many rows come before them.
    u2 = W.uniforms_for(np.array([0, 0, 0, 4], np.int32), seed=99)
    assert np.array_equal(u[5:], u2[2:])
    assert not np.array_equal(W.uniforms_for(cu, 98), u)


def test_bf16_rounding_is_nearest_even():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.normal(0, 10, 100000), [0.0, -0.0, 1e-40, 3.0e38, -7.5, -np.inf, np.inf],
                        # exact halfway cases: ties go to the even 16-bit pattern
                        np.array([0x3F808000, 0x3F818000, 0xBF808000], np.uint32).view(np.float32)]
                       ).astype(np.float32)
    ours = W.to_bf16_bits(x)
    u = x.view(np.uint32).astype(np.uint64)
    ref = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(ours, ref)
    assert list(ours[-3:]) == [0x3F80, 0x3F82, 0xBF80]
    f = W.bf16_bits_to_f32(ours)
    assert np.all(np.abs(f[:100000] - x[:100000]) <= np.abs(x[:100000]) * 2.0 ** -8)


def test_gumbel_draft_tokens_follow_q():
    """Gumbel-max draws are samples of softmax(z / T): chi-square on V = 8."""
    from scipy.special import softmax
    rng = np.random.default_rng(2)
    z = rng.normal(0, 1, 8).astype(np.float32)
    n = 200_000
    toks = W._gumbel_argmax(np.tile(z, (n, 1)), 0.8, np.random.default_rng(3), chunk=n)
    p = softmax(z.astype(np.float64) / 0.8)
    h = np.bincount(toks, minlength=8)
    assert ((h - n * p) ** 2 / (n * p)).sum() < 24.32  # chi-square 7 dof, alpha 0.001


def test_config_recipes_small():
    b1 = W.config1(1, 5)
    assert (b1.B, b1.R_t, b1.R_d, b1.V) == (1, 5, 4, 32000) and b1.target.dtype == np.float32
    assert b1.algorithmic_bytes() == 9 * 32000 * 4
    b2 = W.config2(2, B=8, K=5, V=1000)
    zf = W.bf16_bits_to_f32(b2.target)
    top = np.sort(zf, axis=1)
    assert np.all(top[:, -1] - top[:, -2] >= 1.875)  # +2.0, then one bf16 rounding
    am = zf.argmax(1)
    slots = W._target_rows_of_draft_slots(b2.cu_draft)
    assert 0.4 < (b2.draft_tokens == am[slots]).mean() <= 1.0
    assert b2.algorithmic_bytes() == b2.R_t * 1000 * 2
    b3 = W.config3(3, B=4, K=7, V=5000)
    assert b3.target.dtype == np.uint16 and b3.draft.shape == (28, 5000)
    zt = np.sort(W.bf16_bits_to_f32(b3.target), axis=1)[:, ::-1]
    assert np.median(zt[:, 0] - zt[:, 9]) > 5.0  # peaked rows
    b5 = W.config5(5, B=40, V=512)
    Ks = np.diff(b5.cu_draft)
    assert Ks.min() >= 1 and Ks.max() <= 8 and 0 < b5.mode.sum() < 40
    greedy_rows = np.repeat(b5.mode.astype(bool), Ks)
    assert np.all(b5.draft[greedy_rows] == 0)
    assert b5.draft_rows_read() == int(Ks[b5.mode == 0].sum())


def test_config4_histories_coverage():
    nb = W.config4_histories(4, B=6, L=2048)
    assert nb.histories.shape == (6, 2048) and nb.min_n == nb.max_n == 3 and nb.max_tokens == 5
    # Planted copies: many 8-grams occur twice, which uniform noise over 32000 ids never gives.
    for b in range(6):
        h = nb.histories[b]
        grams = {}
        for s in range(0, 2048 - 8):
            grams.setdefault(h[s:s + 8].tobytes(), 0)
            grams[h[s:s + 8].tobytes()] += 1
        positions_in_copies = sum(c for c in grams.values() if c > 1)
        assert positions_in_copies > 0.3 * 2048  # copies and their sources


def test_selection_uniforms_are_on_the_lattice_and_apart_from_the_verify_uniforms():
    u = W.selection_uniforms(5000, seed=4)
    assert u.dtype == np.float32 and np.all(u >= 0) and np.all(u < 1)
    assert np.all((u * 2 ** 24) == np.floor(u * 2 ** 24))
    cu = np.arange(5001, dtype=np.int32)
    v = W.uniforms_for(cu, seed=4)
    assert not np.any(u == v[::2, 0][:5000])
    assert np.array_equal(u, W.selection_uniforms(5000, seed=4))
    assert abs(float(u.mean()) - 0.5) < 0.02
