"""Pins for the oracle's decode-time attention over an RVQ key cache (no GPU).

Closed forms (one key, zero scale, identical keys, a dominant key, an empty
cache), invariants (masking past the valid length, the grouped-query head
mapping) and an independent rotated-domain computation (scipy's Sylvester
Hadamard, numpy bit unpacking, scipy's softmax) pin oracle_rvq_attend.
"""
import numpy as np
import pytest

D = 128


def _cache(oracle_mod, B, Hkv, S, bits, seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((B * Hkv * S, D)) * rng.uniform(0.5, 2.0, (B * Hkv * S, 1))).astype(np.float16)
    cb = oracle_mod.rvq_codebooks(D, bits)
    e = oracle_mod.rvq_encode(x, bits, *cb[:4])
    W = D * bits // 32
    p1 = e["packed1"].reshape(B, Hkv, S, W)
    p2 = e["packed2"].reshape(B, Hkv, S, W)
    nr = e["norms"].reshape(B, Hkv, S)
    v = rng.standard_normal((B, Hkv, S, D)).astype(np.float16)
    return p1, p2, nr, v, cb


def _q(B, Hq, seed):
    return np.random.default_rng(seed).standard_normal((B, Hq, D)).astype(np.float16)


def test_single_key_gives_its_value(oracle_mod):
    p1, p2, nr, v, cb = _cache(oracle_mod, 2, 2, 4, 2, 1)
    q = _q(2, 4, 2)
    out = oracle_mod.rvq_attend(q, p1, p2, nr, v, 2, cb[0], cb[2], 0.3, lens=np.array([1, 1], np.int32))
    for b in range(2):
        for hq in range(4):
            assert np.array_equal(out[b, hq].view(np.uint16), v[b, hq // 2, 0].view(np.uint16))


def test_zero_scale_is_the_mean_of_the_values(oracle_mod):
    p1, p2, nr, v, cb = _cache(oracle_mod, 1, 2, 9, 4, 3)
    q = _q(1, 2, 4)
    lens = np.array([7], np.int32)
    _, f = oracle_mod.rvq_attend(q, p1, p2, nr, v, 4, cb[0], cb[2], 0.0, lens=lens, want_f64=True)
    mean = v[0, :, :7].astype(np.float64).mean(axis=1)
    np.testing.assert_allclose(f[0], mean, rtol=0, atol=1e-13)


def test_identical_keys_weigh_equally(oracle_mod):
    p1, p2, nr, v, cb = _cache(oracle_mod, 1, 1, 6, 2, 5)
    p1[:] = p1[:, :, :1]
    p2[:] = p2[:, :, :1]
    nr[:] = nr[:, :, :1]
    _, f = oracle_mod.rvq_attend(_q(1, 3, 6), p1, p2, nr, v, 2, cb[0], cb[2], 1.7, want_f64=True)
    mean = v[0, 0].astype(np.float64).mean(axis=0)
    for hq in range(3):
        np.testing.assert_allclose(f[0, hq], mean, rtol=0, atol=1e-13)


def test_dominant_key_takes_all_weight(oracle_mod):
    bits = 2
    p1, p2, nr, v, cb = _cache(oracle_mod, 1, 1, 8, bits, 7)
    j = 5
    kd = oracle_mod.rvq_decode(p1[0, 0, j:j + 1], p2[0, 0, j:j + 1], nr[0, 0, j:j + 1], D, bits, cb[0], cb[2],
                               want_f64=True)[1][0]
    q = (kd / np.linalg.norm(kd)).astype(np.float16).reshape(1, 1, D)
    # every other key is at least a few percent less aligned; a large scale
    # makes the softmax a one-hot up to exp(-(gap) * scale)
    _, f = oracle_mod.rvq_attend(q, p1, p2, nr, v, bits, cb[0], cb[2], 1.0e4, want_f64=True)
    np.testing.assert_allclose(f[0, 0], v[0, 0, j].astype(np.float64), rtol=0, atol=1e-9)


def test_empty_cache_gives_zeros(oracle_mod):
    p1, p2, nr, v, cb = _cache(oracle_mod, 2, 1, 3, 1, 8)
    out = oracle_mod.rvq_attend(_q(2, 2, 9), p1, p2, nr, v, 1, cb[0], cb[2], 0.1,
                                lens=np.array([0, 3], np.int32))
    assert np.all(out[0].astype(np.float32) == 0.0)
    assert np.any(out[1].astype(np.float32) != 0.0)


def test_tokens_past_the_length_are_ignored(oracle_mod):
    p1, p2, nr, v, cb = _cache(oracle_mod, 2, 2, 10, 2, 10)
    q = _q(2, 4, 11)
    lens = np.array([4, 9], np.int32)
    ref = oracle_mod.rvq_attend(q, p1, p2, nr, v, 2, cb[0], cb[2], 0.2, lens=lens)
    rng = np.random.default_rng(12)
    for b, L in enumerate(lens):
        p1[b, :, L:] = rng.integers(0, 2 ** 32, p1[b, :, L:].shape, dtype=np.uint32)
        p2[b, :, L:] = rng.integers(0, 2 ** 32, p2[b, :, L:].shape, dtype=np.uint32)
        nr[b, :, L:] = 1.0e30
        v[b, :, L:] = np.float16(6.0e4)
    out = oracle_mod.rvq_attend(q, p1, p2, nr, v, 2, cb[0], cb[2], 0.2, lens=lens)
    assert np.array_equal(out.view(np.uint16), ref.view(np.uint16))


def test_grouped_query_head_mapping(oracle_mod):
    p1, p2, nr, v, cb = _cache(oracle_mod, 1, 2, 5, 2, 13)
    q = _q(1, 4, 14)
    q[0, 2] = q[0, 0]
    out = oracle_mod.rvq_attend(q, p1, p2, nr, v, 2, cb[0], cb[2], 0.5)
    # swap the two kv heads: heads 0,1 and 2,3 trade kv heads
    sw = lambda a: a[:, ::-1].copy()
    out2 = oracle_mod.rvq_attend(q[:, [2, 3, 0, 1]], sw(p1), sw(p2), sw(nr), sw(v), 2, cb[0], cb[2], 0.5)
    assert np.array_equal(out2[:, [2, 3, 0, 1]].view(np.uint16), out.view(np.uint16))
    # same query on both kv heads with the same cache: same output
    p1[:, 1], p2[:, 1], nr[:, 1], v[:, 1] = p1[:, 0], p2[:, 0], nr[:, 0], v[:, 0]
    out3 = oracle_mod.rvq_attend(q, p1, p2, nr, v, 2, cb[0], cb[2], 0.5)
    assert np.array_equal(out3[0, 0].view(np.uint16), out3[0, 2].view(np.uint16))


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_rotated_domain_scores_independently(oracle_mod, bits):
    """The attention computed from the rotated query (scipy's Sylvester
    Hadamard) against the codebook values of the codes unpacked with numpy
    bit operations, with scipy's softmax: q . k_s = n_s (H q / sqrt D) . y_s."""
    linalg = pytest.importorskip("scipy.linalg")
    special = pytest.importorskip("scipy.special")
    B, Hq, Hkv, S = 2, 4, 2, 11
    p1, p2, nr, v, cb = _cache(oracle_mod, B, Hkv, S, bits, 20 + bits)
    q = _q(B, Hq, 30 + bits)
    lens = np.array([S, 6], np.int32)
    scale = 0.37
    _, f = oracle_mod.rvq_attend(q, p1, p2, nr, v, bits, cb[0], cb[2], scale, lens=lens, want_f64=True)
    H = linalg.hadamard(D).astype(np.float64)
    E = 32 // bits
    mask = (1 << bits) - 1
    c1 = cb[0].astype(np.float64)
    c2 = cb[2].astype(np.float64)

    def codes(words):  # [..., W] -> [..., D], LSB first
        sh = (np.arange(D) % E) * bits
        return (words[..., np.arange(D) // E] >> sh.astype(np.uint32)) & mask

    for b in range(B):
        for hq in range(Hq):
            h = hq // (Hq // Hkv)
            L = lens[b]
            qt = H @ q[b, hq].astype(np.float64) / np.sqrt(D)
            y = c1[codes(p1[b, h, :L])] + c2[codes(p2[b, h, :L])]
            s = scale * nr[b, h, :L].astype(np.float64) * (y @ qt)
            w = special.softmax(s)
            o = w @ v[b, h, :L].astype(np.float64)
            np.testing.assert_allclose(f[b, hq], o, rtol=1e-11, atol=1e-13)
