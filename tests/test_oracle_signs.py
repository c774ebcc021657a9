"""Pins for the oracle's randomised-sign rotation R = H diag(s) (no GPU).

A one-hot input gives the closed form y = s_j H[:, j] / sqrt(D) (column
scaling: a row-scaled diag(s) H or a transposed product fails it); encoding x
with signs equals encoding s*x without them, bit for bit (the sign flip of an
fp16 value is exact); decoding with signs equals s * the plain decode (the
transpose R^T = diag(s) H); attention with signs equals plain attention of the
sign-flipped query over the same codes; the rotation keeps unit norms.
"""
import numpy as np
import pytest

D = 128


def _signs(seed):
    return np.random.default_rng(seed).integers(0, 2 ** 32, 4, dtype=np.uint32)


def _s_vec(signs):
    bits = (signs[np.arange(D) // 32] >> (np.arange(D) % 32).astype(np.uint32)) & 1
    return np.where(bits == 1, -1.0, 1.0)


def _hadamard_entry(i, j):
    return -1.0 if bin(i & j).count("1") % 2 else 1.0


@pytest.mark.parametrize("j", [0, 1, 37, 127])
def test_one_hot_gives_a_signed_hadamard_column(oracle_mod, j):
    signs = _signs(3)
    s = _s_vec(signs)
    x = np.zeros((1, D), np.float16)
    x[0, j] = 1.0
    cb = oracle_mod.rvq_codebooks(D, 2)[:4]
    y = oracle_mod.rvq_encode(x, 2, *cb, want_values=True, signs=signs)["y"][0]
    ref = np.array([s[j] * _hadamard_entry(i, j) for i in range(D)]) / np.sqrt(D)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-15)


def _x(seed, n=300):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, D)) * rng.uniform(0.3, 3.0, (n, 1))).astype(np.float16)


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_encode_with_signs_is_encode_of_flipped_input(oracle_mod, bits):
    x = _x(10 + bits)
    signs = _signs(20 + bits)
    s = _s_vec(signs)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    a = oracle_mod.rvq_encode(x, bits, *cb, want_values=True, signs=signs)
    b = oracle_mod.rvq_encode((x * s).astype(np.float16), bits, *cb, want_values=True)
    for k in ("packed1", "packed2", "norms", "tie1", "tie2", "y", "r"):
        assert np.array_equal(a[k], b[k]), k
    # all-zero signs are the plain rotation
    c = oracle_mod.rvq_encode(x, bits, *cb, signs=np.zeros(4, np.uint32))
    d = oracle_mod.rvq_encode(x, bits, *cb)
    assert np.array_equal(c["packed1"], d["packed1"]) and np.array_equal(c["packed2"], d["packed2"])
    # a different sign vector changes the codes
    e = oracle_mod.rvq_encode(x, bits, *cb, signs=_signs(99))
    assert not np.array_equal(e["packed1"], a["packed1"])


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_rotation_keeps_unit_norm(oracle_mod, bits):
    x = _x(30 + bits, 50)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    y = oracle_mod.rvq_encode(x, bits, *cb, want_values=True, signs=_signs(31))["y"]
    np.testing.assert_allclose(np.sum(y * y, axis=1), 1.0, rtol=0, atol=1e-13)


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_decode_with_signs_is_the_transpose(oracle_mod, bits):
    x = _x(40 + bits, 100)
    signs = _signs(41 + bits)
    s = _s_vec(signs)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    e = oracle_mod.rvq_encode(x, bits, *cb, signs=signs)
    h16, h64 = oracle_mod.rvq_decode(e["packed1"], e["packed2"], e["norms"], D, bits, cb[0], cb[2],
                                     want_f64=True, signs=signs)
    p16, p64 = oracle_mod.rvq_decode(e["packed1"], e["packed2"], e["norms"], D, bits, cb[0], cb[2],
                                     want_f64=True)
    assert np.array_equal(h64, p64 * s)
    assert np.array_equal(h16, (p16 * s).astype(np.float16))
    # the round trip lands back near x (quantizer distortion only)
    xd = x.astype(np.float64)
    err = np.linalg.norm(h64 - xd, axis=1) / np.linalg.norm(xd, axis=1)
    assert err.max() < {1: 0.75, 2: 0.35, 4: 0.06}[bits]


def test_attention_with_signs_is_attention_of_the_flipped_query(oracle_mod):
    bits, B, Hkv, Hq, S = 2, 2, 2, 4, 40
    rng = np.random.default_rng(50)
    signs = _signs(51)
    s = _s_vec(signs)
    cb = oracle_mod.rvq_codebooks(D, bits)
    k = _x(52, B * Hkv * S)
    e = oracle_mod.rvq_encode(k, bits, *cb[:4], signs=signs)
    p1 = e["packed1"].reshape(B, Hkv, S, -1)
    p2 = e["packed2"].reshape(B, Hkv, S, -1)
    nr = e["norms"].reshape(B, Hkv, S)
    v = rng.standard_normal((B, Hkv, S, D)).astype(np.float16)
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    lens = np.array([S, 17], np.int32)
    a16, a64 = oracle_mod.rvq_attend(q, p1, p2, nr, v, bits, cb[0], cb[2], 0.2, lens=lens, want_f64=True,
                                     signs=signs)
    b16, b64 = oracle_mod.rvq_attend((q * s).astype(np.float16), p1, p2, nr, v, bits, cb[0], cb[2], 0.2,
                                     lens=lens, want_f64=True)
    assert np.array_equal(a64, b64)
    # and it is attention over the decoded keys (the transpose rotation)
    kd = oracle_mod.rvq_decode(e["packed1"], e["packed2"], e["norms"], D, bits, cb[0], cb[2], want_f64=True,
                               signs=signs)[1].reshape(B, Hkv, S, D)
    for bb in range(B):
        L = lens[bb]
        for hq in range(Hq):
            h = hq // 2
            sc = 0.2 * (kd[bb, h, :L] @ q[bb, hq].astype(np.float64))
            w = np.exp(sc - sc.max())
            np.testing.assert_allclose(a64[bb, hq], (w / w.sum()) @ v[bb, h, :L].astype(np.float64),
                                       rtol=0, atol=1e-12)
