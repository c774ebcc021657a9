"""Pins for the oracle's attention over a KIVI cache with dequantization
inside the attention (no GPU).

An independent computation (numpy bit unpacking of both code layouts,
reconstruction q*scale + zero, scipy's softmax) must agree to 1e-12; closed
forms (one token, zero scale, residual only, empty cache), masking past the
lengths and the grouped-query head mapping pin the rest.
"""
import numpy as np
import pytest

D = 128


def _cache(oracle_mod, B, Hkv, S_cap, R, bits, G, seed):
    rng = np.random.default_rng(seed)
    k = (rng.standard_normal((B, Hkv, S_cap + R, D)) * rng.uniform(0.5, 2.0, (1, 1, 1, D))).astype(np.float16)
    v = rng.standard_normal((B, Hkv, S_cap + R, D)).astype(np.float16)
    kq = oracle_mod.kivi_quant(k, bits, G, R, True)
    vq = oracle_mod.kivi_quant(v, bits, G, R, False)
    NG = S_cap // G
    c = {
        "k_packed": kq["packed"].reshape(B, Hkv, NG, G * bits // 32, D),
        "k_scale": kq["scale"].reshape(B, Hkv, NG, D), "k_zero": kq["zero"].reshape(B, Hkv, NG, D),
        "v_packed": vq["packed"].reshape(B, Hkv, S_cap, D * bits // 32),
        "v_scale": vq["scale"].reshape(B, Hkv, S_cap, D // G), "v_zero": vq["zero"].reshape(B, Hkv, S_cap, D // G),
        "k_res": np.ascontiguousarray(k[:, :, S_cap:]), "v_res": np.ascontiguousarray(v[:, :, S_cap:]),
    }
    return c


def _attend(oracle_mod, q, c, bits, G, scale, **kw):
    return oracle_mod.kivi_attend(q, c["k_packed"], c["k_scale"], c["k_zero"], c["v_packed"], c["v_scale"],
                                  c["v_zero"], bits, G, scale, k_res=c["k_res"] if c["k_res"].shape[2] else None,
                                  v_res=c["v_res"] if c["v_res"].shape[2] else None, **kw)


def _np_keys(c, bits, G):
    """[B, Hkv, S_cap, D] reconstructed keys from the per-channel layout, in numpy."""
    kp = c["k_packed"]
    B, Hkv, NG, WPG, _ = kp.shape
    E = 32 // bits
    s = np.arange(NG * G)
    words = kp[:, :, s // G, (s % G) // E, :]                      # [B, Hkv, S, D]
    codes = (words >> (((s % G) % E) * bits).astype(np.uint32)[None, None, :, None]) & ((1 << bits) - 1)
    sc = c["k_scale"].astype(np.float64)[:, :, s // G, :]
    ze = c["k_zero"].astype(np.float64)[:, :, s // G, :]
    return codes * sc + ze


def _np_values(c, bits, G):
    vp = c["v_packed"]
    E = 32 // bits
    d = np.arange(D)
    codes = (vp[..., d // E] >> ((d % E) * bits).astype(np.uint32)) & ((1 << bits) - 1)
    return codes * c["v_scale"].astype(np.float64)[..., d // G] + c["v_zero"].astype(np.float64)[..., d // G]


@pytest.mark.parametrize("bits,G", [(2, 32), (4, 64), (1, 128), (2, 128)])
def test_matches_independent_dequantized_softmax(oracle_mod, bits, G):
    special = pytest.importorskip("scipy.special")
    B, Hkv, GQ, S_cap, R = 2, 2, 2, 2 * 128, 5
    c = _cache(oracle_mod, B, Hkv, S_cap, R, bits, G, 10 + bits + G)
    q = np.random.default_rng(11).standard_normal((B, Hkv * GQ, D)).astype(np.float16)
    lens = np.array([S_cap, 77], np.int32)
    res = np.array([R, 2], np.int32)
    _, f = _attend(oracle_mod, q, c, bits, G, 0.13, lens=lens, res_lens=res, want_f64=True)
    K, V = _np_keys(c, bits, G), _np_values(c, bits, G)
    for b in range(B):
        for hq in range(Hkv * GQ):
            h = hq // GQ
            k = np.concatenate([K[b, h, :lens[b]], c["k_res"][b, h, :res[b]].astype(np.float64)])
            v = np.concatenate([V[b, h, :lens[b]], c["v_res"][b, h, :res[b]].astype(np.float64)])
            w = special.softmax(0.13 * (k @ q[b, hq].astype(np.float64)))
            np.testing.assert_allclose(f[b, hq], w @ v, rtol=1e-11, atol=1e-13)


def test_single_token_and_zero_scale(oracle_mod):
    bits, G, S_cap = 2, 32, 64
    c = _cache(oracle_mod, 1, 1, S_cap, 0, bits, G, 20)
    q = np.random.default_rng(21).standard_normal((1, 1, D)).astype(np.float16)
    _, f = _attend(oracle_mod, q, c, bits, G, 0.5, lens=np.array([1], np.int32), want_f64=True)
    np.testing.assert_allclose(f[0, 0], _np_values(c, bits, G)[0, 0, 0], rtol=0, atol=1e-15)
    _, f = _attend(oracle_mod, q, c, bits, G, 0.0, lens=np.array([50], np.int32), want_f64=True)
    np.testing.assert_allclose(f[0, 0], _np_values(c, bits, G)[0, 0, :50].mean(0), rtol=0, atol=1e-13)


def test_residual_only_and_empty(oracle_mod):
    bits, G, S_cap, R = 2, 32, 64, 7
    c = _cache(oracle_mod, 2, 1, S_cap, R, bits, G, 30)
    q = np.random.default_rng(31).standard_normal((2, 1, D)).astype(np.float16)
    out, f = _attend(oracle_mod, q, c, bits, G, 0.2, lens=np.array([0, 0], np.int32),
                     res_lens=np.array([R, 0], np.int32), want_f64=True)
    k = c["k_res"][0, 0].astype(np.float64)
    s = 0.2 * (k @ q[0, 0].astype(np.float64))
    w = np.exp(s - s.max())
    np.testing.assert_allclose(f[0, 0], (w / w.sum()) @ c["v_res"][0, 0].astype(np.float64), rtol=0, atol=1e-13)
    assert np.all(out[1] == 0)


def test_tokens_past_the_lengths_are_ignored(oracle_mod):
    bits, G, S_cap, R = 4, 32, 96, 6
    c = _cache(oracle_mod, 2, 2, S_cap, R, bits, G, 40)
    q = np.random.default_rng(41).standard_normal((2, 4, D)).astype(np.float16)
    lens, res = np.array([40, 96], np.int32), np.array([3, 6], np.int32)
    ref = _attend(oracle_mod, q, c, bits, G, 0.3, lens=lens, res_lens=res)
    rng = np.random.default_rng(42)
    c["v_packed"][0, :, 40:] = rng.integers(0, 2 ** 32, c["v_packed"][0, :, 40:].shape, dtype=np.uint32)
    c["v_scale"][0, :, 40:] = np.float16(100.0)
    c["k_res"][0, :, 3:] = np.float16(300.0)
    c["v_res"][0, :, 3:] = np.float16(-9.0)
    # key words of group 1 also hold tokens 32..39, which take part: only touch group 2
    c["k_packed"][0, :, 2] = rng.integers(0, 2 ** 32, c["k_packed"][0, :, 2].shape, dtype=np.uint32)
    c["k_scale"][0, :, 2] = np.float16(50.0)
    out = _attend(oracle_mod, q, c, bits, G, 0.3, lens=lens, res_lens=res)
    assert np.array_equal(out.view(np.uint16), ref.view(np.uint16))


def test_grouped_query_mapping(oracle_mod):
    bits, G, S_cap = 2, 64, 128
    c = _cache(oracle_mod, 1, 2, S_cap, 4, bits, G, 50)
    q = np.random.default_rng(51).standard_normal((1, 4, D)).astype(np.float16)
    out = _attend(oracle_mod, q, c, bits, G, 0.25)
    sw = {k: np.ascontiguousarray(v[:, ::-1]) for k, v in c.items()}
    out2 = _attend(oracle_mod, q[:, [2, 3, 0, 1]], sw, bits, G, 0.25)
    assert np.array_equal(out2[:, [2, 3, 0, 1]].view(np.uint16), out.view(np.uint16))
