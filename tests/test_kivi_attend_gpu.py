"""Attention over a KIVI cache with the dequantization inside (vq_kivi_attend):
CUDA path vs the oracle (GB300), through the C ABI.

Inputs: seeded fp16 K and V quantized by the oracle's KIVI quantizer (the last
R tokens kept as the fp16 residual window), seeded queries.  Tolerance, as for
the RVQ attention: scores are fp32 sums of 128 code-times-(q*scale) products
plus the zero term, so each output lies within half an fp16 ulp of the
oracle's exact output plus 2e-5 * max|v|, and most outputs equal the oracle's
rounded fp16.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def vq():
    from kv_cache_quantization_turboquantrvq_gb300 import api, build
    build.build()
    api.lib()
    return api


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _cache(oracle_mod, B, Hkv, S_cap, R, bits, G, seed):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    k = synth.kv_tensor(B, Hkv, S_cap + R, D, seed, 4, 20.0)
    v = synth.kv_tensor(B, Hkv, S_cap + R, D, seed + 1, 0, 1.0)
    kq = oracle_mod.kivi_quant(k, bits, G, R, True)
    vq_ = oracle_mod.kivi_quant(v, bits, G, R, False)
    NG = S_cap // G
    host = {
        "k_packed": kq["packed"].reshape(B, Hkv, NG, G * bits // 32, D),
        "k_scale": kq["scale"].reshape(B, Hkv, NG, D), "k_zero": kq["zero"].reshape(B, Hkv, NG, D),
        "v_packed": vq_["packed"].reshape(B, Hkv, S_cap, D * bits // 32),
        "v_scale": vq_["scale"].reshape(B, Hkv, S_cap, D // G), "v_zero": vq_["zero"].reshape(B, Hkv, S_cap, D // G),
    }
    kr = np.ascontiguousarray(k[:, :, S_cap:])
    vr = np.ascontiguousarray(v[:, :, S_cap:])
    dev = {n: _dev(a.view(np.int32) if a.dtype == np.uint32 else a) for n, a in host.items()}
    return host, dev, kr, vr, float(np.abs(v.astype(np.float64)).max())


def _run(vq, oracle_mod, B, Hkv, gq, S_cap, R, bits, G, seed, lens=None, res=None, scale=None, **kw):
    host, dev, kr, vr, vmax = _cache(oracle_mod, B, Hkv, S_cap, R, bits, G, seed)
    q = np.random.default_rng(seed + 2).standard_normal((B, Hkv * gq, D)).astype(np.float16)
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    out = vq.vq_kivi_attend(_dev(q), dev, bits, G, scale, k_res=_dev(kr) if R else None,
                            v_res=_dev(vr) if R else None, lens=None if lens is None else _dev(lens),
                            res_lens=None if res is None else _dev(res), **kw)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    r16, r64 = oracle_mod.kivi_attend(q, host["k_packed"], host["k_scale"], host["k_zero"], host["v_packed"],
                                      host["v_scale"], host["v_zero"], bits, G, scale,
                                      k_res=kr if R else None, v_res=vr if R else None, lens=lens,
                                      res_lens=res, want_f64=True)
    return out.cpu().numpy(), r16, r64, vmax


def _check(o, r16, r64, vmax, min_exact=0.9):
    half_ulp = 0.5 * np.spacing(np.abs(r64).astype(np.float16)).astype(np.float64)
    err = np.abs(o.astype(np.float64) - r64)
    tol = half_ulp + 2e-5 * vmax
    assert np.all(err <= tol), "max excess %g" % float((err - tol).max())
    exact = float(np.mean(o.view(np.uint16) == r16.view(np.uint16)))
    assert exact >= min_exact, exact


@pytest.mark.parametrize("bits,G,gq", [(2, 32, 4), (4, 32, 2), (1, 64, 8), (2, 64, 1), (4, 128, 4),
                                       (2, 128, 8), (1, 32, 1), (4, 64, 8)])
def test_parity_with_window(vq, oracle_mod, bits, G, gq):
    B, Hkv, S_cap, R = 3, 2, 512, 20
    lens = np.array([512, 300, 33], np.int32)
    res = np.array([20, 0, 7], np.int32)
    o, r16, r64, vmax = _run(vq, oracle_mod, B, Hkv, gq, S_cap, R, bits, G, 700 + bits + G + gq, lens, res)
    _check(o, r16, r64, vmax)


@pytest.mark.parametrize("bits,G", [(2, 32), (4, 128)])
def test_parity_no_window_full_and_single_pass(vq, oracle_mod, bits, G):
    """No residual window and no length vectors; the split path (workspace)
    and the single-pass path (no workspace room) agree with the oracle."""
    B, Hkv, gq, S_cap = 2, 2, 4, 1024
    o, r16, r64, vmax = _run(vq, oracle_mod, B, Hkv, gq, S_cap, 0, bits, G, 800 + bits)
    _check(o, r16, r64, vmax)
    o1, _, _, _ = _run(vq, oracle_mod, B, Hkv, gq, S_cap, 0, bits, G, 800 + bits,
                       workspace=torch.empty(4, dtype=torch.float32, device="cuda"))
    _check(o1, r16, r64, vmax)


def test_edge_lengths(vq, oracle_mod):
    """Empty cache (zeros), window only, one quantized token, quantized tokens
    only, lengths past the capacity (clamped)."""
    bits, G, B, Hkv, gq, S_cap, R = 2, 32, 5, 1, 4, 256, 9
    lens = np.array([0, 0, 1, 256, 999], np.int32)
    res = np.array([0, 9, 0, 0, 50], np.int32)
    o, r16, r64, vmax = _run(vq, oracle_mod, B, Hkv, gq, S_cap, R, bits, G, 900, lens, res, scale=0.3)
    _check(o, r16, r64, vmax)
    assert np.all(o[0] == 0)


def test_decode_shape_sampled(vq, oracle_mod):
    """Sequences with 8 kv heads and 32 query heads, 4096-token quantized
    caches of random lengths plus a 128-token window; the oracle on sampled
    sequences."""
    bits, G, B, Hkv, gq, S_cap, R = 2, 32, 16, 8, 4, 4096, 128
    rng = np.random.default_rng(950)
    lens = (rng.integers(1, S_cap // 32 + 1, B) * 32).astype(np.int32)
    res = rng.integers(0, R + 1, B).astype(np.int32)
    host, dev, kr, vr, vmax = _cache(oracle_mod, B, Hkv, S_cap, R, bits, G, 951)
    q = rng.standard_normal((B, Hkv * gq, D)).astype(np.float16)
    scale = 1.0 / np.sqrt(D)
    out = vq.vq_kivi_attend(_dev(q), dev, bits, G, scale, k_res=_dev(kr), v_res=_dev(vr), lens=_dev(lens),
                            res_lens=_dev(res)).cpu().numpy()
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    for b in (0, 9):
        sl = slice(b, b + 1)
        r16, r64 = oracle_mod.kivi_attend(q[sl], host["k_packed"][sl], host["k_scale"][sl], host["k_zero"][sl],
                                          host["v_packed"][sl], host["v_scale"][sl], host["v_zero"][sl], bits, G,
                                          scale, k_res=kr[sl], v_res=vr[sl], lens=lens[sl], res_lens=res[sl],
                                          want_f64=True)
        _check(out[sl], r16, r64, vmax)


def test_rejects_bad_arguments(vq, oracle_mod):
    from kv_cache_quantization_turboquantrvq_gb300.api import VQError
    host, dev, kr, vr, _ = _cache(oracle_mod, 1, 2, 64, 4, 2, 32, 960)
    q = _dev(np.zeros((1, 4, D), np.float16))
    with pytest.raises(VQError) as e:   # a 64-token capacity is not a whole number of 128-token groups
        vq.vq_kivi_attend(q, dev, 2, 128, 0.1)
    assert e.value.status == vq.VQ_ERR_UNSUPPORTED
    with pytest.raises(VQError) as e:   # a window needs a workspace of two parts
        vq.vq_kivi_attend(q, dev, 2, 32, 0.1, k_res=_dev(kr), v_res=_dev(vr),
                          workspace=torch.empty(4, dtype=torch.float32, device="cuda"))
    assert e.value.status == vq.VQ_ERR_INVALID_ARG


@pytest.mark.parametrize("bits,G,gq", [(2, 32, 4), (4, 64, 2), (1, 128, 8)])
def test_rows_past_length_may_hold_anything(vq, oracle_mod, bits, G, gq):
    """Tokens past a sequence's length are never part of the result, whatever
    the cache holds there: the device copy carries NaN and inf value scales
    and zeros past the length and NaN key scales and zeros in groups wholly
    past it (partial tiles stage such rows), the oracle sees finite data."""
    B, Hkv, S_cap, R = 3, 2, 512, 5
    lens = np.array([500, 40, 0], np.int32)
    res = np.array([5, 0, 3], np.int32)
    seed = 1200 + bits + G
    host, dev, kr, vr, vmax = _cache(oracle_mod, B, Hkv, S_cap, R, bits, G, seed)
    bad = {n: a.copy() for n, a in host.items()}
    for b, n in enumerate(lens):
        bad["v_scale"][b, :, n:] = np.float16(np.nan)
        bad["v_zero"][b, :, n:] = np.float16(np.inf)
        g0 = (n + G - 1) // G  # first group with no valid token
        bad["k_scale"][b, :, g0:] = np.float16(np.nan)
        bad["k_zero"][b, :, g0:] = np.float16(-np.inf)
    dev = {n: _dev(a.view(np.int32) if a.dtype == np.uint32 else a) for n, a in bad.items()}
    q = np.random.default_rng(seed + 2).standard_normal((B, Hkv * gq, D)).astype(np.float16)
    out = vq.vq_kivi_attend(_dev(q), dev, bits, G, 0.15, k_res=_dev(kr), v_res=_dev(vr), lens=_dev(lens),
                            res_lens=_dev(res))
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    o = out.cpu().numpy()
    r16, r64 = oracle_mod.kivi_attend(q, host["k_packed"], host["k_scale"], host["k_zero"], host["v_packed"],
                                      host["v_scale"], host["v_zero"], bits, G, 0.15, k_res=kr, v_res=vr,
                                      lens=lens, res_lens=res, want_f64=True)
    assert np.all(np.isfinite(o.astype(np.float64)))
    _check(o, r16, r64, vmax)
