"""KIVI CUDA path vs the oracle (GB300), through the C ABI."""
import numpy as np
import pytest

from parity import check_codes, unpack_kivi_keys, unpack_rows

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


def _np(t):
    return t.cpu().numpy()


def _check_keys(out, ora, bits, G, S_q, strict=True):
    BH = ora["codes"].shape[0]
    kp = _np(out["k_packed"]).reshape(BH, -1, G * bits // 32, D)
    NG = ora["NG"]
    codes = unpack_kivi_keys(kp[:, :NG], bits, G, S_q)
    check_codes(codes, ora["codes"], ora["tie"], "key codes", strict=strict)
    ks = _np(out["k_scale"]).reshape(BH, -1, D)[:, :NG]
    kz = _np(out["k_zero"]).reshape(BH, -1, D)[:, :NG]
    assert np.array_equal(ks.view(np.uint16), ora["scale"].view(np.uint16))
    assert np.array_equal(kz.view(np.uint16), ora["zero"].view(np.uint16))
    # pad slots of a ragged last group hold code 0
    if S_q % G:
        full = unpack_kivi_keys(kp[:, :NG], bits, G, NG * G)
        assert np.all(full[:, S_q:] == 0)


def _check_values(out, ora, bits, G, strict=True):
    BH, S_q, _ = ora["codes"].shape
    vp = _np(out["v_packed"]).reshape(BH, -1, D * bits // 32)[:, :S_q]
    codes = unpack_rows(vp, bits)
    check_codes(codes, ora["codes"], ora["tie"], "value codes", strict=strict)
    vs = _np(out["v_scale"]).reshape(BH, -1, D // G)[:, :S_q]
    vz = _np(out["v_zero"]).reshape(BH, -1, D // G)[:, :S_q]
    assert np.array_equal(vs.view(np.uint16), ora["scale"].view(np.uint16))
    assert np.array_equal(vz.view(np.uint16), ora["zero"].view(np.uint16))


def _gen(shape, seed, scale=1.0, outl=0):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    B, H, S = shape
    return (synth.kv_tensor(B, H, S, D, seed, outl, 20.0).astype(np.float32) * scale).astype(np.float16)


ALL_BG = [(b, g) for b in (1, 2, 4) for g in (32, 64, 128)]


@pytest.mark.parametrize("bits,G", ALL_BG)
@pytest.mark.parametrize("S,R", [(96, 0), (133, 10), (70, 3)])
def test_quant_parity_small(vq, oracle_mod, bits, G, S, R):
    k = _gen((2, 3, S), 11 + bits + G, outl=4)
    v = _gen((2, 3, S), 12 + bits + G)
    k[0, 1, :, 9] = 0.5  # a constant channel: constant key groups
    v[1, 2, 4, :] = -1.25  # a constant token: constant value groups
    out = vq.vq_kivi_quant_pack(_dev(k), _dev(v), bits, G, R)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    S_q = S - R
    _check_keys(out, oracle_mod.kivi_quant(k, bits, G, R, True), bits, G, S_q)
    _check_values(out, oracle_mod.kivi_quant(v, bits, G, R, False), bits, G)


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_exact_half_ties(vq, oracle_mod, bits):
    """Small-integer data puts many t = (x - min)(2^b - 1)/(max - min) exactly
    on half-integers; codes must follow ties-to-even exactly."""
    rng = np.random.default_rng(bits)
    G = 32
    lv = 2 * ((1 << bits) - 1)  # range of 2(2^b - 1) makes t = x/2: exact halves
    k = rng.integers(0, lv + 1, (1, 2, 64, D)).astype(np.float16)
    v = rng.integers(0, lv + 1, (1, 2, 64, D)).astype(np.float16)
    k[..., 0, :] = 0
    k[..., 1, :] = lv
    v[..., 0::G] = 0
    v[..., 1::G] = lv
    out = vq.vq_kivi_quant_pack(_dev(k), _dev(v), bits, G, 0)
    torch.cuda.synchronize()
    ok = oracle_mod.kivi_quant(k, bits, G, 0, True)
    ov = oracle_mod.kivi_quant(v, bits, G, 0, False)
    assert ok["tie"].mean() > 0.1 and ov["tie"].mean() > 0.1
    # ties here are exact, so the exact path must reproduce them: no mismatch at all
    _check_keys(out, ok, bits, G, 64, strict=True)
    _check_values(out, ov, bits, G, strict=True)


def test_residual_window_untouched_and_offsets(vq, oracle_mod):
    bits, G, R = 2, 32, 16
    B, H, S = 3, 2, 80
    S_q = S - R
    k = _gen((B, H, S), 21, outl=4)
    v = _gen((B, H, S), 22)
    off = np.array([0, 64, 128], np.int32)
    S_dst = 192
    shp = vq.kivi_shapes(B, H, S_dst, D, bits, G)
    outs = {
        "k_packed": torch.full(shp["k_packed"], 7, dtype=torch.int32, device="cuda"),
        "k_scale": torch.full(shp["k_scale"], 3.0, dtype=torch.float16, device="cuda"),
        "k_zero": torch.full(shp["k_scale"], 3.0, dtype=torch.float16, device="cuda"),
        "v_packed": torch.full(shp["v_packed"], 7, dtype=torch.int32, device="cuda"),
        "v_scale": torch.full(shp["v_scale"], 3.0, dtype=torch.float16, device="cuda"),
        "v_zero": torch.full(shp["v_scale"], 3.0, dtype=torch.float16, device="cuda"),
    }
    kd, vd = _dev(k), _dev(v)
    k_before = kd.clone()
    vq.vq_kivi_quant_pack(kd, vd, bits, G, R, outs=outs, dst_off=_dev(off), S_dst=S_dst)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    assert torch.equal(kd, k_before)  # inputs (and their residual window) are read-only
    ok = oracle_mod.kivi_quant(k, bits, G, R, True)
    ov = oracle_mod.kivi_quant(v, bits, G, R, False)
    NG = S_q // G
    for b in range(B):
        sub = {n: t[b:b + 1] for n, t in outs.items()}
        g0 = off[b] // G
        sk = {"k_packed": sub["k_packed"][:, :, g0:g0 + NG], "k_scale": sub["k_scale"][:, :, g0:g0 + NG],
              "k_zero": sub["k_zero"][:, :, g0:g0 + NG]}
        okb = {n: (a[b * H:(b + 1) * H] if isinstance(a, np.ndarray) else a) for n, a in ok.items()}
        _check_keys(sk, okb, bits, G, S_q)
        sv = {"v_packed": sub["v_packed"][:, :, off[b]:off[b] + S_q],
              "v_scale": sub["v_scale"][:, :, off[b]:off[b] + S_q],
              "v_zero": sub["v_zero"][:, :, off[b]:off[b] + S_q]}
        ovb = {n: (a[b * H:(b + 1) * H] if isinstance(a, np.ndarray) else a) for n, a in ov.items()}
        _check_values(sv, ovb, bits, G)
    # destination slots outside [off, off + S_q) are untouched
    vp = _np(outs["v_packed"])
    for b in range(B):
        mask = np.ones(S_dst, bool)
        mask[off[b]:off[b] + S_q] = False
        assert np.all(vp[b][:, mask] == 7)


def test_bad_offset_sets_device_error(vq):
    bits, G = 2, 32
    k = _gen((2, 1, 64), 31)
    off = _dev(np.array([0, 16], np.int32))  # not a multiple of G
    out = vq.vq_kivi_quant_pack(_dev(k), None, bits, G, 0, dst_off=off, S_dst=128)
    assert vq.vq_device_error() & vq.VQ_DEVERR_BAD_OFFSET
    assert vq.vq_device_error() == 0


@pytest.mark.parametrize("bits,G", ALL_BG)
def test_dequant_parity_bit_exact(vq, oracle_mod, bits, G):
    """GPU dequant of the oracle's packed storage vs the oracle's dequant."""
    S, R = 3 * G + 5, 0
    k = _gen((1, 3, S), 41 + bits, scale=3.0, outl=4)
    v = _gen((1, 3, S), 42 + bits, scale=0.5)
    ok = oracle_mod.kivi_quant(k, bits, G, R, True)
    ov = oracle_mod.kivi_quant(v, bits, G, R, False)
    S_q = ok["S_q"]
    packs = {
        "k_packed": _dev(ok["packed"].view(np.int32)), "k_scale": _dev(ok["scale"]),
        "k_zero": _dev(ok["zero"]), "v_packed": _dev(ov["packed"].view(np.int32)),
        "v_scale": _dev(ov["scale"]), "v_zero": _dev(ov["zero"]),
    }
    ko, vo = vq.vq_kivi_unpack_dequant(packs, 1, 3, S_q, bits, G)
    torch.cuda.synchronize()
    rk = oracle_mod.kivi_dequant(ok["packed"], ok["scale"], ok["zero"], 3, S_q, D, bits, G, True)
    rv = oracle_mod.kivi_dequant(ov["packed"], ov["scale"], ov["zero"], 3, S_q, D, bits, G, False)
    assert np.array_equal(_np(ko).reshape(3, S_q, D).view(np.uint16), rk.view(np.uint16))
    assert np.array_equal(_np(vo).reshape(3, S_q, D).view(np.uint16), rv.view(np.uint16))


def test_dequant_exact_rounding_edge(vq, oracle_mod):
    """A zero far below the scale makes q*scale + zero inexact in fp32; the
    result must still be the once-rounded fp16."""
    bits, G = 4, 32
    v = np.zeros((1, 1, 4, D), np.float16)
    v[..., :] = np.float16(2.0 ** -14 + 2.0 ** -24)
    v[..., 1::2] = np.float16(1000.0)
    ov = oracle_mod.kivi_quant(v, bits, G, 0, False)
    packs = {"v_packed": _dev(ov["packed"].view(np.int32)), "v_scale": _dev(ov["scale"]),
             "v_zero": _dev(ov["zero"])}
    _, vo = vq.vq_kivi_unpack_dequant(packs, 1, 1, 4, bits, G, want_k=False)
    rv = oracle_mod.kivi_dequant(ov["packed"], ov["scale"], ov["zero"], 1, 4, D, bits, G, False)
    assert np.array_equal(_np(vo).reshape(1, 4, D).view(np.uint16), rv.view(np.uint16))


def test_c2_full_parity(vq, oracle_mod):
    """KIVI 2-bit flush of K and V [1, 32, 4096, 128], G = 32, residual 128: all codes."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    cfg = synth.CONFIGS["c2_kivi_b2_32x4096"]
    k = synth.keys_for(cfg)
    v = synth.values_for(cfg)
    bits, G, R = cfg["bits"], cfg["group"], cfg["residual"]
    out = vq.vq_kivi_quant_pack(_dev(k), _dev(v), bits, G, R)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    ok = oracle_mod.kivi_quant(k, bits, G, R, True)
    ov = oracle_mod.kivi_quant(v, bits, G, R, False)
    _check_keys(out, ok, bits, G, ok["S_q"])
    _check_values(out, ov, bits, G)
    # round trip: GPU dequant of GPU storage equals the oracle dequant of the
    # oracle storage wherever the codes agree (they all do unless tie-flagged)
    ko, vo = vq.vq_kivi_unpack_dequant(out, 1, 32, ok["S_q"], bits, G)
    rk = oracle_mod.kivi_dequant(ok["packed"], ok["scale"], ok["zero"], 32, ok["S_q"], D, bits, G, True)
    rv = oracle_mod.kivi_dequant(ov["packed"], ov["scale"], ov["zero"], 32, ok["S_q"], D, bits, G, False)
    gk = _np(ko).reshape(rk.shape).view(np.uint16)
    gv = _np(vo).reshape(rv.shape).view(np.uint16)
    assert np.array_equal(gk[ok["tie"] == 0], rk.view(np.uint16)[ok["tie"] == 0])
    assert np.array_equal(gv[ov["tie"] == 0], rv.view(np.uint16)[ov["tie"] == 0])


def test_c4_decode_flush(vq, oracle_mod):
    """64 sequences x 8 heads: 128-token flushes at 128-aligned cache lengths."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    cfg = synth.CONFIGS["c4_decode_flush_64x8x128"]
    k = synth.keys_for(cfg)
    v = synth.values_for(cfg)
    off = synth.cache_lengths(cfg["B"], cfg["seed"])
    G, S_dst = cfg["group"], cfg["s_dst"]
    for bits in cfg["kivi_bits"]:
        out = vq.vq_kivi_quant_pack(_dev(k), _dev(v), bits, G, 0, dst_off=_dev(off), S_dst=S_dst)
        torch.cuda.synchronize()
        assert vq.vq_device_error() == 0
        for b in (0, 17, 63):
            ok = oracle_mod.kivi_quant(k[b:b + 1], bits, G, 0, True)
            ov = oracle_mod.kivi_quant(v[b:b + 1], bits, G, 0, False)
            g0 = off[b] // G
            sk = {n: out[n][b:b + 1, :, g0:g0 + 4] for n in ("k_packed", "k_scale", "k_zero")}
            _check_keys(sk, ok, bits, G, 128)
            sv = {n: out[n][b:b + 1, :, off[b]:off[b] + 128] for n in ("v_packed", "v_scale", "v_zero")}
            _check_values(sv, ov, bits, G)


def test_c5_full_size_sampled(vq, oracle_mod):
    """K and V [4, 32, 32768, 128] at full size, 2-bit G = 64, residual 128:
    sampled key groups and value rows checked against the oracle."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    cfg = synth.CONFIGS["c5_long_32k"]
    bits, G, R = cfg["kivi_bits"], cfg["group"], cfg["residual"]
    k = synth.keys_for(cfg)
    v = synth.values_for(cfg)
    out = vq.vq_kivi_quant_pack(_dev(k), _dev(v), bits, G, R)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    B, H, S, _ = k.shape
    S_q = S - R
    NG = S_q // G
    rng = np.random.default_rng(5)
    kp = out["k_packed"]
    for _ in range(40):
        b, h, g = rng.integers(0, B), rng.integers(0, H), rng.integers(0, NG)
        tile = k[b:b + 1, h:h + 1, g * G:(g + 1) * G]
        ok = oracle_mod.kivi_quant(tile, bits, G, 0, True)
        sk = {n: out[n][b:b + 1, h:h + 1, g:g + 1] for n in ("k_packed", "k_scale", "k_zero")}
        _check_keys(sk, ok, bits, G, G)
    for _ in range(40):
        b, h, s = rng.integers(0, B), rng.integers(0, H), rng.integers(0, S_q - 16)
        rows = v[b:b + 1, h:h + 1, s:s + 16]
        ov = oracle_mod.kivi_quant(rows, bits, G, 0, False)
        sv = {n: out[n][b:b + 1, h:h + 1, s:s + 16] for n in ("v_packed", "v_scale", "v_zero")}
        _check_values(sv, ov, bits, G)
    assert kp.shape == (B, H, NG, G * bits // 32, D)
