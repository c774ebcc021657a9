"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: textbook
tables, closed forms, exact rational arithmetic, library routines (numpy's
binary16 conversion, scipy's Sylvester Hadamard and quadrature), brute force
on tiny inputs, or invariants of the method.  Chosen so that a dropped term,
a wrong sign or index, a transposed operand or a wrong rounding rule fails one.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":")
            rows[int(k)] = [float(t) for t in v.split()]
    return rows


def _read_bars(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            out.append([p.strip() for p in line.split("|")])
    return out


# ------------------------------------------------------------------ binary16


def test_f16_to_f64_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.f16_to_f64(int(b)) for b in bits[::7]])
    r = ref[::7]
    fin = np.isfinite(r)
    assert np.array_equal(got[fin], r[fin])
    assert np.array_equal(np.isnan(got), np.isnan(r))


def test_f64_to_f16_matches_numpy_rne(oracle_mod):
    rng = np.random.default_rng(7)
    # random magnitudes over the whole binary16 range, plus exact midpoints
    x = rng.standard_normal(4000) * np.exp(rng.uniform(-20, 11, 4000))
    h = rng.integers(0, 0x7bff, 2000).astype(np.uint16).view(np.float16).astype(np.float64)
    h2 = (rng.integers(0, 0x7bff, 2000).astype(np.uint16) + 1).view(np.float16).astype(np.float64)
    mids = 0.5 * (h + h2)  # halfway points between neighbours: tie cases
    vals = np.concatenate([x, mids, -mids, [0.0, -0.0, 65504.0, 65519.99, 65520.0, 6e-8, 3e-8]])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle_mod.f64_to_f16_rn(v) for v in vals], np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ Hadamard


def test_hadamard_is_sylvester_and_orthogonal(oracle_mod):
    from scipy.linalg import hadamard
    for D in (2, 8, 64, 128):
        H = oracle_mod.hadamard_matrix(D)
        assert np.array_equal(H, hadamard(D).astype(np.float64))
        assert np.array_equal(H @ H.T, D * np.eye(D))
        assert np.array_equal(H, H.T)


def _pages_butterfly(x):
    """The range-based parallel butterfly of the tag "turboquant" page,
    "Kernel 3: Fused Hadamard + Quantize": at each stride the lower lane takes
    a + b and the upper lane b - a, where a is its own value and b its
    partner's; run sequentially on a copy, which is what the barriers ensure."""
    v = np.array(x, dtype=np.float64)
    D = len(v)
    stride = 1
    while stride < D:
        new = v.copy()
        for lane in range(D):
            local = lane % (2 * stride)
            upper = local >= stride
            partner = lane - stride if upper else lane + stride
            a, b = v[lane], v[partner]
            new[lane] = (b - a) if upper else (a + b)
        v = new
        stride *= 2
    return v


def test_hadamard_matrix_equals_pages_butterfly(oracle_mod):
    rng = np.random.default_rng(3)
    H = oracle_mod.hadamard_matrix(128)
    for _ in range(3):
        x = rng.standard_normal(128)
        assert np.allclose(H @ x, _pages_butterfly(x), rtol=0, atol=1e-12)


# ------------------------------------------------------------------ codebooks


@pytest.mark.parametrize("levels", [2, 4, 8, 16])
def test_gaussian_lloyd_max_matches_max_1960(oracle_mod, levels):
    table = _read_table("max1960_gaussian.txt")[levels]
    c = oracle_mod.lloyd_max_gaussian(levels, 1.0)
    assert np.allclose(c[levels // 2:], table, atol=1.5e-4)
    assert np.array_equal(c, -c[::-1])


@pytest.mark.parametrize("levels", [2, 4, 16])
def test_laplace_lloyd_max_matches_paez_glisson(oracle_mod, levels):
    table = _read_table("paez_glisson_laplace.txt")[levels]
    beta = 1.0 / np.sqrt(2.0)
    c = oracle_mod.lloyd_max_laplace(levels, beta)
    assert np.allclose(c[levels // 2:], table, atol=1.5e-4)


def test_laplace_two_level_is_plus_minus_beta(oracle_mod):
    for beta in (0.01, 0.3, 2.0):
        c = oracle_mod.lloyd_max_laplace(2, beta)
        assert np.allclose(c, [-beta, beta], rtol=1e-13, atol=0)


@pytest.mark.parametrize("levels", [4, 16])
def test_lloyd_max_fixed_point_by_quadrature(oracle_mod, levels):
    """Each centroid is the conditional mean of its midpoint cell, computed by
    scipy quadrature (independent of the oracle's closed forms)."""
    from scipy import integrate, stats
    sigma = 1 / np.sqrt(128)
    c = oracle_mod.lloyd_max_gaussian(levels, sigma)
    edges = np.concatenate([[-np.inf], 0.5 * (c[1:] + c[:-1]), [np.inf]])
    pdf = stats.norm(scale=sigma).pdf
    for k in range(levels):
        lo, hi = edges[k], edges[k + 1]
        m = integrate.quad(lambda y: y * pdf(y), lo, hi, epsabs=1e-15)[0]
        p = integrate.quad(pdf, lo, hi, epsabs=1e-15)[0]
        assert abs(m / p - c[k]) < 1e-10 * max(1, abs(c[k]) / sigma) * sigma
    beta = 0.05
    c = oracle_mod.lloyd_max_laplace(levels, beta)
    edges = np.concatenate([[-np.inf], 0.5 * (c[1:] + c[:-1]), [np.inf]])
    lpdf = stats.laplace(scale=beta).pdf
    for k in range(levels):
        lo, hi = edges[k], edges[k + 1]
        pts = [0.0] if lo < 0 < hi else None
        m = integrate.quad(lambda y: y * lpdf(y), lo, hi, points=pts if not np.isinf(lo) and not np.isinf(hi) else None, epsabs=1e-15)[0]
        p = integrate.quad(lpdf, lo, hi, epsabs=1e-15)[0]
        assert abs(m / p - c[k]) < 1e-9 * beta


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_stage2_beta_is_mean_abs_residual(oracle_mod, bits):
    """beta = E|Y - c1[i(Y)]|, Y ~ N(0, 1/D): quadrature and Monte Carlo."""
    from scipy import integrate, stats
    D = 128
    sigma = 1 / np.sqrt(D)
    L = 1 << bits
    c = oracle_mod.lloyd_max_gaussian(L, sigma)
    beta = oracle_mod.stage1_residual_mean_abs(c, sigma)
    edges = np.concatenate([[-np.inf], 0.5 * (c[1:] + c[:-1]), [np.inf]])
    pdf = stats.norm(scale=sigma).pdf
    q = 0.0
    for k in range(L):
        q += integrate.quad(lambda y: abs(y - c[k]) * pdf(y), edges[k], edges[k + 1],
                            points=None if np.isinf(edges[k]) or np.isinf(edges[k + 1]) else [c[k]],
                            epsabs=1e-14)[0]
    assert abs(q - beta) < 1e-11
    rng = np.random.default_rng(11)
    y = rng.standard_normal(2_000_000) * sigma
    idx = np.searchsorted(0.5 * (c[1:] + c[:-1]), y, side="left")
    mc = np.mean(np.abs(y - c[idx]))
    assert abs(mc - beta) < 5e-4 * sigma * 10


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_rvq_codebooks_structure(oracle_mod, bits):
    c1, b1, c2, b2, beta = oracle_mod.rvq_codebooks(128, bits)
    L = 1 << bits
    assert c1.dtype == np.float32 and len(c1) == L and len(b1) == L - 1
    for c, b in ((c1, b1), (c2, b2)):
        assert np.all(np.diff(c) > 0) and np.all(np.diff(b) > 0)
        assert np.array_equal(c, -c[::-1]) and np.array_equal(b, -b[::-1])
        assert np.all(b > c[:-1]) and np.all(b < c[1:])
        mid = 0.5 * (c[:-1].astype(np.float64) + c[1:].astype(np.float64))
        assert np.all(np.abs(b - mid) <= np.spacing(np.abs(b)).astype(np.float64))
    # stage 1 is the Max table scaled by sigma = 1/sqrt(D)
    table = _read_table("max1960_gaussian.txt")[L]
    assert np.allclose(c1[L // 2:] * np.sqrt(128), table, atol=1.5e-4)
    # stage 2 is the unit-variance Laplace table scaled to the fitted beta
    if L in (2, 4, 16):
        t2 = np.array(_read_table("paez_glisson_laplace.txt")[L])
        assert np.allclose(c2[L // 2:] / (beta * np.sqrt(2)), t2, atol=1.5e-4)


# ------------------------------------------------------------------ packing


def test_pack_golden_words(oracle_mod):
    for bits, codes, word in _read_bars("pack_words.txt"):
        bits = int(bits)
        codes = np.array([int(c) for c in codes.split()], np.uint8)
        got = oracle_mod.pack_lsb_first(codes, bits)
        assert got.tolist() == [int(word, 16)]


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_pack_unpack_identity_and_byte_order(oracle_mod, bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, 128 * 5).astype(np.uint8)
    words = oracle_mod.pack_lsb_first(codes, bits)
    assert np.array_equal(oracle_mod.unpack_lsb_first(words, len(codes), bits), codes)
    # the byte packer of the tag "turboquant" page, "Kernel 1: Bit-Packing":
    # one output byte per thread, element i of the byte at shift i * bits.
    per_byte = 8 // bits
    byts = np.zeros(len(codes) // per_byte, np.uint8)
    for bi in range(len(byts)):
        acc = 0
        for i in range(per_byte):
            acc |= int(codes[bi * per_byte + i]) << (i * bits)
        byts[bi] = acc
    assert np.array_equal(words.view(np.uint8), byts)  # little-endian words


# ------------------------------------------------------------------ RVQ


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_boundary_count_equals_argmin(oracle_mod, bits):
    """idx = #{k: y > b_k} is the nearest centroid (ties to the lower index),
    brute-forced on a fine grid that includes every boundary exactly."""
    c1, b1, c2, b2, _ = oracle_mod.rvq_codebooks(128, bits)
    D = 128
    grid = np.concatenate([np.linspace(-0.4, 0.4, 20001), b1.astype(np.float64),
                           np.nextafter(b1, np.inf).astype(np.float64)])
    count = (grid[:, None] > b1.astype(np.float64)[None, :]).sum(1)
    dist = np.abs(grid[:, None] - c1.astype(np.float64)[None, :])
    # boundaries are the fp32-rounded midpoints, so compare on points whose
    # nearest centroid is not tied within that rounding
    srt = np.sort(dist, axis=1)
    clear = (srt[:, 1] - srt[:, 0]) > 1e-7
    assert np.array_equal(count[clear], np.argmin(dist, axis=1)[clear])
    # the oracle's encode applies this rule: a row whose rotation is the
    # constant 1/sqrt(D) (x = e_0) gets count(1/sqrt(D) > b1) everywhere
    x = np.zeros((1, D), np.float16)
    x[0, 0] = 1.0
    out = oracle_mod.rvq_encode(x, bits, c1, b1, c2, b2, want_values=True)
    y0 = 1 / np.sqrt(D)
    assert np.allclose(out["y"], y0, rtol=0, atol=1e-15)
    assert np.all(out["idx1"] == (y0 > b1.astype(np.float64)).sum())
    r0 = y0 - np.float64(c1[(y0 > b1.astype(np.float64)).sum()])
    assert np.all(out["idx2"] == (r0 > b2.astype(np.float64)).sum())
    assert out["norms"][0] == 1.0


def test_rvq_encode_strict_greater_at_exact_boundary(oracle_mod):
    """y exactly on a boundary counts as not above it (strict >)."""
    bits = 2
    c1, b1, c2, b2, _ = oracle_mod.rvq_codebooks(128, bits)
    x = np.zeros((1, 128), np.float16)
    x[0, 0] = 1.0  # y = 1/sqrt(128) everywhere
    y0 = np.float32(1 / np.sqrt(128.0))
    b1x = np.array([-1.0, y0, 1.0], np.float32)  # boundary at y0 (fp32 of y0)
    out = oracle_mod.rvq_encode(x, bits, c1, b1x, c2, b2, want_values=True)
    expect = 1 if out["y"][0, 0] <= float(y0) else 2
    assert np.all(out["idx1"] == expect)
    assert np.all(out["tie1"] == 1) and np.all(out["tie2"] == 1)


@pytest.mark.parametrize("D,bits", [(128, 1), (128, 2), (128, 3), (128, 4), (8, 3), (16, 1), (32, 4),
                                    (64, 2), (64, 3), (256, 3), (256, 4)])
def test_rvq_encode_invariants(oracle_mod, D, bits):
    c1, b1, c2, b2, _ = oracle_mod.rvq_codebooks(D, bits)
    rng = np.random.default_rng(100 + bits + D)
    x = (rng.standard_normal((64, D)) * 0.7).astype(np.float16)
    o = oracle_mod.rvq_encode(x, bits, c1, b1, c2, b2, want_values=True)
    # norm and rotation preserve length
    n = np.sqrt((x.astype(np.float64) ** 2).sum(1))
    assert np.array_equal(o["norms"], n.astype(np.float32))
    assert np.allclose((o["y"] ** 2).sum(1), 1.0, rtol=0, atol=1e-13)
    # scaling the row by a power of two changes only the norm
    o2 = oracle_mod.rvq_encode((x.astype(np.float32) * 4).astype(np.float16), bits,
                               c1, b1, c2, b2)
    assert np.array_equal(o2["packed1"], o["packed1"])
    assert np.array_equal(o2["packed2"], o["packed2"])
    assert np.array_equal(o2["norms"], o["norms"] * 4)
    # negating the row mirrors the codes (symmetric codebooks), except at ties
    o3 = oracle_mod.rvq_encode(-x, bits, c1, b1, c2, b2)
    L = (1 << bits) - 1
    clean = (o["tie2"] == 0) & (o3["tie2"] == 0)
    assert np.array_equal(o3["idx1"][clean], (L - o["idx1"])[clean])
    assert np.array_equal(o3["idx2"][clean], (L - o["idx2"])[clean])
    # packed words are the LSB-first packing of each row's index streams
    for k in ("1", "2"):
        rows = np.stack([oracle_mod.pack_lsb_first(r, bits) for r in o["idx" + k]])
        assert np.array_equal(o["packed" + k], rows)
    # words per row: ceil(D / floor(32/b)) (b = 3: ten codes per word)
    assert o["packed1"].shape == (64, -(-D // (32 // bits)))
    # zero row: u = 0, so y = 0 and every code counts the negative boundaries
    z = oracle_mod.rvq_encode(np.zeros((1, D), np.float16), bits, c1, b1, c2, b2)
    assert z["norms"][0] == 0
    assert np.all(z["idx1"] == (0.0 > b1).sum())


@pytest.mark.parametrize("bits", [2, 4])
def test_rvq_roundtrip_from_centroid_rows(oracle_mod, bits):
    """Rows built in the rotated domain from chosen codes: y_hat = c1[i1] +
    c2[i2], x = n H y_hat / sqrt(D) (rounded to fp16).  Encoding returns the
    chosen codes wherever y_hat is clear of every boundary, and decoding
    returns x to within the fp16 rounding."""
    D = 128
    c1, b1, c2, b2, _ = oracle_mod.rvq_codebooks(D, bits)
    H = oracle_mod.hadamard_matrix(D)
    rng = np.random.default_rng(5)
    L = 1 << bits
    i1 = rng.integers(0, L, (16, D))
    i2 = rng.integers(L // 2 - 1, L // 2 + 1, (16, D))  # small stage-2 offsets
    yh = c1[i1].astype(np.float64) + c2[i2].astype(np.float64)
    yh /= np.linalg.norm(yh, axis=1, keepdims=True)  # unit rotated rows
    n = 3.0
    x = (n * (yh @ H.T) / np.sqrt(D)).astype(np.float16)
    o = oracle_mod.rvq_encode(x, bits, c1, b1, c2, b2, want_values=True)
    assert np.allclose(o["y"], yh, atol=2e-3)
    b1d = b1.astype(np.float64)
    margin1 = np.min(np.abs(yh[..., None] - b1d), axis=-1)
    exp1 = (yh[..., None] > b1d).sum(-1)
    clear = margin1 > 5e-3
    assert clear.sum() > 100
    assert np.array_equal(o["idx1"][clear], exp1[clear])
    dec = oracle_mod.rvq_decode(o["packed1"], o["packed2"], o["norms"], D, bits, c1, c2)
    rec = (c1[o["idx1"]].astype(np.float64) + c2[o["idx2"]].astype(np.float64))
    xr = o["norms"][:, None].astype(np.float64) * (rec @ H.T) / np.sqrt(D)
    assert np.array_equal(dec, xr.astype(np.float16))


def test_rvq_decode_inverts_rotation(oracle_mod):
    """decode(encode(x)) approximates x (quantizer distortion only), and the
    decode is linear in the norm."""
    D, bits = 128, 4
    c1, b1, c2, b2, _ = oracle_mod.rvq_codebooks(D, bits)
    rng = np.random.default_rng(9)
    x = rng.standard_normal((32, D)).astype(np.float16)
    o = oracle_mod.rvq_encode(x, bits, c1, b1, c2, b2)
    dec, f64 = oracle_mod.rvq_decode(o["packed1"], o["packed2"], o["norms"], D, bits, c1, c2,
                                     want_f64=True)
    xd = x.astype(np.float64)
    rel = np.linalg.norm(f64 - xd, axis=1) / np.linalg.norm(xd, axis=1)
    # 8 bits per coordinate in two stages; rows with a rotated coordinate far
    # in the Gaussian tail are clipped by the outermost centroids
    assert np.median(rel) < 0.015 and np.all(rel < 0.2)
    cos = (f64 * xd).sum(1) / np.linalg.norm(f64, axis=1) / np.linalg.norm(xd, axis=1)
    assert np.median(cos) > 0.9998
    dec2, f2 = oracle_mod.rvq_decode(o["packed1"], o["packed2"], o["norms"] * 2, D, bits, c1, c2,
                                     want_f64=True)
    assert np.allclose(f2, 2 * f64, rtol=1e-15, atol=0)


# ------------------------------------------------------------------ KIVI


def _exact_kivi_group(vals, bits):
    """Exact rational KIVI quantization of one group (Python Fractions)."""
    fr = [Fraction(float(v)) for v in vals]
    mn, mx = min(fr), max(fr)
    levels = (1 << bits) - 1
    if mn == mx:
        return [0] * len(fr), 0.0, float(mn)
    q = []
    for v in fr:
        t = (v - mn) * levels / (mx - mn)
        q.append(min(max(round(t), 0), levels))  # Python round: half to even
    scale32 = np.float32(float(Fraction(mx - mn) / levels))  # float() is correctly rounded
    return q, float(np.float16(scale32)), float(mn)


def test_kivi_half_even_golden(oracle_mod):
    for bits, vals, codes in _read_bars("kivi_half_even.txt"):
        bits = int(bits)
        v = np.array([float(t) for t in vals.split()], np.float16)
        x = v.reshape(1, 1, -1, 1)
        o = oracle_mod.kivi_quant(x, bits, len(v), 0, per_channel=True)
        assert o["codes"].ravel().tolist() == [int(c) for c in codes.split()]
        assert np.all(o["tie"].ravel()[np.mod(v.astype(np.float64), 1) == 0.5] == 1)


@pytest.mark.parametrize("bits,G", [(2, 32), (4, 32), (1, 32), (2, 64)])
@pytest.mark.parametrize("per_channel", [True, False])
def test_kivi_quant_matches_exact_rationals(oracle_mod, bits, G, per_channel):
    rng = np.random.default_rng(bits * 10 + G + per_channel)
    S, R = 2 * G + 7, 5  # ragged last key group
    x = (rng.standard_normal((1, 2, S, 128)) * rng.uniform(0.1, 4)).astype(np.float16)
    x[0, 1, :, 3] = 0.75  # constant key groups in one channel
    x[0, 1, 4, 64:64 + G] = -2.0  # one constant value group
    o = oracle_mod.kivi_quant(x, bits, G, R, per_channel)
    S_q = S - R
    xs = x.reshape(2, S, 128)[:, :S_q].astype(np.float64)
    checked = 0
    for bh in range(2):
        if per_channel:
            for g in range((S_q + G - 1) // G):
                for d in range(0, 128, 9):
                    vals = xs[bh, g * G:(g + 1) * G, d]
                    q, sc, ze = _exact_kivi_group(vals, bits)
                    assert o["codes"][bh, g * G:g * G + len(vals), d].tolist() == q
                    assert float(o["scale"][bh, g, d]) == sc
                    assert float(o["zero"][bh, g, d]) == ze
                    checked += 1
        else:
            for s in range(0, S_q, 5):
                for j in range(128 // G):
                    vals = xs[bh, s, j * G:(j + 1) * G]
                    q, sc, ze = _exact_kivi_group(vals, bits)
                    assert o["codes"][bh, s, j * G:(j + 1) * G].tolist() == q
                    assert float(o["scale"][bh, s, j]) == sc
                    assert float(o["zero"][bh, s, j]) == ze
                    checked += 1
    assert checked > 20


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_kivi_layouts_and_dequant(oracle_mod, bits):
    G = 32
    rng = np.random.default_rng(40 + bits)
    S, R = 3 * G + 11, 4
    x = rng.standard_normal((2, 1, S, 128)).astype(np.float16)
    for per_channel in (True, False):
        o = oracle_mod.kivi_quant(x, bits, G, R, per_channel)
        S_q = o["S_q"]
        codes = o["codes"]
        per = 32 // bits
        if per_channel:
            # word w of group g, channel d holds tokens g*G + w*per + j at shift j*bits
            p = o["packed"]
            for g in range(o["NG"]):
                for w in range(G * bits // 32):
                    for j in (0, per - 1):
                        s = g * G + w * per + j
                        v = (p[:, g, w, :] >> (j * bits)) & ((1 << bits) - 1)
                        expect = codes[:, s, :] if s < S_q else 0
                        assert np.array_equal(v, np.broadcast_to(expect, v.shape))
        else:
            words = o["packed"].reshape(-1)
            assert np.array_equal(words, oracle_mod.pack_lsb_first(codes.reshape(-1), bits))
        # min and max of every group reconstruct to within one fp16 step of the scale
        dq = oracle_mod.kivi_dequant(o["packed"], o["scale"], o["zero"], 2, S_q, 128, bits, G,
                                     per_channel)
        xs = x.reshape(2, S, 128)[:, :S_q].astype(np.float64)
        err = np.abs(dq.astype(np.float64) - xs)
        if per_channel:
            sc = np.repeat(o["scale"].astype(np.float64), G, axis=1)[:, :S_q]
        else:
            sc = np.repeat(o["scale"].astype(np.float64), G, axis=2)
        levels = (1 << bits) - 1
        # |x - x_hat| <= scale/2 + levels * (fp16 rounding of scale) + output rounding
        bound = sc * (0.5 + levels * 2 ** -11) + np.abs(xs) * 2 ** -10 + 1e-7
        assert np.all(err <= bound)
        # exact dequant formula on a sample, by rationals
        flat_q = codes.reshape(-1)
        i = rng.integers(0, flat_q.size, 50)
        for k in i:
            bh, s, d = np.unravel_index(k, codes.shape)
            if per_channel:
                scv, zev = o["scale"][bh, s // G, d], o["zero"][bh, s // G, d]
            else:
                scv, zev = o["scale"][bh, s, d // G], o["zero"][bh, s, d // G]
            v = Fraction(int(codes[bh, s, d])) * Fraction(float(scv)) + Fraction(float(zev))
            assert dq[bh, s, d] == np.float16(float(v))


@pytest.mark.parametrize("D", [8, 16, 32, 64, 256])
def test_rotation_closed_forms_at_other_widths(oracle_mod, D):
    """x = e_j gives y_i = (-1)^popcount(i & j) / sqrt(D) (column j of the
    Sylvester matrix), at every width the pages test."""
    c1, b1, c2, b2, _ = oracle_mod.rvq_codebooks(D, 2)
    for j in (0, D - 1, D // 3):
        x = np.zeros((1, D), np.float16)
        x[0, j] = -2.0
        y = oracle_mod.rvq_encode(x, 2, c1, b1, c2, b2, want_values=True)["y"][0]
        ref = np.array([-(-1.0) ** bin(i & j).count("1") for i in range(D)]) / np.sqrt(D)
        np.testing.assert_allclose(y, ref, rtol=0, atol=1e-15)


def test_three_bit_words_leave_the_top_bits_clear(oracle_mod):
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 8, 10 * 37).astype(np.uint8)
    words = oracle_mod.pack_lsb_first(codes, 3)
    assert len(words) == 37 and np.all(words >> 30 == 0)
    assert np.array_equal(oracle_mod.unpack_lsb_first(words, len(codes), 3), codes)
    # a row of D = 128 codes takes 13 words, the last holding 8 codes
    w = oracle_mod.pack_lsb_first(np.full(128, 7, np.uint8), 3)
    assert len(w) == 13 and w[-1] == (1 << 24) - 1


# ---------------------------------------------------------------- tie-band edges
#
# The tie flags decide which GPU mismatches the parity rule forgives, so the
# band's width, its strictness and its units are pinned from both sides: a
# value 0.9 band from a boundary (or a rounding tie) is flagged, one 1.1 band
# away is not.  Distances are checked with exact arithmetic first, so the
# fixtures themselves cannot drift.

RVQ_BAND = 1e-5
KIVI_BAND = 1e-4


def _e0_row():
    x = np.zeros((1, 128), np.float16)
    x[0, 0] = 1.0  # rotates to the constant 1/sqrt(128)
    return x


@pytest.mark.parametrize("frac", [0.9, -0.9, 1.1, -1.1])
def test_rvq_tie_band_edge_stage1(oracle_mod, frac):
    """A stage-1 boundary at y0 + frac * band (y0 = the rotated value of e_0):
    flagged at |frac| = 0.9, not at 1.1, and a stage-1 flag also flags the
    stage-2 code (its input depends on the stage-1 decision)."""
    bits = 2
    _, _, c2, b2, _ = oracle_mod.rvq_codebooks(128, bits)
    y0 = 1 / np.sqrt(128.0)
    b1 = np.array([-0.3, y0 + frac * RVQ_BAND, 0.3], np.float32)
    c1 = np.array([-0.5, 0.0, 0.2, 0.5], np.float32)
    out = oracle_mod.rvq_encode(_e0_row(), bits, c1, b1, c2, b2, want_values=True)
    y = out["y"][0]
    dist = np.abs(y - np.float64(b1[1]))
    assert np.all(np.abs(dist / RVQ_BAND - abs(frac)) < 0.01)  # fixture check
    # the residual is far from every stage-2 boundary: only propagation can flag it
    assert np.min(np.abs(out["r"][0][:, None] - b2.astype(np.float64)[None, :])) > 100 * RVQ_BAND
    flagged = abs(frac) < 1
    assert np.all(out["tie1"] == flagged)
    assert np.all(out["tie2"] == flagged)
    assert np.all(out["idx1"] == (1 if frac > 0 else 2))


@pytest.mark.parametrize("frac", [0.9, -0.9, 1.1, -1.1])
def test_rvq_tie_band_edge_stage2(oracle_mod, frac):
    """The residual r = y0 - c1[i1] placed frac * band from a stage-2 boundary,
    with y0 far from every stage-1 boundary: only tie2 follows the band."""
    bits = 2
    _, _, c2, b2, _ = oracle_mod.rvq_codebooks(128, bits)
    y0 = 1 / np.sqrt(128.0)
    target = np.float64(b2[2]) + frac * RVQ_BAND  # r = y0 - c  ->  c = y0 - target
    c1 = np.array([-0.5, -0.1, y0 - target, 0.5], np.float32)
    b1 = np.array([-0.3, 0.0, 0.3], np.float32)
    out = oracle_mod.rvq_encode(_e0_row(), bits, c1, b1, c2, b2, want_values=True)
    assert np.all(out["idx1"] == 2)
    r = out["r"][0]
    assert np.allclose(r, out["y"][0] - np.float64(c1[2]), rtol=0, atol=1e-17)
    assert np.all(np.abs(np.abs(r - np.float64(b2[2])) / RVQ_BAND - abs(frac)) < 0.01)
    flagged = abs(frac) < 1
    assert np.all(out["tie1"] == 0)
    assert np.all(out["tie2"] == flagged)
    assert np.all(out["idx2"] == (3 if frac > 0 else 2))


# (min, probe, max) fp16 groups whose exact t = (probe - min) (2^b - 1) / (max - min)
# lies the stated distance from a rounding tie k + 1/2; "big" groups have a
# scale near 667 (b = 2) or 133 (b = 4), "small" ones near 7e-4, so a flag
# measured in x units instead of t units would flip one of each pair.
KIVI_EDGES = [
    # bits, regime, frac of band, (min, probe, max)
    (2, "big", 0.9, (-0.11883544921875, 1000.0, 2000.0)),
    (2, "big", 1.1, (-0.145263671875, 1000.0, 2000.0)),
    (2, "small", 0.9, (-1.1920928955078125e-07, 0.0010004043579101562, 0.0020008087158203125)),
    (2, "small", 1.1, (-1.7881393432617188e-07, 0.0012073516845703125, 0.002414703369140625)),
    (4, "big", 0.9, (-0.023773193359375, 1000.0, 2000.0)),
    (4, "big", 1.1, (-0.029052734375, 1000.0, 2000.0)),
]


@pytest.mark.parametrize("per_channel", [True, False])
@pytest.mark.parametrize("bits,regime,frac,grp", KIVI_EDGES)
def test_kivi_tie_band_edge(oracle_mod, bits, regime, frac, grp, per_channel):
    mn, probe, mx = grp
    levels = (1 << bits) - 1
    t = Fraction(levels) * (Fraction(probe) - Fraction(mn)) / (Fraction(mx) - Fraction(mn))
    d = abs(t - (t.numerator // t.denominator) - Fraction(1, 2))
    assert abs(float(d) / KIVI_BAND - frac) < 0.02  # fixture check (exact arithmetic)
    G = 32
    # one group: min, max, the probe, the rest at the min (t = 0, far from a tie)
    g = np.full(G, mn, np.float64)
    g[1], g[2] = mx, probe
    g = g.astype(np.float16)
    assert [float(v) for v in g[:3]] == [mn, mx, probe]  # all exact in fp16
    if per_channel:
        x = np.zeros((1, 1, G, 128), np.float16)
        x[0, 0, :, 7] = g
        o = oracle_mod.kivi_quant(x, bits, G, 0, per_channel=True)
        tie = o["tie"][0, :, 7]
        code = o["codes"][0, 2, 7]
    else:
        x = np.zeros((1, 1, 1, 128), np.float16)
        x[0, 0, 0, 32:64] = g
        o = oracle_mod.kivi_quant(x, bits, G, 0, per_channel=False)
        tie = o["tie"][0, 0, 32:64]
        code = o["codes"][0, 0, 34]
    assert tie[2] == (1 if frac < 1 else 0)
    assert not tie[[0, 1]].any() and not tie[3:].any()
    assert code == round(t)  # Python round of a Fraction: nearest (not a tie here)
