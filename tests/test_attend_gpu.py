"""Decode-time attention over an RVQ key cache: CUDA path vs the oracle (GB300),
through the C ABI.

Inputs: the key cache is either encoded by the oracle from seeded keys or made
of seeded random code words (every bit pattern is a valid code for b in
{1, 2, 4}) with seeded row norms; values and queries are seeded fp16.
Codebooks are the oracle's.

Tolerance (derived from the arithmetic): the kernel forms each score in fp32
(a 128-term dot product of the fp32-rotated query with codebook sums, times
the row norm), so a score carries an absolute error of at most about 1e-5 for
these magnitudes; the weights then carry that relative error and the output,
a weighted mean of values, moves by at most that times 2 max|v|.  With the
final fp16 rounding every output must lie within half an fp16 ulp of the
oracle's exact (binary64) output plus 2e-5 * max|v|.  Most outputs must equal
the oracle's rounded fp16 bit for bit (the typical error is far below the
bound).
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


def _random_cache(B, Hkv, S, bits, seed):
    rng = np.random.default_rng(seed)
    W = D * bits // 32
    p1 = rng.integers(0, 2 ** 32, (B, Hkv, S, W), dtype=np.uint32)
    p2 = rng.integers(0, 2 ** 32, (B, Hkv, S, W), dtype=np.uint32)
    nr = rng.uniform(4.0, 24.0, (B, Hkv, S)).astype(np.float32)
    return p1, p2, nr


def _oracle_cache(oracle_mod, B, Hkv, S, bits, seed, cb):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    k = synth.kv_tensor(B, Hkv, S, D, seed, 4, 20.0)
    e = oracle_mod.rvq_encode(k.reshape(-1, D), bits, *cb[:4])
    W = D * bits // 32
    return (e["packed1"].reshape(B, Hkv, S, W), e["packed2"].reshape(B, Hkv, S, W),
            e["norms"].reshape(B, Hkv, S))


def _values(B, Hkv, S, seed):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    return synth.kv_tensor(B, Hkv, S, D, seed, 0, 1.0)


def _attend(vq, q, p1, p2, nr, v, bits, cb, scale, lens=None, **kw):
    out = vq.vq_rvq_attend(_dev(q), _dev(p1.view(np.int32)), _dev(p2.view(np.int32)), _dev(nr), _dev(v),
                           bits, cb[0], cb[2], scale, lens=None if lens is None else _dev(lens), **kw)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    return out.cpu().numpy()


def _check(o, ref16, ref64, v, min_exact=0.9):
    o = o.reshape(ref16.shape)
    half_ulp = 0.5 * np.spacing(np.abs(ref64).astype(np.float16)).astype(np.float64)
    tol = half_ulp + 2e-5 * float(np.abs(v.astype(np.float64)).max())
    err = np.abs(o.astype(np.float64) - ref64)
    assert np.all(err <= tol), "max excess %g" % float((err - tol).max())
    exact = float(np.mean(o.view(np.uint16) == ref16.view(np.uint16)))
    assert exact >= min_exact, exact
    return exact


@pytest.mark.parametrize("bits", [1, 2, 4])
@pytest.mark.parametrize("gq", [1, 2, 4, 8])
def test_attend_parity_encoded_cache(vq, oracle_mod, bits, gq):
    """Grouped-query ratios 1..8 over an oracle-encoded cache; one full and one
    ragged sequence (several key tiles and a tail)."""
    B, Hkv, S = 2, 2, 300
    cb = oracle_mod.rvq_codebooks(D, bits)
    p1, p2, nr = _oracle_cache(oracle_mod, B, Hkv, S, bits, 60 + 4 * bits + gq, cb)
    v = _values(B, Hkv, S, 61 + 4 * bits + gq)
    q = np.random.default_rng(7 + gq).standard_normal((B, Hkv * gq, D)).astype(np.float16)
    lens = np.array([S, 137], np.int32)
    scale = 1.0 / np.sqrt(D)
    o = _attend(vq, q, p1, p2, nr, v, bits, cb, scale, lens)
    r16, r64 = oracle_mod.rvq_attend(q, p1, p2, nr, v, bits, cb[0], cb[2], scale, lens=lens, want_f64=True)
    _check(o, r16, r64, v)


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_attend_parity_random_codes_no_lens(vq, oracle_mod, bits):
    """Random code words (all code values reached), no length vector, a
    sharper softmax (larger scale)."""
    B, Hkv, gq, S = 3, 2, 4, 1029
    cb = oracle_mod.rvq_codebooks(D, bits)
    p1, p2, nr = _random_cache(B, Hkv, S, bits, 70 + bits)
    v = _values(B, Hkv, S, 71 + bits)
    q = np.random.default_rng(72 + bits).standard_normal((B, Hkv * gq, D)).astype(np.float16)
    scale = 2.0 / np.sqrt(D)
    o = _attend(vq, q, p1, p2, nr, v, bits, cb, scale)
    r16, r64 = oracle_mod.rvq_attend(q, p1, p2, nr, v, bits, cb[0], cb[2], scale, want_f64=True)
    _check(o, r16, r64, v)


def test_attend_edge_lengths_and_splits(vq, oracle_mod):
    """Empty, one-token, ragged and full caches; the split-S path (workspace)
    and the single-pass path (no room in the workspace) both agree with the
    oracle, and an empty cache gives zeros."""
    bits, gq, B, Hkv, S = 2, 4, 5, 1, 700
    cb = oracle_mod.rvq_codebooks(D, bits)
    p1, p2, nr = _random_cache(B, Hkv, S, bits, 90)
    v = _values(B, Hkv, S, 91)
    q = np.random.default_rng(92).standard_normal((B, Hkv * gq, D)).astype(np.float16)
    lens = np.array([0, 1, 33, 700, 512], np.int32)
    scale = 0.9 / np.sqrt(D)
    r16, r64 = oracle_mod.rvq_attend(q, p1, p2, nr, v, bits, cb[0], cb[2], scale, lens=lens, want_f64=True)
    assert vq.vq_rvq_attend_workspace(B, Hkv * gq, Hkv, S) > 0
    full = _attend(vq, q, p1, p2, nr, v, bits, cb, scale, lens)
    one = _attend(vq, q, p1, p2, nr, v, bits, cb, scale, lens,
                  workspace=torch.empty(4, dtype=torch.float32, device="cuda"))
    _check(full, r16, r64, v)
    _check(one, r16, r64, v)
    assert np.all(full[0].astype(np.float32) == 0.0)
    assert np.array_equal(full[1].view(np.uint16), np.repeat(v[1:2, 0, 0], gq, 0).view(np.uint16))


def test_attend_lengths_beyond_capacity_are_clamped(vq, oracle_mod):
    bits, gq, B, Hkv, S = 1, 2, 2, 2, 64
    cb = oracle_mod.rvq_codebooks(D, bits)
    p1, p2, nr = _random_cache(B, Hkv, S, bits, 93)
    v = _values(B, Hkv, S, 94)
    q = np.random.default_rng(95).standard_normal((B, Hkv * gq, D)).astype(np.float16)
    lens = np.array([1000, -5], np.int32)
    o = _attend(vq, q, p1, p2, nr, v, bits, cb, 0.1, lens)
    r16, r64 = oracle_mod.rvq_attend(q, p1, p2, nr, v, bits, cb[0], cb[2], 0.1, lens=lens, want_f64=True)
    _check(o, r16, r64, v)
    assert np.all(o[1].astype(np.float32) == 0.0)


def test_attend_rejects_bad_arguments(vq, oracle_mod):
    from kv_cache_quantization_turboquantrvq_gb300.api import VQError
    bits, B, Hkv, S = 2, 1, 2, 16
    cb = oracle_mod.rvq_codebooks(D, bits)
    p1, p2, nr = _random_cache(B, Hkv, S, bits, 96)
    v = _values(B, Hkv, S, 97)
    q = np.zeros((B, 3, D), np.float16)  # 3 query heads over 2 kv heads
    with pytest.raises(VQError):
        _attend(vq, q, p1, p2, nr, v, bits, cb, 0.1)
    q = np.zeros((B, 4, D), np.float16)
    with pytest.raises(VQError):
        _attend(vq, q, p1, p2, nr, v, 3, cb, 0.1)
    bad = list(cb)
    bad[0] = np.array(cb[0], np.float32)
    bad[0][1] = np.nan
    with pytest.raises(VQError):
        _attend(vq, q, p1, p2, nr, v, bits, bad, 0.1)


def test_attend_decode_shape_sampled(vq, oracle_mod):
    """A decode-time batch shaped like the decode-flush workload (sequences
    with 8 kv heads, 32 query heads, caches of random lengths in [1k, 16k]):
    the oracle on sampled sequences."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    bits, B, Hkv, gq, S = 2, 16, 8, 4, 16384
    lens = synth.cache_lengths(B, 104)
    cb = oracle_mod.rvq_codebooks(D, bits)
    p1, p2, nr = _random_cache(B, Hkv, S, bits, 105)
    v = _values(B, Hkv, S, 106)
    q = np.random.default_rng(107).standard_normal((B, Hkv * gq, D)).astype(np.float16)
    scale = 1.0 / np.sqrt(D)
    o = _attend(vq, q, p1, p2, nr, v, bits, cb, scale, lens)
    for b in (0, 7, 15):
        L = int(lens[b])
        sl = slice(b, b + 1)
        r16, r64 = oracle_mod.rvq_attend(q[sl], p1[sl, :, :L], p2[sl, :, :L], nr[sl, :, :L], v[sl, :, :L],
                                         bits, cb[0], cb[2], scale, want_f64=True)
        _check(o[sl], r16, r64, v[sl, :, :L])


@pytest.mark.parametrize("bits,gq", [(1, 8), (2, 4), (4, 1)])
def test_attend_rows_past_length_may_hold_anything(vq, oracle_mod, bits, gq):
    """Rows past a sequence's length are never part of the result, whatever
    they hold: the device copy carries NaN and inf norms and values there
    (partial tiles read such rows into shared memory), the oracle sees the
    same cache with finite rows.  Outputs must match the oracle's."""
    B, Hkv, S = 3, 2, 512
    cb = oracle_mod.rvq_codebooks(D, bits)
    p1, p2, nr = _random_cache(B, Hkv, S, bits, 1100 + bits)
    v = _values(B, Hkv, S, 1101 + bits)
    q = np.random.default_rng(1102).standard_normal((B, Hkv * gq, D)).astype(np.float16)
    lens = np.array([500, 17, 1], np.int32)
    nr_bad, v_bad = nr.copy(), v.copy()
    for b, n in enumerate(lens):
        nr_bad[b, :, n:] = np.nan
        v_bad[b, :, n:, 0::2] = np.float16(np.nan)
        v_bad[b, :, n:, 1::2] = np.float16(np.inf)
    o = _attend(vq, q, p1, p2, nr_bad, v_bad, bits, cb, 0.2, lens=lens)
    r16, r64 = oracle_mod.rvq_attend(q, p1, p2, nr, v, bits, cb[0], cb[2], 0.2, lens=lens, want_f64=True)
    assert np.all(np.isfinite(o.astype(np.float64)))
    _check(o, r16, r64, v)
