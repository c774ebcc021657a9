"""Randomised-sign rotation (H diag(s)): CUDA path vs the oracle (GB300),
through the _rs entry points of the C ABI.  Same rules as the plain RVQ
parity tests (tests/parity.py); all-zero signs must reproduce the plain calls
bit for bit."""
import numpy as np
import pytest

from parity import check_rvq

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


def _signs(seed):
    return np.random.default_rng(seed).integers(0, 2 ** 32, 4, dtype=np.uint32)


def _rows(shape, seed, outliers=(4, 20.0)):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    B, H, S = shape
    return synth.kv_tensor(B, H, S, D, seed, outliers[0], outliers[1])


@pytest.mark.parametrize("bits", [1, 2, 4])
@pytest.mark.parametrize("shape", [(1, 1, 5), (2, 3, 700), (1, 4, 5000)])
def test_encode_rs_parity(vq, oracle_mod, bits, shape):
    x = _rows(shape, 500 + bits, outliers=(4, 40.0))
    signs = _signs(501 + bits)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    p1, p2, n = vq.vq_rvq_encode_pack(_dev(x), bits, *cb, signs=signs)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb, signs=signs)
    check_rvq(p1.cpu().numpy(), p2.cpu().numpy(), n.cpu().numpy(), ora, bits)


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_zero_signs_match_the_plain_calls(vq, oracle_mod, bits):
    x = _rows((2, 2, 333), 510 + bits)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    z = np.zeros(4, np.uint32)
    a = vq.vq_rvq_encode_pack(_dev(x), bits, *cb, signs=z)
    b = vq.vq_rvq_encode_pack(_dev(x), bits, *cb)
    for u, w in zip(a, b):
        assert torch.equal(u, w)
    da = vq.vq_rvq_unpack_dequant(*a, bits, cb[0], cb[2], signs=z)
    db = vq.vq_rvq_unpack_dequant(*b, bits, cb[0], cb[2])
    assert torch.equal(da, db)


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_decode_rs_parity_and_round_trip(vq, oracle_mod, bits):
    x = _rows((1, 3, 999), 520 + bits)
    signs = _signs(521 + bits)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb, signs=signs)
    ref, ref64 = oracle_mod.rvq_decode(ora["packed1"], ora["packed2"], ora["norms"], D, bits, cb[0], cb[2],
                                       want_f64=True, signs=signs)
    W = 4 * bits
    out = vq.vq_rvq_unpack_dequant(_dev(ora["packed1"].view(np.int32).reshape(1, 3, 999, W)),
                                   _dev(ora["packed2"].view(np.int32).reshape(1, 3, 999, W)),
                                   _dev(ora["norms"].reshape(1, 3, 999)), bits, cb[0], cb[2], signs=signs)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    got = out.cpu().numpy().reshape(-1, D).astype(np.float64)
    n = ora["norms"].astype(np.float64)[:, None]
    assert np.all(np.abs(got - ref64) <= 1e-3 * n + 1e-30)
    assert np.mean(got == ref.astype(np.float64)) > 0.95


@pytest.mark.parametrize("bits,gq", [(1, 8), (2, 4), (4, 1)])
def test_attend_rs_parity(vq, oracle_mod, bits, gq):
    B, Hkv, S = 2, 2, 600
    signs = _signs(530 + bits)
    cb = oracle_mod.rvq_codebooks(D, bits)
    k = _rows((B, Hkv, S), 531 + bits)
    e = oracle_mod.rvq_encode(k.reshape(-1, D), bits, *cb[:4], signs=signs)
    W = 4 * bits
    p1, p2, nr = (e["packed1"].reshape(B, Hkv, S, W), e["packed2"].reshape(B, Hkv, S, W),
                  e["norms"].reshape(B, Hkv, S))
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    v = synth.kv_tensor(B, Hkv, S, D, 532 + bits, 0, 1.0)
    q = np.random.default_rng(533).standard_normal((B, Hkv * gq, D)).astype(np.float16)
    lens = np.array([S, 321], np.int32)
    scale = 1.0 / np.sqrt(D)
    out = vq.vq_rvq_attend(_dev(q), _dev(p1.view(np.int32)), _dev(p2.view(np.int32)), _dev(nr), _dev(v), bits,
                           cb[0], cb[2], scale, lens=_dev(lens), signs=signs).cpu().numpy()
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    r16, r64 = oracle_mod.rvq_attend(q, p1, p2, nr, v, bits, cb[0], cb[2], scale, lens=lens, want_f64=True,
                                     signs=signs)
    tol = 0.5 * np.spacing(np.abs(r64).astype(np.float16)).astype(np.float64) + 2e-5 * float(np.abs(v).max())
    assert np.all(np.abs(out.astype(np.float64) - r64) <= tol)
    assert np.mean(out.view(np.uint16) == r16.view(np.uint16)) > 0.9


def test_rs_calls_refuse_missing_signs(vq):
    import ctypes
    L = vq.lib()
    A = ctypes.c_void_p(1 << 32)
    c = (ctypes.c_float * 4)(-0.1, -0.03, 0.03, 0.1)
    b = (ctypes.c_float * 3)(-0.06, 0.0, 0.06)
    st = L.vq_rvq_encode_pack_rs(A, 1, 1, 16, D, 2, c, b, c, b, A, A, A, None, 16, None, None)
    assert st == vq.VQ_ERR_INVALID_ARG
    st = L.vq_rvq_unpack_dequant_rs(A, A, A, 1, 1, 16, D, 2, c, c, None, A, None)
    assert st == vq.VQ_ERR_INVALID_ARG
