"""C-ABI checks that need no GPU: the library loads, exports every entry point
declared in include/vq.h, rejects bad arguments before touching the device,
and its host-side codebook generator agrees with the oracle's."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from kv_cache_quantization_turboquantrvq_gb300 import api, build
    build.build()
    return api.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "vq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vq_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n
    from kv_cache_quantization_turboquantrvq_gb300 import api
    assert sorted(api.EXPORTED) == names


def test_status_strings(L):
    from kv_cache_quantization_turboquantrvq_gb300 import api
    assert api.vq_status_str(0) == "VQ_OK"
    assert api.vq_status_str(3) == "VQ_ERR_MISALIGNED"
    assert "sm_103a" in api.vq_version()


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_codebook_generator_matches_oracle(L, oracle_mod, bits):
    from kv_cache_quantization_turboquantrvq_gb300 import api
    got = api.vq_rvq_codebook(128, bits)
    ref = oracle_mod.rvq_codebooks(128, bits)[:4]
    for g, r in zip(got, ref):
        # both are fp32 roundings of converged binary64 Lloyd-Max iterations
        assert np.all(np.abs(g.view(np.int32) - r.view(np.int32)) <= 1)


# ---------------------------------------------------------------- validation
# Fake device addresses: validation is pure host arithmetic and must return
# before any CUDA call, so these never reach the device.
A = 1 << 32  # 16-byte aligned fake address
P = ctypes.c_void_p


def _cb(bits):
    from kv_cache_quantization_turboquantrvq_gb300 import api
    return [np.ascontiguousarray(a) for a in api.vq_rvq_codebook(128, bits)]


def _enc(L, k=A, B=1, H=2, S=8, D=128, bits=2, cb=None, p1=A + (1 << 24), p2=A + (2 << 24),
         nrm=A + (3 << 24), off=None, S_dst=None):
    cb = cb or _cb(bits if bits in (1, 2, 4) else 2)
    return L.vq_rvq_encode_pack(P(k), B, H, S, D, bits, *[P(c.ctypes.data) for c in cb], P(p1), P(p2),
                                P(nrm), P(off), S if S_dst is None else S_dst, None)


def test_rvq_encode_validation(L):
    from kv_cache_quantization_turboquantrvq_gb300 import api
    assert _enc(L, D=96) == api.VQ_ERR_UNSUPPORTED   # not a power of two
    assert _enc(L, D=512) == api.VQ_ERR_UNSUPPORTED  # wider than the pages test
    assert _enc(L, bits=5) == api.VQ_ERR_INVALID_ARG
    assert _enc(L, B=-1) == api.VQ_ERR_INVALID_ARG
    assert _enc(L, k=0) == api.VQ_ERR_INVALID_ARG
    assert _enc(L, p1=0) == api.VQ_ERR_INVALID_ARG
    assert _enc(L, k=A + 8) == api.VQ_ERR_MISALIGNED
    assert _enc(L, p2=A + (2 << 24) + 4) == api.VQ_ERR_MISALIGNED
    assert _enc(L, nrm=A + (3 << 24) + 2) == api.VQ_ERR_MISALIGNED
    assert _enc(L, p1=A + 256) == api.VQ_ERR_ALIASING          # packed1 inside the input
    assert _enc(L, p2=A + (1 << 24) + 16) == api.VQ_ERR_ALIASING  # packed2 overlaps packed1
    assert _enc(L, S_dst=9) == api.VQ_ERR_INVALID_ARG  # no dst_off: S_dst must be S
    assert _enc(L, off=A + (4 << 24), S_dst=7) == api.VQ_ERR_INVALID_ARG
    assert _enc(L, off=A + (4 << 24) + 2, S_dst=16) == api.VQ_ERR_MISALIGNED
    assert _enc(L, S=0, k=0, p1=0, p2=0, nrm=0) == api.VQ_OK  # empty: nothing to do
    c1, b1, c2, b2 = _cb(2)
    bad = b1.copy()
    bad[1] = bad[0]  # not strictly increasing
    assert _enc(L, cb=[c1, bad, c2, b2]) == api.VQ_ERR_INVALID_ARG
    bad = b2.copy()
    bad[0] = c2[0]  # boundary not strictly between centroids
    assert _enc(L, cb=[c1, b1, c2, bad]) == api.VQ_ERR_INVALID_ARG
    bad = c1.copy()
    bad[2] = np.nan
    assert _enc(L, cb=[bad, b1, c2, b2]) == api.VQ_ERR_INVALID_ARG


def test_rvq_decode_validation(L):
    from kv_cache_quantization_turboquantrvq_gb300 import api
    c1, _, c2, _ = _cb(2)

    def dec(p1=A, p2=A + (1 << 24), n=A + (2 << 24), out=A + (3 << 24), D=128, bits=2, S=8):
        return L.vq_rvq_unpack_dequant(P(p1), P(p2), P(n), 1, 2, S, D, bits, P(c1.ctypes.data),
                                       P(c2.ctypes.data), P(out), None)
    assert dec(D=512) == api.VQ_ERR_UNSUPPORTED
    assert dec(D=48) == api.VQ_ERR_UNSUPPORTED
    assert dec(out=0) == api.VQ_ERR_INVALID_ARG
    assert dec(out=A + (3 << 24) + 8) == api.VQ_ERR_MISALIGNED
    assert dec(out=A + 64) == api.VQ_ERR_ALIASING
    assert dec(S=0, p1=0, p2=0, n=0, out=0) == api.VQ_OK


def test_kivi_validation(L):
    from kv_cache_quantization_turboquantrvq_gb300 import api

    def q(k=A, v=A + (1 << 26), bits=2, G=32, R=8, S=72, D=128, off=None, S_dst=None,
          kp=A + (2 << 26), ks=A + (3 << 26), kz=A + (4 << 26), vp=A + (5 << 26),
          vs=A + (6 << 26), vz=A + (7 << 26)):
        S_q = max(S - R, 0)
        return L.vq_kivi_quant_pack(P(k), P(v), 1, 2, S, D, bits, G, R, P(kp), P(ks), P(kz), P(vp),
                                    P(vs), P(vz), P(off), S_q if S_dst is None else S_dst, None)
    assert q(D=64) == api.VQ_ERR_UNSUPPORTED
    assert q(G=48) == api.VQ_ERR_INVALID_ARG      # does not divide D
    assert q(G=16, bits=1) == api.VQ_ERR_INVALID_ARG  # G*bits not a multiple of 32
    assert q(G=16, bits=2) == api.VQ_ERR_UNSUPPORTED
    assert q(R=-1) == api.VQ_ERR_INVALID_ARG
    assert q(k=0, v=0) == api.VQ_ERR_INVALID_ARG
    assert q(kp=0) == api.VQ_ERR_INVALID_ARG
    assert q(k=A + 8) == api.VQ_ERR_MISALIGNED
    assert q(ks=A + (3 << 26) + 4) == api.VQ_ERR_MISALIGNED
    assert q(vp=A + 1024) == api.VQ_ERR_ALIASING
    assert q(vz=A + (6 << 26)) == api.VQ_ERR_ALIASING  # v_zero == v_scale
    assert q(S_dst=100) == api.VQ_ERR_INVALID_ARG  # no dst_off: S_dst must be S_q
    assert q(off=A + (8 << 26), S_dst=10) == api.VQ_ERR_INVALID_ARG
    assert q(R=72) == api.VQ_OK  # everything is residual: nothing to flush
    assert q(R=100) == api.VQ_OK


def test_device_error_rejects_null(L):
    from kv_cache_quantization_turboquantrvq_gb300 import api
    assert L.vq_device_error(None, None) == api.VQ_ERR_INVALID_ARG


def test_qjl_validation(L):
    """vq_qjl_encode refuses bad shapes, pointers, alignment and overlaps on
    the host (fake addresses: only refused cases are called)."""
    from kv_cache_quantization_turboquantrvq_gb300 import api

    def q(x=A, s=A + (1 << 26), p=A + (2 << 26), n=A + (3 << 26), N=64, D=128, m=128):
        return L.vq_qjl_encode(P(x), N, D, P(s), m, P(p), P(n), None)
    assert q(D=64) == api.VQ_ERR_UNSUPPORTED
    assert q(m=48) == api.VQ_ERR_UNSUPPORTED       # not a multiple of 32
    assert q(m=512) == api.VQ_ERR_UNSUPPORTED      # above 256
    assert q(m=0) == api.VQ_ERR_INVALID_ARG
    assert q(N=-1) == api.VQ_ERR_INVALID_ARG
    assert q(x=0) == api.VQ_ERR_INVALID_ARG
    assert q(n=0) == api.VQ_ERR_INVALID_ARG
    assert q(x=A + 8) == api.VQ_ERR_MISALIGNED
    assert q(n=A + (3 << 26) + 2) == api.VQ_ERR_MISALIGNED
    assert q(p=A + 1024) == api.VQ_ERR_ALIASING    # packed over the keys
    assert q(n=A + (2 << 26)) == api.VQ_ERR_ALIASING  # norms over packed
    assert q(N=0, x=0, p=0, n=0) == api.VQ_OK       # nothing to do


def test_flush_decode_validation(L):
    """vq_flush_decode refuses bad parts, shapes, alignment and overlaps on the
    host (fake addresses: only refused cases and an empty call reach it)."""
    from kv_cache_quantization_turboquantrvq_gb300 import api
    cb2 = _cb(2)
    M = 1 << 26

    def f(k=A, v=A + M, B=2, H=2, T=40, D=128, R=8, off=None, S_dst=None, rb=2, cb=cb2,
          p1=A + 2 * M, p2=A + 3 * M, nr=A + 4 * M, kb=2, G=32, kp=A + 5 * M, ks=A + 6 * M, kz=A + 7 * M,
          vp=A + 8 * M, vs=A + 9 * M, vz=A + 10 * M, kw=A + 11 * M, vw=A + 12 * M, woff=None, R_cap=8):
        S_q = T - R
        cbp = [None] * 4 if cb is None else [P(c.ctypes.data) for c in cb]
        return L.vq_flush_decode(P(k), P(v), B, H, T, D, R, P(off), S_q if S_dst is None else S_dst, rb, *cbp,
                                 P(p1), P(p2), P(nr), kb, G, P(kp), P(ks), P(kz), P(vp), P(vs), P(vz),
                                 P(kw), P(vw), P(woff), R_cap, None)
    none = dict(p1=0, kp=0, vp=0, kw=0, vw=0)
    assert f(**none) == api.VQ_ERR_INVALID_ARG                     # no part at all
    assert f(D=64) == api.VQ_ERR_UNSUPPORTED
    assert f(R=41) == api.VQ_ERR_INVALID_ARG                       # window longer than the block
    assert f(k=0) == api.VQ_ERR_INVALID_ARG                        # keys' parts need k
    assert f(v=0) == api.VQ_ERR_INVALID_ARG                        # values' parts need v
    assert f(rb=3) == api.VQ_ERR_INVALID_ARG
    assert f(cb=None) == api.VQ_ERR_INVALID_ARG
    c1, b1, c2, b2 = cb2
    asym = c1.copy()
    asym[3] *= np.float32(1.5)
    assert f(cb=[asym, b1, c2, b2]) == api.VQ_ERR_UNSUPPORTED       # not the library's kind of book
    assert f(kb=1, G=32) == api.VQ_ERR_UNSUPPORTED
    assert f(G=128) == api.VQ_ERR_UNSUPPORTED
    assert f(R_cap=4) == api.VQ_ERR_INVALID_ARG                    # window capacity below R
    assert f(S_dst=50) == api.VQ_ERR_INVALID_ARG                   # no dst_off: S_dst must be T - R
    assert f(k=A + 8) == api.VQ_ERR_MISALIGNED
    assert f(nr=A + 4 * M + 2) == api.VQ_ERR_MISALIGNED
    assert f(kw=A + 11 * M + 8) == api.VQ_ERR_MISALIGNED
    assert f(p1=A + 512) == api.VQ_ERR_ALIASING                    # packed1 inside the keys
    assert f(vw=A + 11 * M + 64) == api.VQ_ERR_ALIASING            # the two windows overlap
    assert f(vs=A + 5 * M) == api.VQ_ERR_ALIASING                  # v_scale over k_packed
    assert f(B=0) == api.VQ_OK                                     # nothing to do
