"""CPU oracle for the KV-cache flush codecs (TurboQuantRVQ, KIVI).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never loads it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain single-threaded C, IEEE binary64,
explicit Walsh-Hadamard matrix).  This module compiles it with gcc on first
use (or via :func:`build`) and wraps it for numpy arrays.  Each wrapper names
the page passage it follows; ``oracle.c`` carries the full citations.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    P = ctypes.c_void_p
    L = ctypes.c_long
    I = ctypes.c_int
    D = ctypes.c_double
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f64.restype = D
    lib.oracle_f64_to_f16_rn.argtypes = [D]
    lib.oracle_f64_to_f16_rn.restype = ctypes.c_uint16
    lib.oracle_hadamard_matrix.argtypes = [I, P]
    lib.oracle_lloyd_max_gaussian.argtypes = [I, D, P]
    lib.oracle_lloyd_max_gaussian.restype = I
    lib.oracle_lloyd_max_laplace.argtypes = [I, D, P]
    lib.oracle_lloyd_max_laplace.restype = I
    lib.oracle_stage1_residual_mean_abs.argtypes = [I, P, D]
    lib.oracle_stage1_residual_mean_abs.restype = D
    lib.oracle_rvq_codebooks.argtypes = [I, I, P, P, P, P, P]
    lib.oracle_rvq_codebooks.restype = I
    lib.oracle_pack_lsb_first.argtypes = [P, L, I, P]
    lib.oracle_unpack_lsb_first.argtypes = [P, L, I, P]
    lib.oracle_rvq_encode.argtypes = [P, L, I, I, P, P, P, P] + [P] * 10
    lib.oracle_rvq_decode.argtypes = [P, P, P, L, I, I, P, P, P, P, P]
    lib.oracle_rvq_attend.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, D, P, P, P]
    lib.oracle_kivi_quant.argtypes = [P, L, I, I, I, I, I, I, P, P, P, P, P]
    lib.oracle_kivi_dequant.argtypes = [P, P, P, L, I, I, I, I, I, P]
    lib.oracle_kivi_attend.argtypes = [P] * 11 + [I] * 8 + [D, P, P]
    lib.oracle_qjl_encode.argtypes = [P, L, I, P, I, P, P, P, P]
    _lib = lib
    return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- fp16 / H


def f16_to_f64(bits: int) -> float:
    """Exact value of one IEEE binary16 bit pattern."""
    return _load().oracle_f16_to_f64(int(bits))


def f64_to_f16_rn(x: float) -> int:
    """Bit pattern of the binary16 nearest to x (ties to even)."""
    return int(_load().oracle_f64_to_f16_rn(float(x)))


def hadamard_matrix(D: int) -> np.ndarray:
    """Sylvester-order Walsh-Hadamard matrix H[i, j] = (-1)^popcount(i & j)."""
    H = np.empty((D, D), np.float64)
    _load().oracle_hadamard_matrix(D, _p(H))
    return H


# ---------------------------------------------------------------- codebooks


def lloyd_max_gaussian(levels: int, sigma: float) -> np.ndarray:
    """Lloyd-Max centroids (ascending, binary64) for N(0, sigma^2)."""
    c = np.empty(levels, np.float64)
    it = _load().oracle_lloyd_max_gaussian(levels, sigma, _p(c))
    if it < 0:
        raise RuntimeError("Lloyd-Max (Gaussian) did not converge")
    return c


def lloyd_max_laplace(levels: int, beta: float) -> np.ndarray:
    """Lloyd-Max centroids (ascending, binary64) for Laplace(0, beta)."""
    c = np.empty(levels, np.float64)
    it = _load().oracle_lloyd_max_laplace(levels, beta, _p(c))
    if it < 0:
        raise RuntimeError("Lloyd-Max (Laplace) did not converge")
    return c


def stage1_residual_mean_abs(c: np.ndarray, sigma: float) -> float:
    """E|Y - c[i(Y)]| for Y ~ N(0, sigma^2) under the midpoint-boundary quantizer c."""
    c = _c(c, np.float64)
    return _load().oracle_stage1_residual_mean_abs(len(c), _p(c), sigma)


def rvq_codebooks(D: int, bits: int):
    """Stage-1 (Gaussian) and stage-2 (Laplace-fit) fp32 codebooks.

    Returns (c1, b1, c2, b2, beta): centroids [2^bits] and midpoint boundaries
    [2^bits - 1] for each stage, plus the fitted Laplace scale.
    """
    L = 1 << bits
    c1 = np.empty(L, np.float32)
    b1 = np.empty(L - 1, np.float32)
    c2 = np.empty(L, np.float32)
    b2 = np.empty(L - 1, np.float32)
    beta = ctypes.c_double()
    rc = _load().oracle_rvq_codebooks(D, bits, _p(c1), _p(b1), _p(c2), _p(b2),
                                      ctypes.cast(ctypes.pointer(beta), ctypes.c_void_p))
    if rc != 0:
        raise RuntimeError("codebook generation failed (%d)" % rc)
    return c1, b1, c2, b2, beta.value


# ---------------------------------------------------------------- packing


def pack_lsb_first(codes: np.ndarray, bits: int) -> np.ndarray:
    codes = _c(codes, np.uint8).ravel()
    per = 32 // bits
    words = np.empty((len(codes) + per - 1) // per, np.uint32)
    _load().oracle_pack_lsb_first(_p(codes), len(codes), bits, _p(words))
    return words


def unpack_lsb_first(words: np.ndarray, n: int, bits: int) -> np.ndarray:
    words = _c(words, np.uint32).ravel()
    codes = np.empty(n, np.uint8)
    _load().oracle_unpack_lsb_first(_p(words), n, bits, _p(codes))
    return codes


# ---------------------------------------------------------------- RVQ


def _signs(signs, D):
    """Sign words of the randomised-sign rotation (bit j: coordinate j negated), or None."""
    if signs is None:
        return None
    s = _c(signs, np.uint32).ravel()
    assert s.size == D // 32
    return s


def rvq_encode(x_f16: np.ndarray, bits: int, c1, b1, c2, b2, want_values: bool = False, signs=None):
    """TurboQuantRVQ encode of rows x [..., D] (fp16); `signs` (D/32 uint32
    words) selects the randomised-sign rotation H diag(s).

    Returns a dict with packed1, packed2 [N, D*bits/32] uint32, norms [N] fp32,
    idx1, idx2, tie1, tie2 [N, D] uint8 and, when want_values, y and r [N, D]
    binary64 (the rotated value and the stage-1 residual).
    """
    x = _c(x_f16, np.float16)
    D = x.shape[-1]
    N = x.size // D
    W = -(-D // (32 // bits))  # words per row: floor(32/b) codes each
    out = {
        "packed1": np.empty((N, W), np.uint32), "packed2": np.empty((N, W), np.uint32),
        "norms": np.empty(N, np.float32),
        "idx1": np.empty((N, D), np.uint8), "idx2": np.empty((N, D), np.uint8),
        "tie1": np.empty((N, D), np.uint8), "tie2": np.empty((N, D), np.uint8),
    }
    y = np.empty((N, D), np.float64) if want_values else None
    r = np.empty((N, D), np.float64) if want_values else None
    cb = [_c(v, np.float32) for v in (c1, b1, c2, b2)]
    _load().oracle_rvq_encode(_p(x.view(np.uint16)), N, D, bits, *[_p(v) for v in cb],
                              _p(out["idx1"]), _p(out["idx2"]), _p(out["packed1"]),
                              _p(out["packed2"]), _p(out["norms"]), _p(out["tie1"]),
                              _p(out["tie2"]), _p(y), _p(r), _p(_signs(signs, D)))
    if want_values:
        out["y"], out["r"] = y, r
    return out


def rvq_decode(packed1, packed2, norms, D: int, bits: int, c1, c2, want_f64: bool = False, signs=None):
    """TurboQuantRVQ unpack + dequant; returns fp16 [N, D] (and binary64 if asked)."""
    p1 = _c(packed1, np.uint32)
    p2 = _c(packed2, np.uint32)
    n = _c(norms, np.float32).ravel()
    N = n.size
    out = np.empty((N, D), np.float16)
    f64 = np.empty((N, D), np.float64) if want_f64 else None
    _load().oracle_rvq_decode(_p(p1), _p(p2), _p(n), N, D, bits, _p(_c(c1, np.float32)),
                              _p(_c(c2, np.float32)), _p(out.view(np.uint16)), _p(f64),
                              _p(_signs(signs, D)))
    return (out, f64) if want_f64 else out


def rvq_attend(q, packed1, packed2, norms, v, bits: int, c1, c2, scale: float, lens=None,
               want_f64: bool = False, signs=None):
    """Decode-time attention over an RVQ key cache (see oracle.c).
    q [B, Hq, D] fp16; packed1/2 [B, Hkv, S_cap, W] uint32; norms [B, Hkv, S_cap] fp32;
    v [B, Hkv, S_cap, D] fp16; lens [B] int32 or None.  Returns fp16 [B, Hq, D]
    (and binary64 if asked)."""
    qa = _c(q, np.float16)
    B, Hq, D = qa.shape
    p1 = _c(packed1, np.uint32)
    p2 = _c(packed2, np.uint32)
    _, Hkv, S_cap, _ = p1.shape
    nr = _c(norms, np.float32)
    va = _c(v, np.float16)
    ln = None if lens is None else _c(lens, np.int32)
    out = np.empty((B, Hq, D), np.float16)
    f64 = np.empty((B, Hq, D), np.float64) if want_f64 else None
    _load().oracle_rvq_attend(_p(qa.view(np.uint16)), _p(p1), _p(p2), _p(nr), _p(va.view(np.uint16)),
                              None if ln is None else _p(ln), B, Hq, Hkv, S_cap, D, bits,
                              _p(_c(c1, np.float32)), _p(_c(c2, np.float32)), float(scale),
                              _p(out.view(np.uint16)), _p(f64), _p(_signs(signs, D)))
    return (out, f64) if want_f64 else out


# ---------------------------------------------------------------- KIVI


def kivi_quant(x_f16: np.ndarray, bits: int, group: int, residual_length: int,
               per_channel: bool):
    """KIVI quantization of x [B, H, S, D] (fp16) over tokens [0, S - residual_length).

    per_channel=True: keys (groups of `group` tokens per channel).
    per_channel=False: values (groups of `group` channels per token).
    Returns dict: codes [BH, S_q, D] u8, scale/zero fp16 (group layout),
    packed uint32 (the library's layout), tie [BH, S_q, D] u8, S_q, NG.
    """
    x = _c(x_f16, np.float16)
    B, H, S, D = x.shape
    BH = B * H
    S_q = max(S - residual_length, 0)
    if per_channel:
        NG = (S_q + group - 1) // group
        scale = np.zeros((BH, NG, D), np.uint16)
        zero = np.zeros((BH, NG, D), np.uint16)
        packed = np.zeros((BH, NG, group * bits // 32, D), np.uint32)
    else:
        NG = D // group
        scale = np.zeros((BH, S_q, NG), np.uint16)
        zero = np.zeros((BH, S_q, NG), np.uint16)
        packed = np.zeros((BH, S_q, D * bits // 32), np.uint32)
    codes = np.zeros((BH, S_q, D), np.uint8)
    tie = np.zeros((BH, S_q, D), np.uint8)
    if S_q > 0:
        _load().oracle_kivi_quant(_p(x.view(np.uint16)), BH, S, D, bits, group, S_q,
                                  1 if per_channel else 0, _p(codes), _p(scale), _p(zero),
                                  _p(packed), _p(tie))
    return {"codes": codes, "scale": scale.view(np.float16), "zero": zero.view(np.float16),
            "packed": packed, "tie": tie, "S_q": S_q, "NG": NG}


def kivi_dequant(packed, scale_f16, zero_f16, BH: int, S_q: int, D: int, bits: int,
                 group: int, per_channel: bool) -> np.ndarray:
    """KIVI unpack + dequant to fp16 [BH, S_q, D]."""
    p = _c(packed, np.uint32)
    s = _c(scale_f16, np.float16)
    z = _c(zero_f16, np.float16)
    out = np.empty((BH, S_q, D), np.float16)
    _load().oracle_kivi_dequant(_p(p), _p(s.view(np.uint16)), _p(z.view(np.uint16)), BH, S_q,
                                D, bits, group, 1 if per_channel else 0,
                                _p(out.view(np.uint16)))
    return out


def kivi_attend(q, k_packed, k_scale, k_zero, v_packed, v_scale, v_zero, bits: int, group: int,
                scale: float, k_res=None, v_res=None, lens=None, res_lens=None, want_f64: bool = False):
    """Decode-time attention over a KIVI cache with the dequantization inside
    the attention (see oracle.c).  q [B, Hq, D] fp16; k_packed
    [B, Hkv, NG, G*b/32, D] uint32, k_scale/k_zero [B, Hkv, NG, D] fp16;
    v_packed [B, Hkv, S_cap, D*b/32], v_scale/v_zero [B, Hkv, S_cap, D/G];
    k_res, v_res [B, Hkv, R, D] fp16 or None; lens, res_lens [B] int32 or None.
    Returns fp16 [B, Hq, D] (and binary64 if asked)."""
    qa = _c(q, np.float16)
    B, Hq, D = qa.shape
    vp = _c(v_packed, np.uint32)
    _, Hkv, S_cap, _ = vp.shape
    kp = _c(k_packed, np.uint32)
    ks, kz = _c(k_scale, np.float16), _c(k_zero, np.float16)
    vs, vz = _c(v_scale, np.float16), _c(v_zero, np.float16)
    R = 0 if k_res is None else k_res.shape[2]
    kr = None if k_res is None else _c(k_res, np.float16)
    vr = None if v_res is None else _c(v_res, np.float16)
    ln = None if lens is None else _c(lens, np.int32)
    rl = None if res_lens is None else _c(res_lens, np.int32)
    out = np.empty((B, Hq, D), np.float16)
    f64 = np.empty((B, Hq, D), np.float64) if want_f64 else None
    h16 = lambda a: None if a is None else _p(a.view(np.uint16))
    _load().oracle_kivi_attend(h16(qa), _p(kp), h16(ks), h16(kz), _p(vp), h16(vs), h16(vz), h16(kr), h16(vr),
                               _p(ln), _p(rl), B, Hq, Hkv, S_cap, R, D, bits, group, float(scale),
                               _p(out.view(np.uint16)), _p(f64))
    return (out, f64) if want_f64 else out


def qjl_encode(x_f16: np.ndarray, s_f16: np.ndarray):
    """QJL encode ([TQ] "Kernel 4: QJL Encode"): x [N, d] and the sketch S
    [m, d], both fp16.  Returns packed [N, m/32] uint32 (bit j of word w:
    sign(S x)[32w + j] >= 0), norms [N] fp16, tie [N, m] and norm_tie [N]
    flags (the exact dot products and norms, see oracle.c)."""
    x = np.ascontiguousarray(x_f16, dtype=np.float16)
    s = np.ascontiguousarray(s_f16, dtype=np.float16)
    N, d = x.shape
    m, d2 = s.shape
    assert d2 == d and m % 32 == 0
    packed = np.zeros((N, m // 32), np.uint32)
    norms = np.zeros(N, np.uint16)
    tie = np.zeros((N, m), np.uint8)
    ntie = np.zeros(N, np.uint8)
    _load().oracle_qjl_encode(_p(x.view(np.uint16)), N, d, _p(s.view(np.uint16)), m, _p(packed), _p(norms),
                              _p(tie), _p(ntie))
    return {"packed": packed, "norms": norms.view(np.float16), "tie": tie.astype(bool),
            "norm_tie": ntie.astype(bool)}
