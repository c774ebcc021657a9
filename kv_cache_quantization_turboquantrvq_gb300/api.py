"""Python binding of the C ABI in include/vq.h (ctypes; argument marshalling only).

Every function here has the name of the C entry point it calls.  Tensors are
torch CUDA tensors (torch supplies device memory and the current stream);
codebooks are small host float32 arrays.  All arithmetic runs in the CUDA
library ``libvqflush.so``; if it is missing this module raises on first use,
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvqflush.so")
_lib = None

VQ_OK = 0
VQ_ERR_INVALID_ARG = 1
VQ_ERR_UNSUPPORTED = 2
VQ_ERR_MISALIGNED = 3
VQ_ERR_ALIASING = 4
VQ_ERR_CUDA = 5
VQ_ERR_DEVICE = 6
VQ_DEVERR_WAIT_TIMEOUT = 0x1
VQ_DEVERR_BAD_OFFSET = 0x2

EXPORTED = ("vq_status_str", "vq_version", "vq_rvq_codebook", "vq_rvq_encode_pack",
            "vq_rvq_unpack_dequant", "vq_kivi_quant_pack", "vq_kivi_unpack_dequant",
            "vq_device_error", "vq_rvq_attend_workspace", "vq_rvq_attend", "vq_rvq_attend_noalloc",
            "vq_rvq_encode_pack_rs", "vq_rvq_unpack_dequant_rs", "vq_rvq_attend_rs",
            "vq_kivi_attend_workspace", "vq_kivi_attend", "vq_qjl_encode", "vq_flush_decode")
VQ_ATTEND_SCRATCH_BYTES = 16 * 1024 * 1024


class VQError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s: %s" % (what, lib().vq_status_str(status).decode()))
        self.status = status


def lib():
    """Load libvqflush.so (raises OSError when it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise OSError("libvqflush.so is not built (run __graft_entry__.build()): %s" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    P, I = ctypes.c_void_p, ctypes.c_int
    L.vq_status_str.argtypes = [I]
    L.vq_status_str.restype = ctypes.c_char_p
    L.vq_version.argtypes = []
    L.vq_version.restype = ctypes.c_char_p
    L.vq_rvq_codebook.argtypes = [I, I, P, P, P, P]
    L.vq_rvq_encode_pack.argtypes = [P, I, I, I, I, I, P, P, P, P, P, P, P, P, I, P]
    L.vq_rvq_unpack_dequant.argtypes = [P, P, P, I, I, I, I, I, P, P, P, P]
    L.vq_kivi_quant_pack.argtypes = [P, P, I, I, I, I, I, I, I, P, P, P, P, P, P, P, I, P]
    L.vq_kivi_unpack_dequant.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, P]
    L.vq_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
    L.vq_rvq_attend_workspace.argtypes = [I, I, I, I, ctypes.POINTER(ctypes.c_size_t)]
    L.vq_rvq_attend.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, ctypes.c_float, P, P,
                                ctypes.c_size_t, P]
    L.vq_rvq_attend_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, ctypes.c_float, P, P]
    L.vq_rvq_encode_pack_rs.argtypes = [P, I, I, I, I, I, P, P, P, P, P, P, P, P, I, P, P]
    L.vq_rvq_unpack_dequant_rs.argtypes = [P, P, P, I, I, I, I, I, P, P, P, P, P]
    L.vq_rvq_attend_rs.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, ctypes.c_float, P, P,
                                   ctypes.c_size_t, P]
    L.vq_kivi_attend_workspace.argtypes = [I, I, I, I, I, ctypes.POINTER(ctypes.c_size_t)]
    L.vq_kivi_attend.argtypes = [P] * 11 + [I] * 8 + [ctypes.c_float, P, P, ctypes.c_size_t, P]
    L.vq_qjl_encode.argtypes = [P, I, I, P, I, P, P, P]
    L.vq_flush_decode.argtypes = [P, P, I, I, I, I, I, P, I, I, P, P, P, P, P, P, P, I, I,
                                  P, P, P, P, P, P, P, P, P, I, P]
    for name in EXPORTED[2:]:
        getattr(L, name).restype = I
    _lib = L
    return L


def _check(status: int, what: str):
    if status != VQ_OK:
        raise VQError(status, what)


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _host(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def vq_status_str(status: int) -> str:
    return lib().vq_status_str(status).decode()


def vq_version() -> str:
    return lib().vq_version().decode()


def rvq_words(D: int, bits: int) -> int:
    """Packed words per row and stream: floor(32/b) codes per word."""
    return -(-D // (32 // bits))


def vq_rvq_codebook(D: int, bits: int):
    """(c1, b1, c2, b2) float32 host arrays: Gaussian stage-1 and Laplace-fit stage-2."""
    L = 1 << bits
    c1 = np.empty(L, np.float32)
    b1 = np.empty(L - 1, np.float32)
    c2 = np.empty(L, np.float32)
    b2 = np.empty(L - 1, np.float32)
    _check(lib().vq_rvq_codebook(D, bits, *[a.ctypes.data_as(ctypes.c_void_p) for a in (c1, b1, c2, b2)]),
           "vq_rvq_codebook")
    return c1, b1, c2, b2


def _sign_words(signs):
    s = np.ascontiguousarray(np.asarray(signs, dtype=np.uint32).ravel())
    if s.size != 4:
        raise ValueError("signs: 4 uint32 words (one bit per coordinate of D = 128)")
    return s


def vq_rvq_encode_pack(k, bits: int, c1, b1, c2, b2, packed1=None, packed2=None, norms=None,
                       dst_off=None, S_dst=None, stream=None, signs=None):
    """Encode fp16 keys k [B, H, S, D] into (packed1, packed2, norms); with
    `signs` (4 uint32 words) the randomised-sign rotation H diag(s)."""
    import torch
    B, H, S, D = k.shape
    S_dst = S if S_dst is None else S_dst
    W = rvq_words(D, bits)
    if packed1 is None:
        packed1 = torch.empty((B, H, S_dst, W), dtype=torch.int32, device=k.device)
    if packed2 is None:
        packed2 = torch.empty((B, H, S_dst, W), dtype=torch.int32, device=k.device)
    if norms is None:
        norms = torch.empty((B, H, S_dst), dtype=torch.float32, device=k.device)
    keep = [_host(v) for v in (c1, b1, c2, b2)]
    if signs is None:
        _check(lib().vq_rvq_encode_pack(_ptr(k), B, H, S, D, bits, *[p for _, p in keep],
                                        _ptr(packed1), _ptr(packed2), _ptr(norms), _ptr(dst_off),
                                        S_dst, _stream(stream)), "vq_rvq_encode_pack")
    else:
        sw = _sign_words(signs)
        _check(lib().vq_rvq_encode_pack_rs(_ptr(k), B, H, S, D, bits, *[p for _, p in keep],
                                           _ptr(packed1), _ptr(packed2), _ptr(norms), _ptr(dst_off),
                                           S_dst, sw.ctypes.data_as(ctypes.c_void_p), _stream(stream)),
               "vq_rvq_encode_pack_rs")
    return packed1, packed2, norms


def vq_rvq_unpack_dequant(packed1, packed2, norms, bits: int, c1, c2, out=None, stream=None, signs=None,
                          D: int = 128):
    """Decode (packed1, packed2, norms) [B, H, S, W] back to fp16 keys [B, H, S, D]."""
    import torch
    B, H, S, _ = packed1.shape
    if out is None:
        out = torch.empty((B, H, S, D), dtype=torch.float16, device=packed1.device)
    keep = [_host(v) for v in (c1, c2)]
    if signs is None:
        _check(lib().vq_rvq_unpack_dequant(_ptr(packed1), _ptr(packed2), _ptr(norms), B, H, S, D, bits,
                                           keep[0][1], keep[1][1], _ptr(out), _stream(stream)),
               "vq_rvq_unpack_dequant")
    else:
        sw = _sign_words(signs)
        _check(lib().vq_rvq_unpack_dequant_rs(_ptr(packed1), _ptr(packed2), _ptr(norms), B, H, S, D, bits,
                                              keep[0][1], keep[1][1], sw.ctypes.data_as(ctypes.c_void_p),
                                              _ptr(out), _stream(stream)), "vq_rvq_unpack_dequant_rs")
    return out


def kivi_shapes(B, H, S_dst, D, bits, group):
    """Output shapes of vq_kivi_quant_pack for a destination of S_dst tokens."""
    NG = (S_dst + group - 1) // group
    return {
        "k_packed": (B, H, NG, group * bits // 32, D), "k_scale": (B, H, NG, D),
        "v_packed": (B, H, S_dst, D * bits // 32), "v_scale": (B, H, S_dst, D // group),
    }


def vq_rvq_attend_workspace(B: int, Hq: int, Hkv: int, S_cap: int) -> int:
    """Workspace bytes vq_rvq_attend wants for these shapes on the current device."""
    n = ctypes.c_size_t(0)
    _check(lib().vq_rvq_attend_workspace(B, Hq, Hkv, S_cap, ctypes.byref(n)), "vq_rvq_attend_workspace")
    return int(n.value)


def vq_rvq_attend(q, packed1, packed2, norms, v, bits: int, c1, c2, scale: float, lens=None, out=None,
                  workspace=None, stream=None, signs=None):
    """Decode-time attention of q [B, Hq, 128] over an RVQ key cache
    (packed1, packed2, norms [B, Hkv, S_cap, ...]) and fp16 values v
    [B, Hkv, S_cap, 128]; lens [B] int32 (device) or None.  Returns fp16
    [B, Hq, 128].  The workspace is allocated when not given."""
    import torch
    B, Hq, D = q.shape
    _, Hkv, S_cap, _ = packed1.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float16, device=q.device)
    if workspace is None:
        nbytes = vq_rvq_attend_workspace(B, Hq, Hkv, S_cap)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=q.device)
    wbytes = workspace.numel() * workspace.element_size()
    keep = [_host(t) for t in (c1, c2)]
    if signs is None:
        _check(lib().vq_rvq_attend(_ptr(q), _ptr(packed1), _ptr(packed2), _ptr(norms), _ptr(v), _ptr(lens),
                                   B, Hq, Hkv, S_cap, D, bits, keep[0][1], keep[1][1], float(scale),
                                   _ptr(out), _ptr(workspace), wbytes, _stream(stream)), "vq_rvq_attend")
    else:
        sw = _sign_words(signs)
        _check(lib().vq_rvq_attend_rs(_ptr(q), _ptr(packed1), _ptr(packed2), _ptr(norms), _ptr(v), _ptr(lens),
                                      B, Hq, Hkv, S_cap, D, bits, keep[0][1], keep[1][1],
                                      sw.ctypes.data_as(ctypes.c_void_p), float(scale), _ptr(out),
                                      _ptr(workspace), wbytes, _stream(stream)), "vq_rvq_attend_rs")
    return out


def vq_rvq_attend_noalloc(q, packed1, packed2, norms, v, bits: int, c1, c2, scale: float, lens=None,
                          out=None, stream=None):
    """vq_rvq_attend with the library's static device scratch instead of a
    workspace (calls must not overlap in time on one device)."""
    import torch
    B, Hq, D = q.shape
    _, Hkv, S_cap, _ = packed1.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float16, device=q.device)
    keep = [_host(t) for t in (c1, c2)]
    _check(lib().vq_rvq_attend_noalloc(_ptr(q), _ptr(packed1), _ptr(packed2), _ptr(norms), _ptr(v), _ptr(lens),
                                       B, Hq, Hkv, S_cap, D, bits, keep[0][1], keep[1][1], float(scale),
                                       _ptr(out), _stream(stream)), "vq_rvq_attend_noalloc")
    return out


def vq_kivi_attend_workspace(B: int, Hq: int, Hkv: int, S_cap: int, R: int) -> int:
    """Workspace bytes vq_kivi_attend wants for these shapes on the current device."""
    n = ctypes.c_size_t(0)
    _check(lib().vq_kivi_attend_workspace(B, Hq, Hkv, S_cap, R, ctypes.byref(n)), "vq_kivi_attend_workspace")
    return int(n.value)


def vq_kivi_attend(q, cache: dict, bits: int, group: int, scale: float, k_res=None, v_res=None, lens=None,
                   res_lens=None, out=None, workspace=None, stream=None):
    """Decode-time attention of q [B, Hq, 128] over a KIVI cache (`cache`: the
    dict vq_kivi_quant_pack returns, written with S_dst = S_cap) plus the fp16
    residual window k_res, v_res [B, Hkv, R, 128].  Returns fp16 [B, Hq, 128]."""
    import torch
    B, Hq, D = q.shape
    vp = cache["v_packed"]
    Hkv, S_cap = vp.shape[1], vp.shape[2]
    R = 0 if k_res is None else k_res.shape[2]
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.float16, device=q.device)
    if workspace is None:
        nbytes = vq_kivi_attend_workspace(B, Hq, Hkv, S_cap, R)
        workspace = torch.empty((max(nbytes, 16) + 3) // 4, dtype=torch.float32, device=q.device)
    wbytes = workspace.numel() * workspace.element_size()
    c = cache
    _check(lib().vq_kivi_attend(_ptr(q), _ptr(c["k_packed"]), _ptr(c["k_scale"]), _ptr(c["k_zero"]),
                                _ptr(c["v_packed"]), _ptr(c["v_scale"]), _ptr(c["v_zero"]), _ptr(k_res),
                                _ptr(v_res), _ptr(lens), _ptr(res_lens), B, Hq, Hkv, S_cap, R, D, bits, group,
                                float(scale), _ptr(out), _ptr(workspace), wbytes, _stream(stream)),
           "vq_kivi_attend")
    return out


def vq_kivi_quant_pack(k, v, bits: int, group: int, residual_length: int, outs=None,
                       dst_off=None, S_dst=None, stream=None):
    """KIVI flush of k and/or v ([B, H, S, D] fp16; either may be None).

    Returns a dict with k_packed, k_scale, k_zero, v_packed, v_scale, v_zero
    (allocated when `outs` does not provide them)."""
    import torch
    ref = k if k is not None else v
    B, H, S, D = ref.shape
    S_q = max(S - residual_length, 0)
    S_dst = S_q if S_dst is None else S_dst
    shp = kivi_shapes(B, H, S_dst, D, bits, group)
    outs = dict(outs or {})
    dev = ref.device
    if k is not None:
        outs.setdefault("k_packed", torch.empty(shp["k_packed"], dtype=torch.int32, device=dev))
        outs.setdefault("k_scale", torch.empty(shp["k_scale"], dtype=torch.float16, device=dev))
        outs.setdefault("k_zero", torch.empty(shp["k_scale"], dtype=torch.float16, device=dev))
    if v is not None:
        outs.setdefault("v_packed", torch.empty(shp["v_packed"], dtype=torch.int32, device=dev))
        outs.setdefault("v_scale", torch.empty(shp["v_scale"], dtype=torch.float16, device=dev))
        outs.setdefault("v_zero", torch.empty(shp["v_scale"], dtype=torch.float16, device=dev))
    g = outs.get
    _check(lib().vq_kivi_quant_pack(_ptr(k), _ptr(v), B, H, S, D, bits, group, residual_length,
                                    _ptr(g("k_packed") if k is not None else None),
                                    _ptr(g("k_scale") if k is not None else None),
                                    _ptr(g("k_zero") if k is not None else None),
                                    _ptr(g("v_packed") if v is not None else None),
                                    _ptr(g("v_scale") if v is not None else None),
                                    _ptr(g("v_zero") if v is not None else None),
                                    _ptr(dst_off), S_dst, _stream(stream)), "vq_kivi_quant_pack")
    return outs


def vq_kivi_unpack_dequant(packs: dict, B: int, H: int, S_q: int, bits: int, group: int,
                           k_out=None, v_out=None, want_k=True, want_v=True, stream=None):
    """Dequantize the KIVI storage in `packs` (keys and/or values) to fp16 [B, H, S_q, 128]."""
    import torch
    D = 128
    dk = want_k and "k_packed" in packs
    dv = want_v and "v_packed" in packs
    ref = packs["k_packed"] if dk else packs["v_packed"]
    if dk and k_out is None:
        k_out = torch.empty((B, H, S_q, D), dtype=torch.float16, device=ref.device)
    if dv and v_out is None:
        v_out = torch.empty((B, H, S_q, D), dtype=torch.float16, device=ref.device)
    _check(lib().vq_kivi_unpack_dequant(
        _ptr(packs["k_packed"]) if dk else None, _ptr(packs["k_scale"]) if dk else None,
        _ptr(packs["k_zero"]) if dk else None, _ptr(packs["v_packed"]) if dv else None,
        _ptr(packs["v_scale"]) if dv else None, _ptr(packs["v_zero"]) if dv else None,
        B, H, S_q, D, bits, group, _ptr(k_out) if dk else None, _ptr(v_out) if dv else None,
        _stream(stream)), "vq_kivi_unpack_dequant")
    return k_out, v_out


def vq_device_error(stream=None) -> int:
    """Wait for the stream; read and clear the library's device error bits."""
    code = ctypes.c_int(0)
    st = lib().vq_device_error(_stream(stream), ctypes.byref(code))
    if st not in (VQ_OK, VQ_ERR_DEVICE):
        raise VQError(st, "vq_device_error")
    return code.value


def vq_qjl_encode(x, s, packed=None, norms=None, stream=None):
    """QJL encode of the key rows x [..., 128] fp16 with the sketch s [m, 128]
    fp16: returns (packed [..., m/32] int32 sign words, norms [...] fp16)."""
    import torch
    D = x.shape[-1]
    lead = tuple(x.shape[:-1])
    N = 1
    for v in lead:
        N *= v
    m = s.shape[0]
    if packed is None:
        packed = torch.empty(lead + (m // 32,), dtype=torch.int32, device=x.device)
    if norms is None:
        norms = torch.empty(lead, dtype=torch.float16, device=x.device)
    _check(lib().vq_qjl_encode(_ptr(x), N, D, _ptr(s), m, _ptr(packed), _ptr(norms), _stream(stream)),
           "vq_qjl_encode")
    return packed, norms


def vq_flush_decode(k, v, residual_length: int, dst_off=None, S_dst=None, rvq=None, kivi=None,
                    window=None, stream=None):
    """The decode-time flush of one layer in one launch: k, v [B, H, T, 128]
    fp16 (either may be None when no part needs it); tokens [0, T - R) are
    quantized at the sequences' offsets, tokens [T - R, T) copied to the fp16
    window.  Parts (each optional, outputs allocated when absent):
      rvq = dict(bits, books=(c1, b1, c2, b2)[, packed1, packed2, norms])
      kivi = dict(bits, group[, keys=True, values=True, k_packed, ..., v_zero])
      window = dict([k_win, v_win, win_off, R_cap])
    Returns a dict with every output tensor."""
    import torch
    ref = k if k is not None else v
    B, H, T, D = ref.shape
    R = int(residual_length)
    S_q = T - R
    S_dst = S_q if S_dst is None else S_dst
    dev = ref.device
    out = {}
    keep = []
    rb, rp = 0, [None] * 4
    if rvq is not None:
        rb = int(rvq["bits"])
        keep = [_host(a) for a in rvq["books"]]
        rp = [p_ for _, p_ in keep]
        W = rvq_words(D, rb)
        out["packed1"] = rvq.get("packed1", torch.empty((B, H, S_dst, W), dtype=torch.int32, device=dev))
        out["packed2"] = rvq.get("packed2", torch.empty((B, H, S_dst, W), dtype=torch.int32, device=dev))
        out["norms"] = rvq.get("norms", torch.empty((B, H, S_dst), dtype=torch.float32, device=dev))
    kb, G = 0, 0
    if kivi is not None:
        kb, G = int(kivi["bits"]), int(kivi["group"])
        shp = kivi_shapes(B, H, S_dst, D, kb, G)
        if kivi.get("keys", True):
            out["k_packed"] = kivi.get("k_packed", torch.empty(shp["k_packed"], dtype=torch.int32, device=dev))
            out["k_scale"] = kivi.get("k_scale", torch.empty(shp["k_scale"], dtype=torch.float16, device=dev))
            out["k_zero"] = kivi.get("k_zero", torch.empty(shp["k_scale"], dtype=torch.float16, device=dev))
        if kivi.get("values", True):
            out["v_packed"] = kivi.get("v_packed", torch.empty(shp["v_packed"], dtype=torch.int32, device=dev))
            out["v_scale"] = kivi.get("v_scale", torch.empty(shp["v_scale"], dtype=torch.float16, device=dev))
            out["v_zero"] = kivi.get("v_zero", torch.empty(shp["v_scale"], dtype=torch.float16, device=dev))
    win_off, R_cap = None, 0
    if window is not None and R > 0:
        R_cap = int(window.get("R_cap", R))
        win_off = window.get("win_off")
        if k is not None:
            out["k_win"] = window.get("k_win", torch.empty((B, H, R_cap, D), dtype=torch.float16, device=dev))
        if v is not None:
            out["v_win"] = window.get("v_win", torch.empty((B, H, R_cap, D), dtype=torch.float16, device=dev))
    g = out.get
    _check(lib().vq_flush_decode(_ptr(k), _ptr(v), B, H, T, D, R, _ptr(dst_off), S_dst, rb, *rp,
                                 _ptr(g("packed1")), _ptr(g("packed2")), _ptr(g("norms")), kb, G,
                                 _ptr(g("k_packed")), _ptr(g("k_scale")), _ptr(g("k_zero")),
                                 _ptr(g("v_packed")), _ptr(g("v_scale")), _ptr(g("v_zero")),
                                 _ptr(g("k_win")), _ptr(g("v_win")), _ptr(win_off), R_cap, _stream(stream)),
           "vq_flush_decode")
    return out
