"""vq_rvq_attend_noalloc: decode attention with the library's static device
scratch instead of a caller workspace.

CPU tests check the declaration, the export and host-side validation; GPU
tests check that the output is bit-identical to vq_rvq_attend with a full
workspace (same chunking), agrees with the oracle, never reads partials left
by an earlier call, and that a plan too large for the scratch is refused
before any launch.  The file runs on its own or after the rest of the suite.
"""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
D = 128


@pytest.fixture(scope="module")
def api():
    from kv_cache_quantization_turboquantrvq_gb300 import api as a, build
    build.build()
    a.lib()
    return a


def test_declared_exported_and_sized(api):
    src = open(os.path.join(ROOT, "include", "vq.h")).read()
    assert re.search(r"\bvq_status\s+vq_rvq_attend_noalloc\s*\(", src)
    m = re.search(r"#define\s+VQ_ATTEND_SCRATCH_BYTES\s+\((\d+)u\s*\*\s*(\d+)u\s*\*\s*(\d+)u\)", src)
    assert m and int(m.group(1)) * int(m.group(2)) * int(m.group(3)) == api.VQ_ATTEND_SCRATCH_BYTES
    assert hasattr(api.lib(), "vq_rvq_attend_noalloc")
    assert "vq_rvq_attend_noalloc" in api.EXPORTED


def test_host_validation_before_any_device_call(api):
    # fake, aligned addresses: every case below must be refused on the host
    A = ctypes.c_void_p(1 << 32)
    c = (ctypes.c_float * 4)(-0.1, -0.03, 0.03, 0.1)
    L = api.lib()

    def call(B, Hq, Hkv, S, D_, bits, scale=0.1):
        return L.vq_rvq_attend_noalloc(A, A, A, A, A, None, B, Hq, Hkv, S, D_, bits, c, c,
                                       ctypes.c_float(scale), A, None)
    assert call(1, 3, 2, 16, D, 2) == api.VQ_ERR_INVALID_ARG        # Hq not a multiple of Hkv
    assert call(1, 32, 2, 16, D, 2) == api.VQ_ERR_UNSUPPORTED       # 16 query heads per kv head
    assert call(1, 4, 2, 16, 64, 2) == api.VQ_ERR_UNSUPPORTED       # D != 128
    assert call(1, 4, 2, 16, D, 3) == api.VQ_ERR_UNSUPPORTED        # 3-bit codes
    assert call(1, 4, 2, 16, D, 2, float("inf")) == api.VQ_ERR_INVALID_ARG
    assert call(-1, 4, 2, 16, D, 2) == api.VQ_ERR_INVALID_ARG
    assert call(0, 4, 2, 16, D, 2) == api.VQ_OK                     # nothing to do


def _dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _case(B, Hkv, gq, S, bits, seed):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    rng = np.random.default_rng(seed)
    W = D * bits // 32
    p1 = rng.integers(0, 2 ** 32, (B, Hkv, S, W), dtype=np.uint32)
    p2 = rng.integers(0, 2 ** 32, (B, Hkv, S, W), dtype=np.uint32)
    nr = rng.uniform(4.0, 24.0, (B, Hkv, S)).astype(np.float32)
    v = synth.kv_tensor(B, Hkv, S, D, seed + 1, 0, 1.0)
    q = rng.standard_normal((B, Hkv * gq, D)).astype(np.float16)
    return q, p1, p2, nr, v


@pytest.mark.gpu
@pytest.mark.parametrize("bits,gq", [(1, 8), (2, 4), (4, 2)])
def test_bit_identical_to_workspace_call_and_oracle(api, oracle_mod, bits, gq):
    import torch
    B, Hkv, S = 6, 2, 3000
    q, p1, p2, nr, v = _case(B, Hkv, gq, S, bits, 200 + bits)
    lens = np.array([3000, 1, 0, 2999, 1234, 2048], np.int32)
    cb = oracle_mod.rvq_codebooks(D, bits)
    args = [_dev(q), _dev(p1.view(np.int32)), _dev(p2.view(np.int32)), _dev(nr), _dev(v), bits, cb[0], cb[2],
            1.0 / np.sqrt(D)]
    assert api.vq_rvq_attend_workspace(B, Hkv * gq, Hkv, S) > 0  # the split path runs
    ref = api.vq_rvq_attend(*args, lens=_dev(lens)).cpu().numpy()
    got = api.vq_rvq_attend_noalloc(*args, lens=_dev(lens)).cpu().numpy()
    torch.cuda.synchronize()
    assert api.vq_device_error() == 0
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))
    r16, r64 = oracle_mod.rvq_attend(q, p1, p2, nr, v, bits, cb[0], cb[2], 1.0 / np.sqrt(D), lens=lens,
                                     want_f64=True)
    tol = 0.5 * np.spacing(np.abs(r64).astype(np.float16)).astype(np.float64) + 2e-5 * float(np.abs(v).max())
    assert np.all(np.abs(got.astype(np.float64) - r64) <= tol)
    assert np.all(got[2] == 0)


@pytest.mark.gpu
def test_partials_of_an_earlier_call_are_never_read(api, oracle_mod):
    """A long call fills many chunks of the scratch; a following call with
    shorter caches (fewer chunks) must not pick any of them up."""
    import torch
    bits, gq, B, Hkv, S = 2, 4, 4, 2, 4096
    cb = oracle_mod.rvq_codebooks(D, bits)
    q, p1, p2, nr, v = _case(B, Hkv, gq, S, bits, 300)
    args = [_dev(q), _dev(p1.view(np.int32)), _dev(p2.view(np.int32)), _dev(nr), _dev(v), bits, cb[0], cb[2], 0.2]
    api.vq_rvq_attend_noalloc(*args, lens=_dev(np.full(B, S, np.int32)))
    short = np.array([700, 5, 0, 2100], np.int32)
    got = api.vq_rvq_attend_noalloc(*args, lens=_dev(short)).cpu().numpy()
    torch.cuda.synchronize()
    assert api.vq_device_error() == 0
    ref = api.vq_rvq_attend(*args, lens=_dev(short)).cpu().numpy()
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))
    r16 = oracle_mod.rvq_attend(q, p1, p2, nr, v, bits, cb[0], cb[2], 0.2, lens=short)
    assert np.mean(got.view(np.uint16) == r16.view(np.uint16)) > 0.9


@pytest.mark.gpu
def test_plan_larger_than_the_scratch_is_refused(api):
    """64 sequences x 8 kv heads x 64 query heads over 16k caches: the
    default chunking needs 64 * 64 * 8 partials of 520 bytes (17 MB), more than
    the 16 MiB scratch, so the call returns VQ_ERR_UNSUPPORTED before any
    launch.  The buffers are real, full-size allocations all the same."""
    import torch
    B, Hkv, gq, S, bits = 64, 8, 8, 16384, 1
    Hq = Hkv * gq
    W = D * bits // 32
    assert api.vq_rvq_attend_workspace(B, Hq, Hkv, S) > api.VQ_ATTEND_SCRATCH_BYTES
    p1 = torch.empty((B, Hkv, S, W), dtype=torch.int32, device="cuda")
    p2 = torch.empty_like(p1)
    nr = torch.empty((B, Hkv, S), dtype=torch.float32, device="cuda")
    v = torch.empty((B, Hkv, S, D), dtype=torch.float16, device="cuda")
    q = torch.zeros((B, Hq, D), dtype=torch.float16, device="cuda")
    c = np.array([-0.07, 0.07], np.float32)
    with pytest.raises(api.VQError) as e:
        api.vq_rvq_attend_noalloc(q, p1, p2, nr, v, bits, c, c, 0.1)
    assert e.value.status == api.VQ_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert api.vq_device_error() == 0
    del p1, p2, nr, v
    torch.cuda.empty_cache()
