"""Every row inside the guard band (GB300): the tensor-memory encoder's exact
recompute at full load.

Rows (a, a, 0, ..., 0) rotate to exact zeros at half their coordinates (the
odd ones; with randomised signs, those of one parity), and 0 is a boundary of
the library's books at b = 2 and b = 4, so every row is flagged: far more
rows per CTA than the fixup warps' list holds (the epilogue then recomputes
the rest itself) and, at b = 4, more than the fixup warps keep up with.  The
exact value y = 0 leaves no room for a tie: every code must equal the
oracle's (turboquant page, "The pipeline, as it actually runs": codes are
counts of boundaries below the value).  Also through the one-launch decode
flush, whose RVQ part runs the same encoder body.
"""
import numpy as np
import pytest

from parity import unpack_rows

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


def _pair_rows(B, H, S, seed):
    rng = np.random.default_rng(seed)
    x = np.zeros((B, H, S, D), np.float16)
    a = rng.standard_normal((B, H, S)).astype(np.float16)
    a[a == 0] = np.float16(1.0)
    x[..., 0] = a
    x[..., 1] = a
    return x


def _exact(vq, oracle_mod, x, bits, cb, p1, p2, nr, signs=None):
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb, signs=signs)
    W = 4 * bits
    g1 = unpack_rows(p1.cpu().numpy().reshape(-1, W), bits)
    g2 = unpack_rows(p2.cpu().numpy().reshape(-1, W), bits)
    assert ora["tie1"].any(axis=1).all(), "every row should hold an exact zero"
    assert np.array_equal(g1, ora["idx1"]), "stage-1: %d mismatches" % (g1 != ora["idx1"]).sum()
    assert np.array_equal(g2, ora["idx2"]), "stage-2: %d mismatches" % (g2 != ora["idx2"]).sum()
    assert np.array_equal(p1.cpu().numpy().view(np.uint32).reshape(-1, W), ora["packed1"])
    assert np.array_equal(p2.cpu().numpy().view(np.uint32).reshape(-1, W), ora["packed2"])
    gn = nr.cpu().numpy().reshape(-1).astype(np.float64)
    rn = ora["norms"].astype(np.float64)
    assert np.all(np.abs(gn - rn) <= 6e-8 * rn)  # recomputed rows: within one rounding


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("signed", [False, True])
def test_every_row_flagged(vq, oracle_mod, bits, signed):
    x = _pair_rows(1, 8, 32768, 700 + bits)  # 262,144 rows: ~1,700 per CTA
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    assert np.min(np.abs(cb[1])) == 0.0  # 0 is a stage-1 boundary
    signs = np.random.default_rng(710 + bits).integers(0, 2 ** 32, 4, dtype=np.uint32) if signed else None
    p1, p2, nr = vq.vq_rvq_encode_pack(_dev(x), bits, *cb, signs=signs)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    _exact(vq, oracle_mod, x, bits, cb, p1, p2, nr, signs)


@pytest.mark.parametrize("bits", [2, 4])
def test_every_row_flagged_in_the_flush(vq, oracle_mod, bits):
    x = _pair_rows(64, 8, 128, 720 + bits)  # a decode flush: 65,536 rows
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    out = vq.vq_flush_decode(_dev(x), None, 0, rvq=dict(bits=bits, books=cb))
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    _exact(vq, oracle_mod, x, bits, cb, out["packed1"], out["packed2"], out["norms"])
