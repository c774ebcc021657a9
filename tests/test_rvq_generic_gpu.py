"""TurboQuantRVQ at the other head widths and bit counts the pages test
(D = 8 .. 256, b = 1 .. 4; b = 3 packs ten codes per word): CUDA path vs the
oracle (GB300), through the same C ABI entry points as D = 128.  Same rules as
tests/parity.py."""
import numpy as np
import pytest

from parity import check_rvq

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SHAPES = [(D, b) for D in (8, 16, 32, 64, 256) for b in (1, 2, 3, 4)] + [(128, 3)]


@pytest.fixture(scope="module")
def vq():
    from kv_cache_quantization_turboquantrvq_gb300 import api, build
    build.build()
    api.lib()
    return api


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _rows(B, H, S, D, seed, outliers=(2, 20.0)):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    n = min(outliers[0], D // 4)
    return synth.kv_tensor(B, H, S, D, seed, n, outliers[1])


@pytest.mark.parametrize("D,bits", SHAPES)
def test_encode_parity(vq, oracle_mod, D, bits):
    x = _rows(2, 3, 333, D, 1000 + D + bits)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    p1, p2, n = vq.vq_rvq_encode_pack(_dev(x), bits, *cb)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    assert p1.shape[-1] == -(-D // (32 // bits))
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb)
    check_rvq(p1.cpu().numpy(), p2.cpu().numpy(), n.cpu().numpy(), ora, bits, D=D)


@pytest.mark.parametrize("D,bits", [(256, 4), (256, 3), (64, 4), (8, 3)])
def test_encode_parity_guard_band_rows(vq, oracle_mod, D, bits):
    """Enough rows that many steps go through the binary64 recompute."""
    x = _rows(1, 4, 6000, D, 1100 + D + bits, outliers=(4, 40.0))
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    p1, p2, n = vq.vq_rvq_encode_pack(_dev(x), bits, *cb)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb, want_values=True)
    near = np.min(np.abs(ora["y"][..., None] - cb[1].astype(np.float64)), -1) < 1e-6
    assert near.any(axis=1).sum() >= 1  # the binary64 recompute really ran
    check_rvq(p1.cpu().numpy(), p2.cpu().numpy(), n.cpu().numpy(), ora, bits, D=D)


@pytest.mark.parametrize("D,bits", [(16, 3), (64, 2), (256, 1)])
def test_encode_special_rows_and_offsets(vq, oracle_mod, D, bits):
    """Zero, one-hot, fp16-extreme and subnormal rows, written at per-batch
    offsets into a larger destination."""
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    rows = [np.zeros(D), np.eye(D)[0], -3.0 * np.eye(D)[D - 1], np.where(np.arange(D) % 2, 65504.0, -65504.0),
            np.full(D, 2.0 ** -24), np.linspace(-1000, 1000, D)]
    x = np.array(rows * 4).astype(np.float16).reshape(2, 1, 12, D)
    off = np.array([5, 0], np.int32)
    S_dst = 20
    W = -(-D // (32 // bits))
    p1 = torch.zeros((2, 1, S_dst, W), dtype=torch.int32, device="cuda")
    p2 = torch.zeros_like(p1)
    nr = torch.zeros((2, 1, S_dst), dtype=torch.float32, device="cuda")
    vq.vq_rvq_encode_pack(_dev(x), bits, *cb, packed1=p1, packed2=p2, norms=nr, dst_off=_dev(off), S_dst=S_dst)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb)
    g1 = np.concatenate([p1.cpu().numpy()[0, 0, 5:17], p1.cpu().numpy()[1, 0, 0:12]])
    g2 = np.concatenate([p2.cpu().numpy()[0, 0, 5:17], p2.cpu().numpy()[1, 0, 0:12]])
    gn = np.concatenate([nr.cpu().numpy()[0, 0, 5:17], nr.cpu().numpy()[1, 0, 0:12]])
    check_rvq(g1, g2, gn, ora, bits, strict=False, D=D)
    assert np.all(p1.cpu().numpy()[0, 0, :5] == 0) and np.all(p1.cpu().numpy()[1, 0, 12:] == 0)


@pytest.mark.parametrize("D,bits", SHAPES)
def test_decode_parity(vq, oracle_mod, D, bits):
    x = _rows(1, 3, 555, D, 1200 + D + bits)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb)
    ref, ref64 = oracle_mod.rvq_decode(ora["packed1"], ora["packed2"], ora["norms"], D, bits, cb[0], cb[2],
                                       want_f64=True)
    W = ora["packed1"].shape[-1]
    out = vq.vq_rvq_unpack_dequant(_dev(ora["packed1"].view(np.int32).reshape(1, 3, 555, W)),
                                   _dev(ora["packed2"].view(np.int32).reshape(1, 3, 555, W)),
                                   _dev(ora["norms"].reshape(1, 3, 555)), bits, cb[0], cb[2], D=D)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    got = out.cpu().numpy().reshape(-1, D).astype(np.float64)
    n = ora["norms"].astype(np.float64)[:, None]
    assert np.all(np.abs(got - ref64) <= 1e-3 * n + 1e-30)
    assert np.mean(got == ref.astype(np.float64)) > 0.95


def test_signs_need_the_dedicated_shape(vq, oracle_mod):
    from kv_cache_quantization_turboquantrvq_gb300.api import VQError
    cb = oracle_mod.rvq_codebooks(64, 2)[:4]
    x = _dev(np.zeros((1, 1, 4, 64), np.float16))
    with pytest.raises(VQError) as e:
        vq.vq_rvq_encode_pack(x, 2, *cb, signs=np.zeros(4, np.uint32))
    assert e.value.status == vq.VQ_ERR_UNSUPPORTED
