"""QJL encode (turboquant page, "Kernel 4: QJL Encode"): CUDA path vs the
oracle through the C ABI.

Bits: the oracle's signs are exact; the tensor-core dot products are fp32
sums of exact products, so a bit may differ only where the oracle flags the
dot product as a tie (|dot| < 1e-5 sum |S_jd x_d|), and such differences must
stay below 1e-6 of all bits.  Norms: equal to the oracle's fp16 norm except
on rows it flags as within 1e-6 of an fp16 rounding boundary.
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


def _bits(words, m):
    w = np.asarray(words).view(np.uint32).reshape(-1, m // 32)
    j = np.arange(m)
    return ((w[:, j // 32] >> (j % 32).astype(np.uint32)) & 1).astype(bool)


def _check(vq, oracle_mod, x, S):
    m = S.shape[0]
    p, n = vq.vq_qjl_encode(torch.from_numpy(x).cuda(), torch.from_numpy(S).cuda())
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    ora = oracle_mod.qjl_encode(x.reshape(-1, D), S)
    got = _bits(p.cpu().numpy(), m)
    ref = _bits(ora["packed"], m)
    bad = (got != ref) & ~ora["tie"]
    assert not bad.any(), "%d sign bits differ outside the tie band" % bad.sum()
    assert (got != ref).sum() <= max(1, int(1e-6 * got.size))
    gn = n.cpu().numpy().reshape(-1)
    ok = (gn.view(np.uint16) == ora["norms"].view(np.uint16)) | ora["norm_tie"]
    assert ok.all(), "norms differ on %d rows" % (~ok).sum()
    return got, gn


@pytest.mark.parametrize("m", [32, 64, 96, 128, 224, 256])
@pytest.mark.parametrize("N", [1, 5, 33, 700])
def test_parity_small_and_ragged(vq, oracle_mod, m, N):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    x = synth.kv_tensor(1, 1, N, D, 2000 + N + m, 4, 20.0).reshape(N, D)
    S = np.random.default_rng(2100 + m).standard_normal((m, D)).astype(np.float16)
    _check(vq, oracle_mod, x, S)


def test_special_rows(vq, oracle_mod):
    rows = [np.zeros(D), np.full(D, 65504.0), np.full(D, -65504.0), np.full(D, 2.0 ** -24)]
    e = np.zeros(D)
    e[7] = 1.0
    rows.append(e)
    alt = np.full(D, 0.5)
    alt[1::2] = -0.5
    rows.append(alt)
    x = np.array(rows * 3).astype(np.float16)
    S = np.random.default_rng(2200).standard_normal((128, D)).astype(np.float16)
    S[5] = 0.0  # a zero sketch row: every dot 0, every bit 1
    got, gn = _check(vq, oracle_mod, x, S)
    assert got[0].all() and gn[0] == 0  # zero key: dots 0 (>= 0) and norm 0
    assert got[:, 5].all()


def test_long_context_keys_sampled(vq, oracle_mod):
    """Keys [4, 32, 32768, 128] (1 GiB) with m = 128, in one call; sampled
    rows checked against the oracle."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    B, H, S_len, m = 4, 32, 32768, 128
    dev = torch.device("cuda")
    x = torch.empty((B, H, S_len, D), dtype=torch.float16, device=dev)
    for b in range(B):
        x[b].copy_(torch.from_numpy(synth.kv_tensor(1, H, S_len, D, 2300 + b, 4, 40.0)[0]))
    S = np.random.default_rng(2400).standard_normal((m, D)).astype(np.float16)
    p, n = vq.vq_qjl_encode(x, torch.from_numpy(S).cuda())
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    N = B * H * S_len
    idx = np.sort(np.random.default_rng(2500).choice(N, 3000, replace=False))
    xs = x.reshape(N, D)[torch.from_numpy(idx).cuda()].cpu().numpy()
    ora = oracle_mod.qjl_encode(xs, S)
    got = _bits(p.reshape(N, m // 32)[torch.from_numpy(idx).cuda()].cpu().numpy(), m)
    ref = _bits(ora["packed"], m)
    assert not ((got != ref) & ~ora["tie"]).any()
    gn = n.reshape(N)[torch.from_numpy(idx).cuda()].cpu().numpy()
    assert ((gn.view(np.uint16) == ora["norms"].view(np.uint16)) | ora["norm_tie"]).all()
    del x, p, n
    torch.cuda.empty_cache()
