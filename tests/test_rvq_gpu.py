"""TurboQuantRVQ CUDA path vs the oracle (GB300).  Calls go through the C ABI
(the ctypes binding); inputs come from the seeded generators."""
import numpy as np
import pytest

from parity import check_rvq, unpack_rows

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


def _encode(vq, x, bits, cb, **kw):
    p1, p2, n = vq.vq_rvq_encode_pack(_dev(x), bits, *cb, **kw)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    return p1.cpu().numpy(), p2.cpu().numpy(), n.cpu().numpy()


def _rows(shape, seed, outliers=(4, 20.0)):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    B, H, S = shape
    return synth.kv_tensor(B, H, S, D, seed, outliers[0], outliers[1])


@pytest.mark.parametrize("bits", [1, 2, 4])
@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 1, 5), (1, 1, 33), (2, 3, 700)])
def test_encode_parity_small(vq, oracle_mod, bits, shape):
    x = _rows(shape, 7 + bits)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    p1, p2, n = _encode(vq, x, bits, cb)
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb)
    check_rvq(p1, p2, n, ora, bits)


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_encode_parity_guard_band_rows(vq, oracle_mod, bits):
    """Enough rows that a few percent go through the exact recompute path."""
    x = _rows((1, 4, 5000), 300 + bits, outliers=(4, 40.0))
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    p1, p2, n = _encode(vq, x, bits, cb)
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb, want_values=True)
    b1 = cb[1].astype(np.float64)
    near = np.min(np.abs(ora["y"][..., None] - b1), -1) < 2.5e-7
    assert near.any(axis=1).sum() >= 3  # the exact path really ran
    check_rvq(p1, p2, n, ora, bits)


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_encode_special_rows(vq, oracle_mod, bits):
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    rows = []
    rows.append(np.zeros(D))                       # zero row
    e0 = np.zeros(D); e0[0] = 1.0; rows.append(e0)  # rotation is constant 1/sqrt(D)
    rows.append(-e0 * 3.0)
    big = np.full(D, 65504.0); big[::2] = -65504.0; rows.append(big)     # fp16 extremes
    rows.append(np.full(D, 2.0 ** -24))                                   # subnormals
    tiny = np.zeros(D); tiny[5] = 2.0 ** -24; tiny[77] = -3 * 2.0 ** -24; rows.append(tiny)
    mixed = np.linspace(-1000, 1000, D); mixed[3] = 2.0 ** -20; rows.append(mixed)
    onehot_pair = np.zeros(D); onehot_pair[1] = 1; onehot_pair[2] = 1; rows.append(onehot_pair)
    x = np.array(rows).astype(np.float16).reshape(1, 1, -1, D)
    p1, p2, n = _encode(vq, x, bits, cb)
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb)
    # rows whose y sits exactly on a boundary are ties by construction: any
    # mismatch must be tie-flagged, but the count is not held to the rate
    check_rvq(p1, p2, n, ora, bits, strict=False)
    assert n.reshape(-1)[0] == 0.0


@pytest.mark.parametrize("bits", [2, 4])
def test_encode_wide_dynamic_range_rows(vq, oracle_mod, bits):
    """Rows that stress the fast rotation's accumulation: one large value among
    values near the bottom of the fp16 range, and rows whose values spread
    over the whole fp16 exponent range.  Codes must still equal exact
    arithmetic (a row the fast path cannot decide is recomputed)."""
    rng = np.random.default_rng(2024 + bits)
    n = 1536
    x = rng.standard_normal((n, D)) * 2.0 ** rng.integers(-24, 0, (n, D))
    big = rng.integers(0, D, n)
    x[np.arange(n), big] = rng.choice([-1.0, 1.0], n) * 2.0 ** rng.integers(0, 16, n) * rng.uniform(1, 1.99, n)
    x[n // 2:] = rng.standard_normal((n - n // 2, D)) * 2.0 ** rng.integers(-14, 15, (n - n // 2, D))
    x = np.clip(x, -65504, 65504).astype(np.float16).reshape(1, 2, n // 2, D)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    p1, p2, nr = _encode(vq, x, bits, cb)
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb)
    check_rvq(p1, p2, nr, ora, bits)


def test_encode_custom_codebook_boundary_at_rotated_value(vq, oracle_mod):
    """A boundary placed at fp32(1/sqrt(D)) (where x = e_0 rotates to) forces the
    exact path; its decision must follow exact arithmetic."""
    bits = 2
    c1, b1, c2, b2 = oracle_mod.rvq_codebooks(D, bits)[:4]
    y0 = np.float32(1 / np.sqrt(128.0))
    b1x = np.array([-0.3, y0, 0.3], np.float32)
    c1x = np.array([-0.5, -0.1, 0.2, 0.5], np.float32)
    x = np.zeros((1, 1, 3, D), np.float16)
    x[0, 0, 0, 0] = 1.0
    x[0, 0, 1, 0] = 1.0
    x[0, 0, 1, 1] = 2.0 ** -11
    x[0, 0, 2, :] = np.float16(0.25)
    p1, p2, n = _encode(vq, x, bits, (c1x, b1x, c2, b2))
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, c1x, b1x, c2, b2)
    check_rvq(p1, p2, n, ora, bits, strict=False)
    g1 = unpack_rows(p1.reshape(-1, 8), bits)
    assert np.array_equal(g1[0], ora["idx1"][0])


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_encode_asymmetric_codebook(vq, oracle_mod, bits):
    """A codebook that is not antisymmetric takes the shuffle-table path."""
    c1, b1, c2, b2 = [a.copy() for a in oracle_mod.rvq_codebooks(D, bits)[:4]]
    L = 1 << bits
    c1[L // 2:] *= np.float32(1.3)
    b1[L // 2 - 1:] = np.float32(0.5) * (c1[L // 2 - 1:-1] + c1[L // 2:])
    c2[: L // 2] *= np.float32(0.8)
    b2[: L // 2] = np.float32(0.5) * (c2[: L // 2] + c2[1: L // 2 + 1])
    assert np.all(c1[:-1] < b1) and np.all(b1 < c1[1:]) and np.all(c2[:-1] < b2) and np.all(b2 < c2[1:])
    x = _rows((1, 2, 700), 77 + bits)
    p1, p2, n = _encode(vq, x, bits, (c1, b1, c2, b2))
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, c1, b1, c2, b2)
    check_rvq(p1, p2, n, ora, bits)


@pytest.mark.parametrize("outer", [0.24, 0.3])
def test_encode_symmetric_books_wide_boundaries(vq, oracle_mod, outer):
    """Symmetric 4-level books scaled so that the stage-1 outer boundary is
    `outer`: below 1/4 they take the tensor-core encoder (whose scaled boundary
    test is argued for B, E < 1/4), at 0.3 the shuffle-table encoder; both
    must equal exact arithmetic."""
    bits = 2
    c1, b1, c2, b2 = [a.astype(np.float64) for a in oracle_mod.rvq_codebooks(D, bits)[:4]]
    f = outer / b1[2]
    c1, b1, c2, b2 = [np.float32(f) * a.astype(np.float32) for a in (c1, b1, c2, b2)]
    assert b1[1] == 0 and np.all(c1 == -c1[::-1]) and np.all(b1 == -b1[::-1])
    x = _rows((1, 3, 800), 123, outliers=(4, 40.0))
    p1, p2, n = _encode(vq, x, bits, (c1, b1, c2, b2))
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, c1, b1, c2, b2)
    check_rvq(p1, p2, n, ora, bits)


@pytest.mark.parametrize("bits", [2, 4])
def test_encode_plain_count_fallback(vq, oracle_mod, bits):
    """A codebook with two boundaries inside one guard band has no lookup
    table; the encoder then counts boundaries one by one."""
    c1, b1, c2, b2 = [a.copy() for a in oracle_mod.rvq_codebooks(D, bits)[:4]]
    L = 1 << bits
    mid = L // 2
    b1[mid] = np.float32(1e-7)   # 1e-7 above the middle boundary b1[mid - 1] = 0
    c1[mid] = np.float32(5e-8)   # keep the centroid between its two boundaries
    assert np.all(c1[:-1] < b1) and np.all(b1 < c1[1:])
    x = _rows((1, 2, 300), 91 + bits)
    p1, p2, n = _encode(vq, x, bits, (c1, b1, c2, b2))
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, c1, b1, c2, b2)
    check_rvq(p1, p2, n, ora, bits)


def test_encode_dst_offsets(vq, oracle_mod):
    bits = 2
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    B, H, S, S_dst = 3, 2, 9, 48
    x = _rows((B, H, S), 55)
    off = np.array([0, 17, 39], np.int32)
    W = 8
    sentinel = np.int32(-1431655766)  # 0xAAAAAAAA
    p1 = torch.full((B, H, S_dst, W), int(sentinel), dtype=torch.int32, device="cuda")
    p2 = torch.full((B, H, S_dst, W), int(sentinel), dtype=torch.int32, device="cuda")
    nr = torch.full((B, H, S_dst), -1.0, dtype=torch.float32, device="cuda")
    vq.vq_rvq_encode_pack(_dev(x), bits, *cb, packed1=p1, packed2=p2, norms=nr,
                          dst_off=_dev(off), S_dst=S_dst)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    p1, p2, nr = p1.cpu().numpy(), p2.cpu().numpy(), nr.cpu().numpy()
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb)
    g1 = np.stack([p1[b, :, off[b]:off[b] + S] for b in range(B)])
    g2 = np.stack([p2[b, :, off[b]:off[b] + S] for b in range(B)])
    gn = np.stack([nr[b, :, off[b]:off[b] + S] for b in range(B)])
    check_rvq(g1, g2, gn, ora, bits)
    mask = np.ones((B, H, S_dst), bool)
    for b in range(B):
        mask[b, :, off[b]:off[b] + S] = False
    assert np.all(p1[mask] == sentinel) and np.all(nr[mask] == -1.0)


def test_encode_bad_offset_sets_device_error(vq, oracle_mod):
    bits = 2
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    x = _rows((2, 1, 8), 56)
    off = _dev(np.array([0, 30], np.int32))  # 30 + 8 > 32
    p1 = torch.zeros((2, 1, 32, 8), dtype=torch.int32, device="cuda")
    p2 = torch.zeros_like(p1)
    nr = torch.zeros((2, 1, 32), dtype=torch.float32, device="cuda")
    vq.vq_rvq_encode_pack(_dev(x), bits, *cb, packed1=p1, packed2=p2, norms=nr, dst_off=off, S_dst=32)
    assert vq.vq_device_error() & vq.VQ_DEVERR_BAD_OFFSET
    assert vq.vq_device_error() == 0  # cleared by the read
    assert torch.count_nonzero(p1[1]).item() == 0  # the bad batch was skipped
    assert torch.count_nonzero(nr[0]).item() > 0


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_decode_parity(vq, oracle_mod, bits):
    """GPU dequant of the oracle's packed codes vs the oracle's dequant."""
    x = _rows((1, 3, 999), 70 + bits)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb)
    ref, ref64 = oracle_mod.rvq_decode(ora["packed1"], ora["packed2"], ora["norms"], D, bits,
                                       cb[0], cb[2], want_f64=True)
    W = 4 * bits
    out = vq.vq_rvq_unpack_dequant(_dev(ora["packed1"].view(np.int32).reshape(1, 3, 999, W)),
                                   _dev(ora["packed2"].view(np.int32).reshape(1, 3, 999, W)),
                                   _dev(ora["norms"].reshape(1, 3, 999)), bits, cb[0], cb[2])
    got = out.cpu().numpy().reshape(-1, D).astype(np.float64)
    n = ora["norms"].astype(np.float64)[:, None]
    assert np.all(np.abs(got - ref64) <= 1e-3 * n + 1e-30)
    # fp32 arithmetic: most outputs also round to the same fp16 as binary64
    assert np.mean(got == ref.astype(np.float64)) > 0.95


@pytest.mark.parametrize("bits", [1, 2, 4])
@pytest.mark.parametrize("shape,signed", [((1, 1, 1), False), ((1, 1, 31), True), ((1, 1, 32), False),
                                          ((1, 1, 33), True), ((1, 2, 4000), False), ((3, 1, 6113), True)])
def test_decode_parity_shapes(vq, oracle_mod, bits, shape, signed):
    """Decode of a single row, one short block, exactly one 32-row block, one
    block and a row, and launches whose blocks do not fill the grid or end in
    a partial block (6113 = 191 blocks of 32 and one row at b = 2, 4; 382
    blocks of 16 and one row at b = 1), with and without the randomised signs;
    every output against the oracle's binary64 dequant."""
    x = _rows(shape, 90 + bits + shape[2])
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    signs = np.random.default_rng(91 + bits).integers(0, 2 ** 32, 4, dtype=np.uint32) if signed else None
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb, signs=signs)
    ref, ref64 = oracle_mod.rvq_decode(ora["packed1"], ora["packed2"], ora["norms"], D, bits,
                                       cb[0], cb[2], want_f64=True, signs=signs)
    W = 4 * bits
    B, H, S = shape
    out = vq.vq_rvq_unpack_dequant(_dev(ora["packed1"].view(np.int32).reshape(B, H, S, W)),
                                   _dev(ora["packed2"].view(np.int32).reshape(B, H, S, W)),
                                   _dev(ora["norms"].reshape(B, H, S)), bits, cb[0], cb[2], signs=signs)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    assert out.shape == (B, H, S, D)
    got = out.cpu().numpy().reshape(-1, D).astype(np.float64)
    n = ora["norms"].astype(np.float64)[:, None]
    assert np.all(np.abs(got - ref64) <= 1e-3 * n + 1e-30)
    if got.shape[0] >= 32:
        assert np.mean(got == ref.astype(np.float64)) > 0.95


def test_c1_full_parity_and_roundtrip(vq, oracle_mod):
    """TurboQuantRVQ b=2 on keys [1, 8, 512, 128] with per-channel scales."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    cfg = synth.CONFIGS["c1_rvq_b2_8x512"]
    x = synth.keys_for(cfg)
    bits = cfg["bits"]
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    p1, p2, n = _encode(vq, x, bits, cb)
    assert p1.shape == (1, 8, 512, 8)
    ora = oracle_mod.rvq_encode(x.reshape(-1, D), bits, *cb)
    check_rvq(p1, p2, n, ora, bits)
    out = vq.vq_rvq_unpack_dequant(_dev(p1), _dev(p2), _dev(n), bits, cb[0], cb[2])
    ref64 = oracle_mod.rvq_decode(ora["packed1"], ora["packed2"], ora["norms"], D, bits, cb[0],
                                  cb[2], want_f64=True)[1]
    got = out.cpu().numpy().reshape(-1, D).astype(np.float64)
    same = (ora["tie2"].reshape(-1, D).any(1) == 0)
    assert np.all(np.abs(got - ref64)[same] <= 1e-3 * ora["norms"][same, None])


def _sampled_rows(N, k, seed):
    rng = np.random.default_rng(seed)
    idx = np.unique(np.concatenate([rng.choice(N, k, replace=False), [0, N - 1]]))
    return idx


def test_c3_layer_full_size_sampled(vq, oracle_mod):
    """One layer of the 8k-context key cache at full size, b = 4, checked on
    sampled rows, in the launch configuration the benchmark uses."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    cfg = synth.CONFIGS["c3_rvq_b4_32L_8k"]
    bits = cfg["bits"]
    x = synth.keys_for(cfg, layer=5)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    p1, p2, n = _encode(vq, x, bits, cb)
    N = x.shape[1] * x.shape[2]
    idx = _sampled_rows(N, 3000, 1)
    ora = oracle_mod.rvq_encode(x.reshape(-1, D)[idx], bits, *cb)
    check_rvq(p1.reshape(N, -1)[idx], p2.reshape(N, -1)[idx], n.reshape(-1)[idx], ora, bits)
    dec = vq.vq_rvq_unpack_dequant(_dev(p1), _dev(p2), _dev(n), bits, cb[0], cb[2])
    got = dec.cpu().numpy().reshape(N, D)[idx].astype(np.float64)
    ref64 = oracle_mod.rvq_decode(ora["packed1"], ora["packed2"], ora["norms"], D, bits, cb[0],
                                  cb[2], want_f64=True)[1]
    clean = ora["tie2"].reshape(-1, D).any(1) == 0
    assert np.all(np.abs(got - ref64)[clean] <= 1e-3 * ora["norms"][clean, None])


def test_c4_decode_flush_offsets(vq, oracle_mod):
    """64 sequences x 8 heads x 128 new tokens flushed at random cache lengths."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    cfg = synth.CONFIGS["c4_decode_flush_64x8x128"]
    x = synth.keys_for(cfg)
    off = synth.cache_lengths(cfg["B"], cfg["seed"])
    S_dst = cfg["s_dst"]
    for bits in cfg["rvq_bits"]:
        cb = oracle_mod.rvq_codebooks(D, bits)[:4]
        p1, p2, n = _encode(vq, x, bits, cb, dst_off=_dev(off), S_dst=S_dst)
        rng = np.random.default_rng(bits)
        bsel = rng.choice(cfg["B"], 6, replace=False)
        for b in bsel:
            xs = x[b].reshape(-1, D)
            ora = oracle_mod.rvq_encode(xs, bits, *cb)
            g1 = p1[b, :, off[b]:off[b] + 128]
            g2 = p2[b, :, off[b]:off[b] + 128]
            gn = n[b, :, off[b]:off[b] + 128]
            check_rvq(g1, g2, gn, ora, bits)


def test_c5_keys_full_size_sampled(vq, oracle_mod):
    """Long-context keys [4, 32, 32768, 128] (1 GiB), b = 2, sampled rows."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    cfg = synth.CONFIGS["c5_long_32k"]
    bits = cfg["rvq_bits"]
    x = synth.keys_for(cfg)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    p1, p2, n = _encode(vq, x, bits, cb)
    N = x.size // D
    idx = _sampled_rows(N, 3000, 2)
    ora = oracle_mod.rvq_encode(x.reshape(-1, D)[idx], bits, *cb)
    check_rvq(p1.reshape(N, -1)[idx], p2.reshape(N, -1)[idx], n.reshape(-1)[idx], ora, bits)
