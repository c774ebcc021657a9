"""The decode-time flush in one launch (vq_flush_decode) on GB300, through the
C ABI: every part equals the stand-alone calls bit for bit (RVQ encode of the
keys, KIVI keys and values, the fp16 window copy), rows outside the flushed
windows stay untouched, the whole decode flush (64 sequences x 8 heads x 128
tokens) matches the oracle for every sequence, and the call replays in a
CUDA graph."""
import numpy as np
import pytest

import full_parity as fp

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

D = 128
SENT = -1431655766  # 0xAAAAAAAA


@pytest.fixture(scope="module")
def vq():
    from kv_cache_quantization_turboquantrvq_gb300 import api, build
    build.build()
    api.lib()
    return api


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _filled(shape, dtype):
    if dtype == torch.int32:
        return torch.full(shape, SENT, dtype=dtype, device="cuda")
    return torch.full(shape, -7.0, dtype=dtype, device="cuda")


def _outputs(vq, B, H, S_dst, rbits, kbits, G, R_cap):
    W = vq.rvq_words(D, rbits)
    shp = vq.kivi_shapes(B, H, S_dst, D, kbits, G)
    return {
        "packed1": _filled((B, H, S_dst, W), torch.int32), "packed2": _filled((B, H, S_dst, W), torch.int32),
        "norms": _filled((B, H, S_dst), torch.float32),
        "k_packed": _filled(shp["k_packed"], torch.int32), "k_scale": _filled(shp["k_scale"], torch.float16),
        "k_zero": _filled(shp["k_scale"], torch.float16), "v_packed": _filled(shp["v_packed"], torch.int32),
        "v_scale": _filled(shp["v_scale"], torch.float16), "v_zero": _filled(shp["v_scale"], torch.float16),
        "k_win": _filled((B, H, R_cap, D), torch.float16), "v_win": _filled((B, H, R_cap, D), torch.float16),
    }


def _separate(vq, k, v, R, off, S_dst, rbits, kbits, G, outs, win_off):
    """The same flush as stand-alone calls (the reference for bit-identity)."""
    T = k.shape[2]
    cb = vq.vq_rvq_codebook(D, rbits)
    vq.vq_rvq_encode_pack(k[:, :, :T - R].contiguous(), rbits, *cb, packed1=outs["packed1"],
                          packed2=outs["packed2"], norms=outs["norms"], dst_off=off, S_dst=S_dst)
    vq.vq_kivi_quant_pack(k, v, kbits, G, R, outs=outs, dst_off=off, S_dst=S_dst)
    if R > 0:
        wo = np.zeros(k.shape[0], np.int32) if win_off is None else win_off.cpu().numpy()
        for b in range(k.shape[0]):
            outs["k_win"][b, :, wo[b]:wo[b] + R] = k[b, :, T - R:]
            outs["v_win"][b, :, wo[b]:wo[b] + R] = v[b, :, T - R:]


def _fused(vq, k, v, R, off, S_dst, rbits, kbits, G, outs, win_off, R_cap):
    cb = vq.vq_rvq_codebook(D, rbits)
    rvq = dict(bits=rbits, books=cb, packed1=outs["packed1"], packed2=outs["packed2"], norms=outs["norms"])
    kivi = dict(bits=kbits, group=G, **{n: outs[n] for n in ("k_packed", "k_scale", "k_zero", "v_packed",
                                                            "v_scale", "v_zero")})
    window = dict(k_win=outs["k_win"], v_win=outs["v_win"], win_off=win_off, R_cap=R_cap) if R > 0 else None
    return vq.vq_flush_decode(k, v, R, dst_off=off, S_dst=S_dst, rvq=rvq, kivi=kivi, window=window)


def _same(a, b):
    for n in a:
        assert torch.equal(a[n], b[n]), n


@pytest.mark.parametrize("rbits,kbits,G", [(1, 2, 32), (2, 2, 32), (4, 4, 32), (2, 4, 64), (4, 2, 64)])
@pytest.mark.parametrize("T,R", [(128, 0), (160, 32), (77, 13), (90, 10)])
def test_fused_equals_separate_calls(vq, rbits, kbits, G, T, R):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    B, H = 5, 3
    S_q = T - R
    k = _dev(synth.kv_tensor(B, H, T, D, 500 + T + rbits, 4, 20.0))
    v = _dev(synth.kv_tensor(B, H, T, D, 600 + T + kbits))
    # cache offsets: multiples of G; a ragged last key group must end the cache
    ragged = S_q % G != 0
    S_dst = 4 * G + S_q if not ragged else 3 * G + S_q
    off = _dev(np.array([0, G, 2 * G, 3 * G if not ragged else 2 * G, G], np.int32)[:B])
    if ragged:
        off = _dev(np.full(B, S_dst - S_q, np.int32))
    R_cap = R + 9
    win_off = _dev(np.array([0, 9, 3, 1, 9], np.int32)[:B]) if R > 0 else None
    ref = _outputs(vq, B, H, S_dst, rbits, kbits, G, max(R_cap, 1))
    got = _outputs(vq, B, H, S_dst, rbits, kbits, G, max(R_cap, 1))
    _separate(vq, k, v, R, off, S_dst, rbits, kbits, G, ref, win_off)
    _fused(vq, k, v, R, off, S_dst, rbits, kbits, G, got, win_off, R_cap)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    _same(ref, got)


@pytest.mark.parametrize("parts", ["rvq", "keys", "values", "window", "kivi", "rvq+window"])
def test_fused_single_parts(vq, parts):
    """Each part alone touches only its own outputs."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    B, H, T, R, G = 3, 2, 96, 32, 32
    k = _dev(synth.kv_tensor(B, H, T, D, 71, 4, 20.0))
    v = _dev(synth.kv_tensor(B, H, T, D, 72))
    off = _dev(np.array([0, 64, 32], np.int32))
    S_dst = 64 + T - R
    ref = _outputs(vq, B, H, S_dst, 2, 2, G, R)
    got = _outputs(vq, B, H, S_dst, 2, 2, G, R)
    _separate(vq, k, v, R, off, S_dst, 2, 2, G, ref, None)
    cb = vq.vq_rvq_codebook(D, 2)
    rvq = dict(bits=2, books=cb, packed1=got["packed1"], packed2=got["packed2"], norms=got["norms"])
    kw = {n: got[n] for n in ("k_packed", "k_scale", "k_zero", "v_packed", "v_scale", "v_zero")}
    window = dict(k_win=got["k_win"], v_win=got["v_win"], R_cap=R)
    use = {"rvq": dict(rvq=rvq), "keys": dict(kivi=dict(bits=2, group=G, values=False, **kw)),
           "values": dict(kivi=dict(bits=2, group=G, keys=False, **kw)), "window": dict(window=window),
           "kivi": dict(kivi=dict(bits=2, group=G, **kw)), "rvq+window": dict(rvq=rvq, window=window)}[parts]
    kin = None if parts == "values" else k
    vin = None if parts in ("rvq", "keys") else v
    if parts == "window":
        kin, vin = k, v
    vq.vq_flush_decode(kin, vin, R, dst_off=off, S_dst=S_dst, **use)
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0
    names = {"rvq": ["packed1", "packed2", "norms"], "keys": ["k_packed", "k_scale", "k_zero"],
             "values": ["v_packed", "v_scale", "v_zero"], "window": ["k_win", "v_win"]}
    wrote = set()
    for part in parts.replace("kivi", "keys+values").split("+"):
        wrote |= set(names[part])
    fresh = _outputs(vq, B, H, S_dst, 2, 2, G, R)
    for n in got:
        assert torch.equal(got[n], ref[n] if n in wrote else fresh[n]), n


def test_fused_bad_window_offset_sets_device_error(vq):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    B, H, T, R = 2, 2, 64, 16
    k = _dev(synth.kv_tensor(B, H, T, D, 81))
    v = _dev(synth.kv_tensor(B, H, T, D, 82))
    kw = torch.zeros((B, H, R, D), dtype=torch.float16, device="cuda")
    vw = torch.zeros_like(kw)
    bad = _dev(np.array([0, 5], np.int32))  # 5 + 16 > R_cap = 16
    vq.vq_flush_decode(k, v, R, window=dict(k_win=kw, v_win=vw, win_off=bad, R_cap=R))
    assert vq.vq_device_error() & vq.VQ_DEVERR_BAD_OFFSET
    assert vq.vq_device_error() == 0
    assert torch.equal(kw[0], k[0, :, T - R:]) and torch.count_nonzero(kw[1]).item() == 0


def test_fused_decode_flush_every_sequence_vs_oracle(vq, oracle_mod):
    """The decode-time flush (64 sequences x 8 heads x 128 new tokens into
    caches at random lengths), RVQ b = 2 and b = 4 keys with KIVI 2- and
    4-bit keys and values in one launch each: every code against the oracle."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    cfg = synth.CONFIGS["c4_decode_flush_64x8x128"]
    k_np, v_np = synth.keys_for(cfg), synth.values_for(cfg)
    off_np = synth.cache_lengths(cfg["B"], cfg["seed"])
    B, H, S, _ = k_np.shape
    S_dst, G = cfg["s_dst"], cfg["group"]
    k, v, off = _dev(k_np), _dev(v_np), _dev(off_np)
    reports = []
    with fp.Pool() as pool:
        for rbits, kbits in ((2, 2), (4, 4)):
            cb = oracle_mod.rvq_codebooks(D, rbits)[:4]
            outs = _outputs(vq, B, H, S_dst, rbits, kbits, G, 1)
            _fused(vq, k, v, 0, off, S_dst, rbits, kbits, G, outs, None, 0)
            torch.cuda.synchronize()
            assert vq.vq_device_error() == 0
            o = {n: t.cpu().numpy() for n, t in outs.items()}
            rt = [dict(x=k_np[b].reshape(-1, D), p1=o["packed1"][b, :, off_np[b]:off_np[b] + S],
                       p2=o["packed2"][b, :, off_np[b]:off_np[b] + S], norms=o["norms"][b, :, off_np[b]:off_np[b] + S],
                       dec=None, bits=rbits, cb=cb) for b in range(B)]
            kt = [dict(x=k_np[b:b + 1], per_channel=True, bits=kbits, G=G, R=0, dec=None,
                       packed=o["k_packed"][b, :, off_np[b] // G:off_np[b] // G + S // G],
                       scale=o["k_scale"][b, :, off_np[b] // G:off_np[b] // G + S // G],
                       zero=o["k_zero"][b, :, off_np[b] // G:off_np[b] // G + S // G]) for b in range(B)]
            vt = [dict(x=v_np[b:b + 1], per_channel=False, bits=kbits, G=G, R=0, dec=None,
                       packed=o["v_packed"][b, :, off_np[b]:off_np[b] + S],
                       scale=o["v_scale"][b, :, off_np[b]:off_np[b] + S],
                       zero=o["v_zero"][b, :, off_np[b]:off_np[b] + S]) for b in range(B)]
            reports.append(fp.assert_rule(fp.merge(pool.map(fp.rvq_slice, rt)), ["s1_", "s2_"],
                                          "fused flush RVQ b=%d" % rbits))
            reports.append(fp.assert_rule(fp.merge(pool.map(fp.kivi_slice, kt)), [""], "fused flush KIVI keys b=%d" % kbits))
            reports.append(fp.assert_rule(fp.merge(pool.map(fp.kivi_slice, vt)), [""], "fused flush KIVI values b=%d" % kbits))
            # nothing outside the flushed windows changed
            for b in range(B):
                o["packed1"][b, :, off_np[b]:off_np[b] + S] = SENT
                o["v_packed"][b, :, off_np[b]:off_np[b] + S] = SENT
                o["k_packed"][b, :, off_np[b] // G:off_np[b] // G + S // G] = SENT
            assert np.all(o["packed1"] == SENT) and np.all(o["v_packed"] == SENT) and np.all(o["k_packed"] == SENT)
    print("\n" + "\n".join(reports))


def test_fused_flush_replays_in_a_graph(vq):
    """Captured once, replayed with new tokens and offsets: each replay equals
    an eager call on the same inputs."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    B, H, T, R, G = 8, 4, 160, 32, 32
    S_dst = 1024
    k = _dev(synth.kv_tensor(B, H, T, D, 91, 4, 20.0))
    v = _dev(synth.kv_tensor(B, H, T, D, 92))
    off = _dev(np.arange(B, dtype=np.int32) * 64)
    woff = _dev(np.zeros(B, np.int32))
    got = _outputs(vq, B, H, S_dst, 2, 2, G, 64)
    vq.vq_rvq_codebook(D, 2)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _fused(vq, k, v, R, off, S_dst, 2, 2, G, got, woff, 64)  # warm-up: tables and module load
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _fused(vq, k, v, R, off, S_dst, 2, 2, G, got, woff, 64)
    for rep in range(3):
        k.copy_(_dev(synth.kv_tensor(B, H, T, D, 1000 + rep, 4, 20.0)))
        v.copy_(_dev(synth.kv_tensor(B, H, T, D, 2000 + rep)))
        off.copy_(_dev(np.random.default_rng(rep).permutation(B).astype(np.int32) * 64))
        woff.copy_(_dev(np.random.default_rng(rep).integers(0, 33, B).astype(np.int32)))
        g.replay()
        torch.cuda.synchronize()
        ref = _outputs(vq, B, H, S_dst, 2, 2, G, 64)
        for n in ref:
            ref[n].copy_(got[n])  # the replay's outputs, then overwrite the flushed parts eagerly
        _fused(vq, k, v, R, off, S_dst, 2, 2, G, ref, woff, 64)
        torch.cuda.synchronize()
        assert vq.vq_device_error() == 0
        _same(ref, got)
