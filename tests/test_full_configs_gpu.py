"""Every code of the full-size configurations against the oracle (GB300).

The 8k-context key cache (32 layers of keys [1, 32, 8192, 128], b = 4), the
decode-time flush (64 sequences x 8 heads x 128 tokens into caches at random
lengths; RVQ b in {1, 2, 4}, KIVI b in {2, 4}) and the long-context flush (K
and V [4, 32, 32768, 128]; RVQ b = 2 on K, KIVI 2-bit G = 64 residual 128 on K
and V) run on the GPU through the C ABI, in the launch configuration the
benchmark times, and every output is checked: codes under the parity rule
(mismatches only where the oracle flags a tie, fewer than 1e-6 of codes),
norms, scale/zero, and both dequants of the GPU's own storage (KIVI
bit-exact, RVQ within 1e-3 * ||x||).  The oracle runs on every host core in
spawn-method worker processes (tests/full_parity.py); the counts are printed.
"""
import numpy as np
import pytest

import full_parity as fp

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

D = 128


@pytest.fixture(scope="module")
def vq():
    from kv_cache_quantization_turboquantrvq_gb300 import api, build
    build.build()
    api.lib()
    return api


@pytest.fixture(scope="module")
def pool(oracle_mod):
    with fp.Pool() as p:
        yield p


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _host(t):
    return t.cpu().numpy()


def _synced(vq):
    torch.cuda.synchronize()
    assert vq.vq_device_error() == 0


def test_c3_every_code_32_layers(vq, oracle_mod, pool):
    """b = 4 encode + decode of all 32 layers, every row."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    cfg = synth.CONFIGS["c3_rvq_b4_32L_8k"]
    bits, L = cfg["bits"], cfg["layers"]
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    jobs = []
    for layer in range(L):
        x = synth.keys_for(cfg, layer=layer)
        B, H, S, _ = x.shape
        p1, p2, n = vq.vq_rvq_encode_pack(_dev(x), bits, *cb)
        dec = vq.vq_rvq_unpack_dequant(p1, p2, n, bits, cb[0], cb[2])
        _synced(vq)
        P1, P2, N, DEC = _host(p1), _host(p2), _host(n), _host(dec)
        del p1, p2, n, dec
        tasks = [dict(x=x[0, h:h + 4].reshape(-1, D), p1=P1[0, h:h + 4], p2=P2[0, h:h + 4],
                      norms=N[0, h:h + 4], dec=DEC[0, h:h + 4], bits=bits, cb=cb)
                 for h in range(0, H, 4)]
        jobs.append(pool.submit(fp.rvq_slice, tasks))
    st = fp.merge(s for j in jobs for s in j.get())
    assert st["rows"] == L * 32 * 8192
    print("\n" + fp.assert_rule(st, ["s1_", "s2_"], "C3 RVQ b=4, 32 layers") +
          "; dequant max |err|/||x|| %.3g, %.4f of outputs equal the oracle's fp16" %
          (st["dec_max_rel"], st["dec_same_fp16"] / st["dec_values"]))


def test_c4_every_sequence(vq, oracle_mod, pool):
    """The decode-time flush: all 64 sequences, at their cache offsets, for every
    width; rows outside the flushed windows stay untouched."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    cfg = synth.CONFIGS["c4_decode_flush_64x8x128"]
    k = synth.keys_for(cfg)
    v = synth.values_for(cfg)
    off = synth.cache_lengths(cfg["B"], cfg["seed"])
    B, H, S, _ = k.shape
    S_dst, G = cfg["s_dst"], cfg["group"]
    kd, vd, offd = _dev(k), _dev(v), _dev(off)
    sentinel = -1431655766  # 0xAAAAAAAA
    reports = []
    for bits in cfg["rvq_bits"]:
        cb = oracle_mod.rvq_codebooks(D, bits)[:4]
        W = 4 * bits
        p1 = torch.full((B, H, S_dst, W), sentinel, dtype=torch.int32, device="cuda")
        p2 = torch.full_like(p1, sentinel)
        nr = torch.full((B, H, S_dst), -1.0, dtype=torch.float32, device="cuda")
        vq.vq_rvq_encode_pack(kd, bits, *cb, packed1=p1, packed2=p2, norms=nr, dst_off=offd, S_dst=S_dst)
        _synced(vq)
        P1, P2, N = _host(p1), _host(p2), _host(nr)
        tasks = [dict(x=k[b].reshape(-1, D), p1=P1[b, :, off[b]:off[b] + S], p2=P2[b, :, off[b]:off[b] + S],
                      norms=N[b, :, off[b]:off[b] + S], dec=None, bits=bits, cb=cb) for b in range(B)]
        st = fp.merge(pool.map(fp.rvq_slice, tasks))
        # (the tasks hold views of the outputs: blank the windows only now)
        for b in range(B):
            P1[b, :, off[b]:off[b] + S] = sentinel
            P2[b, :, off[b]:off[b] + S] = sentinel
            N[b, :, off[b]:off[b] + S] = -1.0
        assert np.all(P1 == sentinel) and np.all(P2 == sentinel) and np.all(N == -1.0)
        reports.append(fp.assert_rule(st, ["s1_", "s2_"], "C4 RVQ b=%d" % bits))
        del p1, p2, nr
    for bits in cfg["kivi_bits"]:
        out = vq.vq_kivi_quant_pack(kd, vd, bits, G, 0, dst_off=offd, S_dst=S_dst)
        _synced(vq)
        o = {name: _host(t) for name, t in out.items()}
        del out
        kt, vt = [], []
        for b in range(B):
            g0 = off[b] // G
            kt.append(dict(x=k[b:b + 1], per_channel=True, bits=bits, G=G, R=0, dec=None,
                           packed=o["k_packed"][b, :, g0:g0 + S // G], scale=o["k_scale"][b, :, g0:g0 + S // G],
                           zero=o["k_zero"][b, :, g0:g0 + S // G]))
            vt.append(dict(x=v[b:b + 1], per_channel=False, bits=bits, G=G, R=0, dec=None,
                           packed=o["v_packed"][b, :, off[b]:off[b] + S], scale=o["v_scale"][b, :, off[b]:off[b] + S],
                           zero=o["v_zero"][b, :, off[b]:off[b] + S]))
        reports.append(fp.assert_rule(fp.merge(pool.map(fp.kivi_slice, kt)), [""], "C4 KIVI keys b=%d" % bits))
        reports.append(fp.assert_rule(fp.merge(pool.map(fp.kivi_slice, vt)), [""], "C4 KIVI values b=%d" % bits))
    print("\n" + "\n".join(reports))


def test_c5_every_code(vq, oracle_mod, pool):
    """RVQ b = 2 on K and KIVI 2-bit G = 64 on K and V, [4, 32, 32768, 128],
    then both dequants: every row, group and output value."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    cfg = synth.CONFIGS["c5_long_32k"]
    k = synth.keys_for(cfg)
    v = synth.values_for(cfg)
    B, H, S, _ = k.shape
    bits, kb, G, R = cfg["rvq_bits"], cfg["kivi_bits"], cfg["group"], cfg["residual"]
    S_q = S - R
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    kd, vd = _dev(k), _dev(v)
    p1, p2, n = vq.vq_rvq_encode_pack(kd, bits, *cb)
    dec = vq.vq_rvq_unpack_dequant(p1, p2, n, bits, cb[0], cb[2])
    packs = vq.vq_kivi_quant_pack(kd, vd, kb, G, R)
    ko, vo = vq.vq_kivi_unpack_dequant(packs, B, H, S_q, kb, G)
    _synced(vq)
    P1, P2, N, DEC = _host(p1), _host(p2), _host(n), _host(dec)
    o = {name: _host(t) for name, t in packs.items()}
    KO, VO = _host(ko), _host(vo)
    del kd, vd, p1, p2, n, dec, packs, ko, vo
    torch.cuda.empty_cache()
    NG = o["k_packed"].shape[2]
    bh = [(b, h) for b in range(B) for h in range(H)]
    rj = pool.submit(fp.rvq_slice, [dict(x=k[b, h], p1=P1[b, h], p2=P2[b, h], norms=N[b, h], dec=DEC[b, h],
                                         bits=bits, cb=cb) for b, h in bh])
    kj = pool.submit(fp.kivi_slice, [dict(x=k[b:b + 1, h:h + 1], per_channel=True, bits=kb, G=G, R=R,
                                          packed=o["k_packed"][b, h], scale=o["k_scale"][b, h],
                                          zero=o["k_zero"][b, h], dec=KO[b, h]) for b, h in bh])
    vj = pool.submit(fp.kivi_slice, [dict(x=v[b:b + 1, h:h + 1], per_channel=False, bits=kb, G=G, R=R,
                                          packed=o["v_packed"][b, h], scale=o["v_scale"][b, h],
                                          zero=o["v_zero"][b, h], dec=VO[b, h]) for b, h in bh])
    sr, sk, sv = fp.merge(rj.get()), fp.merge(kj.get()), fp.merge(vj.get())
    assert sr["rows"] == B * H * S and sk["codes"] == B * H * S_q * D and NG == S_q // G
    print("\n" + fp.assert_rule(sr, ["s1_", "s2_"], "C5 RVQ b=2 keys") +
          "; dequant max |err|/||x|| %.3g" % sr["dec_max_rel"] + "\n" +
          fp.assert_rule(sk, [""], "C5 KIVI keys") + "\n" + fp.assert_rule(sv, [""], "C5 KIVI values"))
