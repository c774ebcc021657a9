"""The library's calls inside CUDA graphs.

Decode-time flushes and decode attention are launch-bound, so a caller
captures them once and replays the graph every step.  Every entry point
allocates nothing and never synchronizes, so it can be captured; a replay
after new inputs are copied into the captured buffers must give results
bit-identical to eager calls on the same inputs, and the replayed RVQ words
must agree with the oracle.
"""
import numpy as np
import pytest

from parity import check_rvq

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module")
def vq():
    from kv_cache_quantization_turboquantrvq_gb300 import api, build
    build.build()
    api.lib()
    return api


def _kv(B, H, T, seed):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    k = synth.kv_tensor(B, H, T, D, seed, 4, 20.0)
    v = synth.kv_tensor(B, H, T, D, seed + 1)
    return k, v


def _capture(fn, stream):
    """Run fn once eagerly on `stream` (first-use set-up), then capture it."""
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def test_decode_flush_graph_replays_match_eager_and_oracle(vq, oracle_mod):
    """128 new tokens per sequence into caches at per-sequence offsets: RVQ
    b=2 on K and KIVI 2-bit G=32 on K and V, captured as one graph."""
    B, H, T, S_dst, bits, G = 3, 2, 128, 640, 2, 32
    dev = torch.device("cuda")
    c1, b1, c2, b2 = oracle_mod.rvq_codebooks(D, bits)[:4]
    k_in = torch.empty((B, H, T, D), dtype=torch.float16, device=dev)
    v_in = torch.empty_like(k_in)
    off = torch.tensor([0, 256, 512], dtype=torch.int32, device=dev)
    W = D * bits // 32

    def buffers():
        rvq = [torch.zeros((B, H, S_dst, W), dtype=torch.int32, device=dev),
               torch.zeros((B, H, S_dst, W), dtype=torch.int32, device=dev),
               torch.zeros((B, H, S_dst), dtype=torch.float32, device=dev)]
        shp = vq.kivi_shapes(B, H, S_dst, D, bits, G)
        kivi = {"k_packed": torch.zeros(shp["k_packed"], dtype=torch.int32, device=dev),
                "k_scale": torch.zeros(shp["k_scale"], dtype=torch.float16, device=dev),
                "k_zero": torch.zeros(shp["k_scale"], dtype=torch.float16, device=dev),
                "v_packed": torch.zeros(shp["v_packed"], dtype=torch.int32, device=dev),
                "v_scale": torch.zeros(shp["v_scale"], dtype=torch.float16, device=dev),
                "v_zero": torch.zeros(shp["v_scale"], dtype=torch.float16, device=dev)}
        return rvq, kivi

    def flush(k, v, rvq, kivi):
        vq.vq_rvq_encode_pack(k, bits, c1, b1, c2, b2, packed1=rvq[0], packed2=rvq[1], norms=rvq[2],
                              dst_off=off, S_dst=S_dst)
        vq.vq_kivi_quant_pack(k, v, bits, G, 0, outs=kivi, dst_off=off, S_dst=S_dst)

    g_rvq, g_kivi = buffers()
    side = torch.cuda.Stream()
    k0, v0 = _kv(B, H, T, 1500)
    k_in.copy_(torch.from_numpy(k0))
    v_in.copy_(torch.from_numpy(v0))
    graph = _capture(lambda: flush(k_in, v_in, g_rvq, g_kivi), side)
    for step, seed in enumerate((1510, 1520)):
        k, v = _kv(B, H, T, seed)
        k_in.copy_(torch.from_numpy(k))
        v_in.copy_(torch.from_numpy(v))
        graph.replay()
        e_rvq, e_kivi = buffers()
        flush(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), e_rvq, e_kivi)
        torch.cuda.synchronize()
        assert vq.vq_device_error() == 0
        for a, b in zip(g_rvq, e_rvq):
            assert torch.equal(a, b), "RVQ outputs of the replay differ from the eager call"
        for n in e_kivi:
            assert torch.equal(g_kivi[n], e_kivi[n]), "KIVI %s of the replay differs" % n
        ora = oracle_mod.rvq_encode(k.reshape(-1, D), bits, c1, b1, c2, b2)
        offs = off.cpu().numpy()
        rows = lambda t: np.concatenate([t.cpu().numpy()[b, :, o:o + T] for b, o in enumerate(offs)])
        check_rvq(rows(g_rvq[0]), rows(g_rvq[1]), rows(g_rvq[2]), ora, bits)


def test_attention_graphs_replay_bit_identical(vq, oracle_mod):
    """RVQ attention (workspace and no-alloc variants) and KIVI attention
    captured once, replayed with new queries and lengths."""
    B, Hkv, gq, S, bits, G, R = 4, 2, 4, 1024, 2, 32, 16
    Hq = Hkv * gq
    dev = torch.device("cuda")
    rng = np.random.default_rng(1600)
    W = D * bits // 32
    p1 = torch.from_numpy(rng.integers(0, 2 ** 32, (B, Hkv, S, W), dtype=np.uint32).view(np.int32)).cuda()
    p2 = torch.from_numpy(rng.integers(0, 2 ** 32, (B, Hkv, S, W), dtype=np.uint32).view(np.int32)).cuda()
    nr = torch.from_numpy(rng.uniform(4.0, 24.0, (B, Hkv, S)).astype(np.float32)).cuda()
    v = torch.from_numpy(rng.standard_normal((B, Hkv, S, D)).astype(np.float16)).cuda()
    c1, _, c2, _ = oracle_mod.rvq_codebooks(D, bits)[:4]
    shp = vq.kivi_shapes(B, Hkv, S, D, bits, G)
    ri = lambda shape: torch.from_numpy(rng.integers(0, 2 ** 32, shape, dtype=np.uint32).view(np.int32)).cuda()
    cache = {"k_packed": ri(shp["k_packed"]), "v_packed": ri(shp["v_packed"]),
             "k_scale": torch.from_numpy(rng.uniform(0.05, 0.5, shp["k_scale"]).astype(np.float16)).cuda(),
             "k_zero": torch.from_numpy(rng.standard_normal(shp["k_scale"]).astype(np.float16)).cuda(),
             "v_scale": torch.from_numpy(rng.uniform(0.05, 0.5, shp["v_scale"]).astype(np.float16)).cuda(),
             "v_zero": torch.from_numpy(rng.standard_normal(shp["v_scale"]).astype(np.float16)).cuda()}
    kr = torch.from_numpy(rng.standard_normal((B, Hkv, R, D)).astype(np.float16)).cuda()
    vr = torch.from_numpy(rng.standard_normal((B, Hkv, R, D)).astype(np.float16)).cuda()
    q = torch.empty((B, Hq, D), dtype=torch.float16, device=dev)
    lens = torch.empty(B, dtype=torch.int32, device=dev)
    res = torch.empty(B, dtype=torch.int32, device=dev)
    ws = torch.empty((vq.vq_rvq_attend_workspace(B, Hq, Hkv, S) + 3) // 4, dtype=torch.float32, device=dev)
    kws = torch.empty((vq.vq_kivi_attend_workspace(B, Hq, Hkv, S, R) + 3) // 4, dtype=torch.float32, device=dev)
    outs = [torch.empty((B, Hq, D), dtype=torch.float16, device=dev) for _ in range(3)]

    def calls(o):
        vq.vq_rvq_attend(q, p1, p2, nr, v, bits, c1, c2, 0.1, lens=lens, out=o[0], workspace=ws)
        vq.vq_rvq_attend_noalloc(q, p1, p2, nr, v, bits, c1, c2, 0.1, lens=lens, out=o[1])
        vq.vq_kivi_attend(q, cache, bits, G, 0.1, k_res=kr, v_res=vr, lens=lens, res_lens=res, out=o[2],
                          workspace=kws)

    q.copy_(torch.from_numpy(rng.standard_normal((B, Hq, D)).astype(np.float16)))
    lens.copy_(torch.tensor([S, 1, 700, 0], dtype=torch.int32))
    res.copy_(torch.tensor([R, 3, 0, 5], dtype=torch.int32))
    graph = _capture(lambda: calls(outs), torch.cuda.Stream())
    for step in range(2):
        qn = rng.standard_normal((B, Hq, D)).astype(np.float16)
        ln = rng.integers(0, S + 1, B).astype(np.int32)
        rn = rng.integers(0, R + 1, B).astype(np.int32)
        q.copy_(torch.from_numpy(qn))
        lens.copy_(torch.from_numpy(ln))
        res.copy_(torch.from_numpy(rn))
        graph.replay()
        torch.cuda.synchronize()
        got = [o.clone() for o in outs]
        eager = [torch.empty_like(o) for o in outs]
        calls(eager)
        torch.cuda.synchronize()
        assert vq.vq_device_error() == 0
        for a, b in zip(got, eager):
            assert torch.equal(a, b), "attention replay differs from the eager call"
        assert torch.equal(got[0], got[1])  # same chunking: the no-alloc variant is bit-identical
