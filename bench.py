#!/usr/bin/env python3
"""Benchmark of the KV-cache flush path on GB300.

One step = one pass of the whole path over one batch of synthetic KV data:
TurboQuantRVQ encode+pack, KIVI quant+pack of K and V, then unpack+dequant of
all three.  Metric: HBM GB/s of algorithmic bytes (fp16 in + packed / norms /
scales out, and the reverse for the dequant kernels) per second, with the
fraction of the measured GB300 copy bandwidth, plus Gelem/s.

Default workload (N = 1): K and V [4, 32, 32768, 128] fp16 (long-context
stress), RVQ b = 2 on K, KIVI 2-bit G = 64 with a 128-token residual window on
K and V.  Inputs are 2 GiB, larger than L2 (129 MB), so no L2 flush is needed
between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload c5|c3|c2|c1|c4|attn|kattn|qjl]

--impl reference times the CPU oracle (single-threaded binary64 C) on a
bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

D = 128
METRIC = "fused KV quantize+pack HBM GB/s (% of GB300 peak) and Gelem/s, 1 GPU"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# --------------------------------------------------------------------------- workloads


class Op:
    """One timed call.  `launches` counts the launches of `kernel` (per-launch
    figures divide by it); `gpu_launches` counts every kernel the call starts."""

    def __init__(self, name, kernel, run, nbytes, nelem, launches=1, gpu_launches=None, stream=None):
        self.name, self.kernel, self.run = name, kernel, run
        self.nbytes, self.nelem, self.launches = nbytes, nelem, launches
        self.gpu_launches = launches if gpu_launches is None else gpu_launches
        self.stream = stream  # the stream the call launches on (None: the step's stream)


def rvq_bytes(rows, bits, d=D):
    """Algorithmic bytes of RVQ encode (or decode) of `rows` rows of width d:
    the fp16 row, two streams of floor(32/b)-code words and the fp32 norm."""
    return rows * (2 * d + 2 * 4 * -(-d // (32 // bits)) + 4)


def kivi_bytes(bh, s_q, bits, G, per_channel):
    n = bh * s_q * D
    ng = (s_q + G - 1) // G if per_channel else s_q
    groups = bh * ng * (D if per_channel else D // G)
    words = bh * ng * G * bits // 32 * D if per_channel else bh * s_q * D * bits // 32
    return n * 2 + words * 4 + groups * 4


def attend_bytes(lens, Hkv, Hq, bits):
    """Algorithmic bytes of one decode-attention call: every valid key's two
    code streams, norm and fp16 value row, plus the queries in and outputs out."""
    keys = int(np.sum(np.asarray(lens, np.int64))) * Hkv
    return keys * (2 * (D * bits // 8) + 4 + 2 * D) + len(lens) * Hq * D * 2 * 2


def qjl_bytes(rows, m):
    """Algorithmic bytes of QJL encode: the fp16 key rows in, m sign bits and
    an fp16 norm per row out."""
    return rows * (2 * D + m // 8 + 2)


def kattend_bytes(lens, res_lens, Hkv, Hq, bits, G):
    """Algorithmic bytes of one KIVI attention call: every valid quantized
    token's key and value codes, its share of the key group's scale/zero and
    its value groups' scales/zeros, every residual token's fp16 key and value
    rows, plus the queries in and outputs out."""
    per_tok = 2 * (D * bits // 8) + 4 * D // G + 4 * (D // G)
    q = int(np.sum(np.asarray(lens, np.int64))) * Hkv * per_tok
    r = int(np.sum(np.asarray(res_lens, np.int64))) * Hkv * 4 * D
    return q + r + len(lens) * Hq * D * 2 * 2


def describe(name):
    return {
        "kattn": "decode attention over KIVI 2-bit G=32 caches with the dequantization inside: 64 seqs x 8 kv "
                 "heads x 32 query heads, capacity 16384 (lengths uniform in [1k,16k]) + 128-token fp16 window",
        "attn": "decode attention over RVQ b=2 key caches (fp16 values): 64 seqs x 8 kv heads x "
                "32 query heads, capacity 16384, lengths uniform in [1k,16k]",
        "qjl": "QJL encode of long-context keys [4,32,32768,128] fp16 (4x40 outlier channels per head): "
               "128 sign bits of S x (seeded N(0,1) fp16 sketch) and the fp16 norm per key",
        "c5": "long-context K,V [4,32,32768,128] fp16 (4x40 outlier channels per head): RVQ b=2 "
              "encode+pack on K; KIVI 2-bit G=64 residual 128 on K and V; unpack+dequant of all",
        "c3": "RVQ b=4 encode+pack over 32 layers of keys [1,32,8192,128] fp16 (4x20 outliers), "
              "then unpack+dequant",
        "c2": "KIVI 2-bit flush on K,V [1,32,4096,128] G=32 residual 128, then unpack+dequant",
        "c1": "RVQ b=2 encode+pack of keys [1,8,512,128], then unpack+dequant",
        "c4": "decode flush: 64 seqs x 8 heads x 128 new tokens into caches of random lengths; "
              "RVQ b=2 on K and KIVI 2-bit G=32 on K and V, written at the sequences' offsets, "
              "in one launch (vq_flush_decode)",
        "c4s": "decode flush: 64 seqs x 8 heads x 128 new tokens into caches of random lengths; "
               "RVQ b=2 on K and KIVI 2-bit G=32 on K and V, written at the sequences' offsets, "
               "as three separate calls",
        "gen": "RVQ encode+pack then unpack+dequant at the general widths: keys [4,32,32768,64] b=2, "
               "[1,32,32768,256] b=4 and [2,32,32768,128] b=3 (ten 3-bit codes per word), fp16 N(0,1) "
               "with 4x20 outlier channels per head",
    }[name]


def max_over_ranks(x: float, world: int, dev) -> float:
    """The largest of the ranks' values of x (a time): an all-reduce MAX on a
    one-element tensor on `dev` (the rank's GPU under NCCL, the CPU under gloo)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard_configs(rank: int) -> dict:
    """The named configurations with rank-dependent seeds: under torchrun every
    rank processes its own shard (same shapes, independent data)."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    return {k: dict(v, seed=v["seed"] + 100003 * rank) for k, v in synth.CONFIGS.items()}


def build_workload(name, dev, rank=0, layers=None, batch=None, chunked=False, chunk_stream=None, lanes=None):
    """Device buffers and the op list for one step; also host inputs for e2e.

    With chunked=True, also returns the same step split into chunks that own
    their inputs (views of the full device inputs), ops and results, for the
    pipelined end-to-end measurement (C5: per batch, C3: per layer).  C3 with
    `lanes` (a list of streams): layer l launches on lanes[l % len(lanes)]."""
    import torch
    from kv_cache_quantization_turboquantrvq_gb300 import api, synth

    ops, inputs, results = [], [], []
    stream = torch.cuda.current_stream()

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def rvq_ops(tag, k_dev, bits, dst_off=None, S_dst=None, ops=ops, results=results, stream=stream):
        B, H, S, _ = k_dev.shape
        S_dst = S if S_dst is None else S_dst
        cb = [np.ascontiguousarray(a) for a in api.vq_rvq_codebook(D, bits)]
        W = D * bits // 32
        p1 = torch.empty((B, H, S_dst, W), dtype=torch.int32, device=dev)
        p2 = torch.empty_like(p1)
        nr = torch.empty((B, H, S_dst), dtype=torch.float32, device=dev)
        out = torch.empty((B, H, S, D), dtype=torch.float16, device=dev)
        rows = B * H * S

        def enc():
            api.vq_rvq_encode_pack(k_dev, bits, *cb, packed1=p1, packed2=p2, norms=nr,
                                   dst_off=dst_off, S_dst=S_dst, stream=stream)

        if dst_off is None:
            def dec():
                api.vq_rvq_unpack_dequant(p1, p2, nr, bits, cb[0], cb[2], out=out, stream=stream)
        else:
            dec = None
        # the library's books take the tensor-core encoders (b = 2: symmetric
        # books, b = 4: the pair table)
        ekern = "rvq_encode_tc_kernel" if bits in (2, 4) else "rvq_encode_kernel"
        ops.append(Op(tag + "rvq_encode", ekern, enc, rvq_bytes(rows, bits), rows * D, stream=stream))
        if dec is not None:
            dkern = "rvq_decode_row_kernel" if bits in (2, 4) else "rvq_decode_kernel"
            ops.append(Op(tag + "rvq_decode", dkern, dec, rvq_bytes(rows, bits), rows * D, stream=stream))
        results.extend([p1, p2, nr])
        if dec is not None:
            results.append(out)  # the round trip's reconstruction leaves the device too

    def kivi_ops(tag, k_dev, v_dev, bits, G, R, dst_off=None, S_dst=None, ops=ops, results=results,
                 stream=stream):
        B, H, S, _ = k_dev.shape
        S_q = S - R
        S_dst = S_q if S_dst is None else S_dst
        shp = api.kivi_shapes(B, H, S_dst, D, bits, G)
        outs = {
            "k_packed": torch.empty(shp["k_packed"], dtype=torch.int32, device=dev),
            "k_scale": torch.empty(shp["k_scale"], dtype=torch.float16, device=dev),
            "k_zero": torch.empty(shp["k_scale"], dtype=torch.float16, device=dev),
            "v_packed": torch.empty(shp["v_packed"], dtype=torch.int32, device=dev),
            "v_scale": torch.empty(shp["v_scale"], dtype=torch.float16, device=dev),
            "v_zero": torch.empty(shp["v_scale"], dtype=torch.float16, device=dev),
        }
        ko = torch.empty((B, H, S_q, D), dtype=torch.float16, device=dev)
        vo = torch.empty_like(ko)
        kb = kivi_bytes(B * H, S_q, bits, G, True)
        vb = kivi_bytes(B * H, S_q, bits, G, False)
        ops.append(Op(tag + "kivi_quant_k", "kivi_keys_kernel", lambda: api.vq_kivi_quant_pack(
            k_dev, None, bits, G, R, outs=outs, dst_off=dst_off, S_dst=S_dst, stream=stream), kb, B * H * S_q * D))
        ops.append(Op(tag + "kivi_quant_v", "kivi_values_kernel", lambda: api.vq_kivi_quant_pack(
            None, v_dev, bits, G, R, outs=outs, dst_off=dst_off, S_dst=S_dst, stream=stream), vb, B * H * S_q * D))
        if dst_off is None:
            ops.append(Op(tag + "kivi_dequant_k", "kivi_keys_dequant_kernel", lambda: api.vq_kivi_unpack_dequant(
                outs, B, H, S_q, bits, G, k_out=ko, want_v=False, stream=stream), kb, B * H * S_q * D))
            ops.append(Op(tag + "kivi_dequant_v", "kivi_values_dequant_kernel", lambda: api.vq_kivi_unpack_dequant(
                outs, B, H, S_q, bits, G, v_out=vo, want_k=False, stream=stream), vb, B * H * S_q * D))
        results.extend(outs.values())
        if dst_off is None:
            results.extend([ko, vo])

    chunks = []

    def new_chunk(chunk_inputs):
        c = {"inputs": chunk_inputs, "ops": [], "results": []}
        chunks.append(c)
        return c

    cfgs = shard_configs(rank)
    if name == "c5":
        cfg = cfgs["c5_long_32k"]
        k_np, v_np = synth.keys_for(cfg, B=batch), synth.values_for(cfg, B=batch)
        k, v = t(k_np), t(v_np)
        inputs = [(k_np, k), (v_np, v)]
        rvq_ops("", k, cfg["rvq_bits"])
        kivi_ops("", k, v, cfg["kivi_bits"], cfg["group"], cfg["residual"])
        # order the step as the path runs: encode everything, then decode everything
        order = ["rvq_encode", "kivi_quant_k", "kivi_quant_v", "rvq_decode", "kivi_dequant_k", "kivi_dequant_v"]
        ops.sort(key=lambda o: order.index(o.name))
        if chunked:
            for b in range(k.shape[0]):
                c = new_chunk([(k_np[b:b + 1], k[b:b + 1]), (v_np[b:b + 1], v[b:b + 1])])
                rvq_ops("", k[b:b + 1], cfg["rvq_bits"], ops=c["ops"], results=c["results"], stream=chunk_stream)
                kivi_ops("", k[b:b + 1], v[b:b + 1], cfg["kivi_bits"], cfg["group"], cfg["residual"],
                         ops=c["ops"], results=c["results"], stream=chunk_stream)
                c["ops"].sort(key=lambda o: order.index(o.name))
    elif name == "qjl":
        cfg = cfgs["qjl_long_32k_m128"]
        k_np = synth.keys_for(cfg, B=batch)
        k = t(k_np)
        m = cfg["m"]
        s_dev = t(np.random.default_rng(cfg["seed"]).standard_normal((m, D)).astype(np.float16))
        inputs = [(k_np, k)]

        def qjl_op(kd, ops_, results_, st):
            Bq, H, S, _ = kd.shape
            pk = torch.empty((Bq, H, S, m // 32), dtype=torch.int32, device=dev)
            nr = torch.empty((Bq, H, S), dtype=torch.float16, device=dev)
            ops_.append(Op("qjl_encode", "qjl_encode_tc_kernel",
                           lambda: api.vq_qjl_encode(kd, s_dev, packed=pk, norms=nr, stream=st),
                           qjl_bytes(Bq * H * S, m), Bq * H * S * D))
            results_.extend([pk, nr])
        qjl_op(k, ops, results, stream)
        if chunked:
            for b in range(k.shape[0]):
                c = new_chunk([(k_np[b:b + 1], k[b:b + 1])])
                qjl_op(k[b:b + 1], c["ops"], c["results"], chunk_stream)
    elif name == "c3":
        cfg = cfgs["c3_rvq_b4_32L_8k"]
        for layer in range(cfg["layers"] if layers is None else layers):
            k_np = synth.keys_for(cfg, layer=layer)
            k = t(k_np)
            inputs.append((k_np, k))
            rvq_ops("L%02d_" % layer, k, cfg["bits"], stream=stream if lanes is None else lanes[layer % len(lanes)])
            if chunked:
                c = new_chunk([(k_np, k)])
                rvq_ops("L%02d_" % layer, k, cfg["bits"], ops=c["ops"], results=c["results"], stream=chunk_stream)
        ops.sort(key=lambda o: (not o.kernel.startswith("rvq_encode"), o.name))
    elif name == "gen":
        # the general-width path (rvq_generic.cu): other widths and b = 3
        for tag, (Bg, Dg, bits) in (("D64b2_", (4, 64, 2)), ("D256b4_", (1, 256, 4)), ("D128b3_", (2, 128, 3))):
            xg_np = synth.kv_tensor(Bg, 32, 32768, Dg, 120 + Dg + bits, 4, 20.0)
            xg = t(xg_np)
            inputs.append((xg_np, xg))
            cbg = [np.ascontiguousarray(a) for a in api.vq_rvq_codebook(Dg, bits)]
            Wg = api.rvq_words(Dg, bits)
            rows = Bg * 32 * 32768
            g1 = torch.empty((Bg, 32, 32768, Wg), dtype=torch.int32, device=dev)
            g2 = torch.empty_like(g1)
            gn = torch.empty((Bg, 32, 32768), dtype=torch.float32, device=dev)
            go = torch.empty_like(xg)

            def genc(xg=xg, bits=bits, cbg=cbg, g1=g1, g2=g2, gn=gn):
                api.vq_rvq_encode_pack(xg, bits, *cbg, packed1=g1, packed2=g2, norms=gn, stream=stream)

            def gdec(bits=bits, cbg=cbg, g1=g1, g2=g2, gn=gn, go=go, Dg=Dg):
                api.vq_rvq_unpack_dequant(g1, g2, gn, bits, cbg[0], cbg[2], out=go, stream=stream, D=Dg)
            ops.append(Op(tag + "rvq_encode", "rvq_generic_encode_kernel<%d, %d>" % (Dg, bits), genc,
                          rvq_bytes(rows, bits, Dg), rows * Dg))
            ops.append(Op(tag + "rvq_decode", "rvq_generic_decode_kernel<%d, %d>" % (Dg, bits), gdec,
                          rvq_bytes(rows, bits, Dg), rows * Dg))
            results.extend([g1, g2, gn, go])
    elif name == "c2":
        cfg = cfgs["c2_kivi_b2_32x4096"]
        k_np, v_np = synth.keys_for(cfg), synth.values_for(cfg)
        k, v = t(k_np), t(v_np)
        inputs = [(k_np, k), (v_np, v)]
        kivi_ops("", k, v, cfg["bits"], cfg["group"], cfg["residual"])
    elif name == "c1":
        cfg = cfgs["c1_rvq_b2_8x512"]
        k_np = synth.keys_for(cfg)
        k = t(k_np)
        inputs = [(k_np, k)]
        rvq_ops("", k, cfg["bits"])
    elif name in ("c4", "c4s"):
        cfg = cfgs["c4_decode_flush_64x8x128"]
        k_np, v_np = synth.keys_for(cfg), synth.values_for(cfg)
        k, v = t(k_np), t(v_np)
        off = t(synth.cache_lengths(cfg["B"], cfg["seed"]))
        inputs = [(k_np, k), (v_np, v)]
        if name == "c4s":  # the same flush as three separate calls
            rvq_ops("", k, 2, dst_off=off, S_dst=cfg["s_dst"])
            kivi_ops("", k, v, 2, cfg["group"], 0, dst_off=off, S_dst=cfg["s_dst"])
        else:  # one launch (vq_flush_decode): RVQ b=2 keys, KIVI 2-bit keys and values
            Bc, Hc, Sc, G, S_dst = cfg["B"], cfg["H"], cfg["S"], cfg["group"], cfg["s_dst"]
            cbf = [np.ascontiguousarray(a) for a in api.vq_rvq_codebook(D, 2)]
            shp = api.kivi_shapes(Bc, Hc, S_dst, D, 2, G)
            fo = {"packed1": torch.empty((Bc, Hc, S_dst, 8), dtype=torch.int32, device=dev),
                  "packed2": torch.empty((Bc, Hc, S_dst, 8), dtype=torch.int32, device=dev),
                  "norms": torch.empty((Bc, Hc, S_dst), dtype=torch.float32, device=dev),
                  "k_packed": torch.empty(shp["k_packed"], dtype=torch.int32, device=dev),
                  "k_scale": torch.empty(shp["k_scale"], dtype=torch.float16, device=dev),
                  "k_zero": torch.empty(shp["k_scale"], dtype=torch.float16, device=dev),
                  "v_packed": torch.empty(shp["v_packed"], dtype=torch.int32, device=dev),
                  "v_scale": torch.empty(shp["v_scale"], dtype=torch.float16, device=dev),
                  "v_zero": torch.empty(shp["v_scale"], dtype=torch.float16, device=dev)}
            rows = Bc * Hc * Sc

            def flush(stream=stream):
                api.vq_flush_decode(k, v, 0, dst_off=off, S_dst=S_dst,
                                    rvq=dict(bits=2, books=cbf, packed1=fo["packed1"], packed2=fo["packed2"],
                                             norms=fo["norms"]),
                                    kivi=dict(bits=2, group=G, **{n: fo[n] for n in fo if n[0] in "kv"}),
                                    stream=stream)
            nb = rvq_bytes(rows, 2) + kivi_bytes(Bc * Hc, Sc, 2, G, True) + kivi_bytes(Bc * Hc, Sc, 2, G, False)
            ops.append(Op("flush_decode", "vq_flush_kernel", flush, nb, 2 * rows * D))
            results.extend(fo.values())
    elif name == "attn":
        # the cache (codes, norms, values) is resident state; a step's input is
        # the batch of queries and its result the attention output
        cfg = cfgs["attn_decode_64x8x32_16k"]
        B, Hkv, Hq, S, bits = cfg["B"], cfg["Hkv"], cfg["Hq"], cfg["S_cap"], cfg["bits"]
        B = B if batch is None else batch
        lens_np = synth.cache_lengths(B, cfg["seed"])
        rng = np.random.default_rng(cfg["seed"])
        W = D * bits // 32
        g = torch.Generator(device=dev)
        g.manual_seed(cfg["seed"])
        p1 = torch.randint(-2 ** 31, 2 ** 31 - 1, (B, Hkv, S, W), dtype=torch.int32, device=dev, generator=g)
        p2 = torch.randint(-2 ** 31, 2 ** 31 - 1, (B, Hkv, S, W), dtype=torch.int32, device=dev, generator=g)
        nr = torch.empty((B, Hkv, S), dtype=torch.float32, device=dev).uniform_(4.0, 24.0, generator=g)
        vv = torch.randn((B, Hkv, S, D), dtype=torch.float16, device=dev, generator=g)
        q_np = rng.standard_normal((B, Hq, D)).astype(np.float16)
        q, lens = t(q_np), t(lens_np)
        c1, _, c2, _ = [np.ascontiguousarray(a) for a in api.vq_rvq_codebook(D, bits)]
        out = torch.empty((B, Hq, D), dtype=torch.float16, device=dev)
        ws = torch.empty((max(api.vq_rvq_attend_workspace(B, Hq, Hkv, S), 16) + 3) // 4,
                         dtype=torch.float32, device=dev)
        nsplit = 2 if ws.numel() > 4 else 1

        def att(stream=stream):
            api.vq_rvq_attend(q, p1, p2, nr, vv, bits, c1, c2, 1.0 / np.sqrt(D), lens=lens, out=out,
                              workspace=ws, stream=stream)
        ops.append(Op("rvq_attend", "rvq_attend_kernel", att, attend_bytes(lens_np, Hkv, Hq, bits),
                      int(lens_np.sum()) * Hkv * D, gpu_launches=nsplit))
        inputs = [(q_np, q)]
        results.append(out)
        if chunked:
            c = new_chunk(inputs)
            c["ops"] = [Op("rvq_attend", "rvq_attend_kernel", lambda: att(chunk_stream),
                           attend_bytes(lens_np, Hkv, Hq, bits), int(lens_np.sum()) * Hkv * D,
                           gpu_launches=nsplit)]
            c["results"] = [out]
    elif name == "kattn":
        # resident KIVI cache (random codes, positive scales, N(0,1) zeros) and
        # fp16 window; a step's input is the batch of queries
        cfg = cfgs["kattn_decode_64x8x32_16k"]
        B, Hkv, Hq, S, R, bits, G = (cfg["B"], cfg["Hkv"], cfg["Hq"], cfg["S_cap"], cfg["R"], cfg["bits"],
                                     cfg["group"])
        B = B if batch is None else batch
        lens_np = (synth.cache_lengths(B, cfg["seed"]) // 32 * 32).astype(np.int32)
        rng = np.random.default_rng(cfg["seed"])
        res_np = rng.integers(0, R + 1, B).astype(np.int32)
        g = torch.Generator(device=dev)
        g.manual_seed(cfg["seed"])
        NG = S // G
        ri = lambda shape: torch.randint(-2 ** 31, 2 ** 31 - 1, shape, dtype=torch.int32, device=dev, generator=g)
        cache = {
            "k_packed": ri((B, Hkv, NG, G * bits // 32, D)),
            "k_scale": torch.empty((B, Hkv, NG, D), dtype=torch.float16, device=dev).uniform_(0.05, 0.5, generator=g),
            "k_zero": torch.randn((B, Hkv, NG, D), dtype=torch.float16, device=dev, generator=g),
            "v_packed": ri((B, Hkv, S, D * bits // 32)),
            "v_scale": torch.empty((B, Hkv, S, D // G), dtype=torch.float16, device=dev).uniform_(0.05, 0.5, generator=g),
            "v_zero": torch.randn((B, Hkv, S, D // G), dtype=torch.float16, device=dev, generator=g),
        }
        kr = torch.randn((B, Hkv, R, D), dtype=torch.float16, device=dev, generator=g)
        vr = torch.randn((B, Hkv, R, D), dtype=torch.float16, device=dev, generator=g)
        q_np = rng.standard_normal((B, Hq, D)).astype(np.float16)
        q, lens, res = t(q_np), t(lens_np), t(res_np)
        out = torch.empty((B, Hq, D), dtype=torch.float16, device=dev)
        ws = torch.empty((max(api.vq_kivi_attend_workspace(B, Hq, Hkv, S, R), 16) + 3) // 4,
                         dtype=torch.float32, device=dev)
        nb = kattend_bytes(lens_np, res_np, Hkv, Hq, bits, G)
        ne = int(lens_np.sum() + res_np.sum()) * Hkv * D

        def katt(stream=stream):
            api.vq_kivi_attend(q, cache, bits, G, 1.0 / np.sqrt(D), k_res=kr, v_res=vr, lens=lens, res_lens=res,
                               out=out, workspace=ws, stream=stream)
        ops.append(Op("kivi_attend", "kivi_attend_kernel", katt, nb, ne, gpu_launches=2))
        inputs = [(q_np, q)]
        results.append(out)
        if chunked:
            c = new_chunk(inputs)
            c["ops"] = [Op("kivi_attend", "kivi_attend_kernel", lambda: katt(chunk_stream), nb, ne, gpu_launches=2)]
            c["results"] = [out]
    else:
        raise ValueError(name)
    if chunked and not chunks:
        # no split for this workload: one chunk, the step's own ops on the chunk stream
        c = new_chunk(inputs)
        c["ops"] = ops
        c["results"] = results
        c["own_stream"] = False
    if chunked:
        return ops, inputs, results, chunks
    return ops, inputs, results


# --------------------------------------------------------------------------- clocks


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.06)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        for line in out.splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"), p[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- oracle timing


def oracle_sample_plan(name, target_s=2.0):
    """Bounded samples of each op of the workload for the CPU oracle: per op a
    function of a unit count, the algorithmic bytes per unit and the unit count
    that takes about target_s (found by untimed doubling).  Returns
    ([(op, fn, bytes_per_unit, units)], description)."""
    import oracle
    from kv_cache_quantization_turboquantrvq_gb300 import synth

    plan, desc = [], []
    cfgs = synth.CONFIGS

    def sized(fn, nbytes_per_unit, units0, max_units=1 << 22):
        units = min(units0, max_units)
        while True:
            t0 = time.perf_counter()
            fn(units)
            dt = time.perf_counter() - t0
            if dt >= target_s or units >= max_units:
                return units
            units = min(max_units, int(units * max(2.0, 1.1 * target_s / max(dt, 1e-4))))

    def timed(fn, nbytes_per_unit, units0, max_units=1 << 22, op=None):
        n = sized(fn, nbytes_per_unit, units0, max_units)
        plan.append((op, fn, nbytes_per_unit, n))
        return None, n, None

    def rvq_rates(bits, x_rows, d=D, tag=""):
        c1, b1, c2, b2, _ = oracle.rvq_codebooks(d, bits)
        o = oracle.rvq_encode(x_rows[:1], bits, c1, b1, c2, b2)

        def enc(n):
            oracle.rvq_encode(x_rows[:n], bits, c1, b1, c2, b2)

        def dec(n):
            reps = np.repeat(o["packed1"], n, 0), np.repeat(o["packed2"], n, 0), np.repeat(o["norms"], n)
            oracle.rvq_decode(*reps, d, bits, c1, c2)
        _, n1, _ = timed(enc, rvq_bytes(1, bits, d), 64, len(x_rows), op=tag + "rvq_encode")
        _, n2, _ = timed(dec, rvq_bytes(1, bits, d), 64, op=tag + "rvq_decode")
        return n1, n2

    def kivi_rates(bits, G, x):
        def kq(n):
            oracle.kivi_quant(x[:, :, :G * n], bits, G, 0, True)

        def vq_(n):
            oracle.kivi_quant(x[:, :, :n], bits, G, 0, False)
        _, nk, _ = timed(kq, kivi_bytes(1, G, bits, G, True), 1, x.shape[2] // G, op="kivi_quant_k")
        _, nv, _ = timed(vq_, kivi_bytes(1, 1, bits, G, False), 64, x.shape[2], op="kivi_quant_v")
        ok = oracle.kivi_quant(x[:, :, :G], bits, G, 0, True)
        ov = oracle.kivi_quant(x[:, :, :G], bits, G, 0, False)

        def kd(n):
            oracle.kivi_dequant(np.repeat(ok["packed"], n, 1), np.repeat(ok["scale"], n, 1),
                                np.repeat(ok["zero"], n, 1), 1, G * n, D, bits, G, True)

        def vd(n):
            m = max(1, n // G)
            oracle.kivi_dequant(np.repeat(ov["packed"], m, 1), np.repeat(ov["scale"], m, 1),
                                np.repeat(ov["zero"], m, 1), 1, G * m, D, bits, G, False)
        timed(kd, kivi_bytes(1, G, bits, G, True), 1, op="kivi_dequant_k")
        timed(vd, kivi_bytes(1, 1, bits, G, False), 64, op="kivi_dequant_v")
        return nk, nv

    if name in ("c5", "c1", "c3", "c4", "c4s"):
        bits = {"c5": 2, "c1": 2, "c3": 4, "c4": 2, "c4s": 2}[name]
        cfg = {"c5": cfgs["c5_long_32k"], "c1": cfgs["c1_rvq_b2_8x512"],
               "c3": cfgs["c3_rvq_b4_32L_8k"], "c4": cfgs["c4_decode_flush_64x8x128"],
               "c4s": cfgs["c4_decode_flush_64x8x128"]}[name]
        x = synth.kv_tensor(1, 1, 1 << 16, D, cfg["seed"], *cfg.get("k_outliers", (0, 1.0))).reshape(-1, D)
        n1, n2 = rvq_rates(bits, x)
        desc.append("RVQ b=%d encode %d rows, decode %d rows" % (bits, n1, n2))
    if name == "gen":
        for tag, (dg, bits) in (("D64b2_", (64, 2)), ("D256b4_", (256, 4)), ("D128b3_", (128, 3))):
            x = synth.kv_tensor(1, 1, 1 << 14, dg, 120 + dg + bits, 4, 20.0).reshape(-1, dg)
            n1, n2 = rvq_rates(bits, x, dg, tag)
            desc.append("RVQ D=%d b=%d encode %d rows, decode %d rows" % (dg, bits, n1, n2))
    if name in ("c5", "c2", "c4", "c4s"):
        cfg = {"c5": cfgs["c5_long_32k"], "c2": cfgs["c2_kivi_b2_32x4096"],
               "c4": cfgs["c4_decode_flush_64x8x128"], "c4s": cfgs["c4_decode_flush_64x8x128"]}[name]
        G = cfg["group"]
        x = synth.kv_tensor(1, 1, 1 << 16, D, cfg["seed"], 4, 20.0)
        nk, nv = kivi_rates(2, G, x)
        desc.append("KIVI 2-bit G=%d: %d key groups, %d value rows (and their dequant)" % (G, nk * D, nv))
    if name == "attn":
        cfg = cfgs["attn_decode_64x8x32_16k"]
        bits, gq = cfg["bits"], cfg["Hq"] // cfg["Hkv"]
        c1, _, c2, _, _ = oracle.rvq_codebooks(D, bits)
        smax = 1 << 17
        rng = np.random.default_rng(cfg["seed"])
        W = D * bits // 32
        p1 = rng.integers(0, 2 ** 32, (1, 1, smax, W), dtype=np.uint32)
        p2 = rng.integers(0, 2 ** 32, (1, 1, smax, W), dtype=np.uint32)
        nr = rng.uniform(4.0, 24.0, (1, 1, smax)).astype(np.float32)
        v = rng.standard_normal((1, 1, smax, D)).astype(np.float16)
        q = rng.standard_normal((1, gq, D)).astype(np.float16)

        def att(n):
            oracle.rvq_attend(q, p1[:, :, :n], p2[:, :, :n], nr[:, :, :n], v[:, :, :n], bits, c1, c2,
                              1.0 / np.sqrt(D))
        _, n, _ = timed(att, attend_bytes([1], 1, 0, bits), 256, smax, op="rvq_attend")
        desc.append("RVQ b=%d attention of %d query heads over one kv head of %d keys" % (bits, gq, n))
    if name == "qjl":
        cfg = cfgs["qjl_long_32k_m128"]
        m = cfg["m"]
        x = synth.kv_tensor(1, 1, 1 << 15, D, cfg["seed"], 4, 40.0).reshape(-1, D)
        sk = np.random.default_rng(cfg["seed"]).standard_normal((m, D)).astype(np.float16)

        def qe(n):
            oracle.qjl_encode(x[:n], sk)
        _, n, _ = timed(qe, qjl_bytes(1, m), 64, len(x), op="qjl_encode")
        desc.append("QJL encode (m=%d) of %d key rows" % (m, n))
    if name == "kattn":
        cfg = cfgs["kattn_decode_64x8x32_16k"]
        bits, G, gq, R = cfg["bits"], cfg["group"], cfg["Hq"] // cfg["Hkv"], cfg["R"]
        smax = 1 << 15
        rng = np.random.default_rng(cfg["seed"])
        kk = rng.standard_normal((1, 1, smax + R, D)).astype(np.float16)
        vv = rng.standard_normal((1, 1, smax + R, D)).astype(np.float16)
        kq = oracle.kivi_quant(kk, bits, G, R, True)
        vq_ = oracle.kivi_quant(vv, bits, G, R, False)
        qq = rng.standard_normal((1, gq, D)).astype(np.float16)
        NG = smax // G

        def katt(n):
            ng = max(1, n // G)
            oracle.kivi_attend(qq, kq["packed"].reshape(1, 1, NG, -1, D)[:, :, :ng],
                               kq["scale"].reshape(1, 1, NG, D)[:, :, :ng], kq["zero"].reshape(1, 1, NG, D)[:, :, :ng],
                               vq_["packed"].reshape(1, 1, smax, -1)[:, :, :ng * G],
                               vq_["scale"].reshape(1, 1, smax, -1)[:, :, :ng * G],
                               vq_["zero"].reshape(1, 1, smax, -1)[:, :, :ng * G], bits, G, 1.0 / np.sqrt(D))
        per_tok = kattend_bytes([1], [0], 1, 0, bits, G)
        _, n, _ = timed(katt, per_tok, 256, smax, op="kivi_attend")
        desc.append("KIVI %d-bit G=%d attention of %d query heads over one kv head of %d tokens" % (bits, G, gq, n))
    return plan, "; ".join(desc)


def time_plan(plan):
    """Run each op of a sample plan once; returns ({op: bytes/s}, seconds)."""
    rates, total = {}, 0.0
    for op, fn, nbytes_per_unit, n in plan:
        t0 = time.perf_counter()
        fn(n)
        dt = time.perf_counter() - t0
        rates[op] = n * nbytes_per_unit / dt
        total += dt
    return rates, total


def oracle_sample_rates(name, target_s=2.0):
    """The oracle's rate per op on samples of about target_s each."""
    plan, desc = oracle_sample_plan(name, target_s)
    rates, total = time_plan(plan)
    return rates, desc + " (%.1f s of CPU for %d ops)" % (total, len(plan))


def step_rate_from_ops(ops, rates):
    """Whole-step bytes/s if each op ran at its sampled rate."""
    t = 0.0
    for o in ops:
        base = o.name.split("_", 1)[1] if o.name.startswith("L") else o.name
        t += o.nbytes / rates[base if base in rates else o.name]
    return sum(o.nbytes for o in ops) / t


# --------------------------------------------------------------------------- traffic record


def recorded_traffic(kernel):
    """dram bytes per unit from the committed ncu summary, if the kernel source
    is unchanged since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(kernel)
    except Exception:
        return None
    if not rec:
        return None
    # the kernel's source files (one name or a list), hashed in order
    names = rec["source"] if isinstance(rec["source"], list) else [rec["source"]]
    hsh = hashlib.sha256()
    try:
        for n in names:
            hsh.update(open(os.path.join(ROOT, "kv_cache_quantization_turboquantrvq_gb300", "csrc", n), "rb").read())
    except Exception:
        return None
    h = hsh.hexdigest()[:16]
    if h != rec.get("source_sha256_16"):
        return None
    return rec


# --------------------------------------------------------------------------- main


HEAD_START_CYCLES = 40_000_000  # ~20 ms at the GB300's 2 GHz SM clock


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=("c5", "c3", "c2", "c1", "c4", "c4s", "attn", "kattn", "qjl", "gen"),
                    default="c5")
    ap.add_argument("--graph", action="store_true",
                    help="also capture the step in a CUDA graph and time its replays "
                         "(launch-bound workloads: c4, c1); `value` is then the graph's")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="c5 and attn only: batch size B (default 4 and 64; fewer for small profiling runs)")
    ap.add_argument("--layers", type=int, default=None,
                    help="c3 only: number of layers (default 32; fewer for small profiling runs)")
    ap.add_argument("--streams", type=int, default=1,
                    help="c3 only: the layers round-robin over this many streams (a layer's decode "
                         "waits for its own encode only), so that one launch's tail overlaps the "
                         "next one's start; per-kernel times then overlap")
    args = ap.parse_args()
    if args.streams < 1 or (args.streams > 1 and args.workload != "c3"):
        raise SystemExit("--streams N > 1 applies to --workload c3 only")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args, world)

    import torch
    import torch.distributed as dist
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    from kv_cache_quantization_turboquantrvq_gb300 import api, build
    build.build()
    api.lib()  # fails loudly if the CUDA library is missing

    if args.graph:
        # a graph is captured on a side stream: run the whole bench there
        torch.cuda.set_stream(torch.cuda.Stream())
    s_run = torch.cuda.Stream()  # e2e kernel stream
    stream = torch.cuda.current_stream()
    lanes = [stream] + [torch.cuda.Stream() for _ in range(args.streams - 1)] if args.streams > 1 else None
    built = build_workload(args.workload, dev, rank, layers=args.layers, batch=args.batch,
                           chunked=not args.no_e2e, chunk_stream=s_run, lanes=lanes)
    ops, inputs, results = built[:3]
    chunks = built[3] if len(built) > 3 else []
    K, W = args.steps, max(args.warmup, 3)
    # per-op events: one stream, op i runs from event i to event i + 1; several
    # streams, op i from event 2i to event 2i + 1 on its own stream
    n_ev = len(ops) + 1 if lanes is None else 2 * len(ops)

    def step(evs=None):
        if lanes is None:
            for i, o in enumerate(ops):
                if evs is not None:
                    evs[i].record(stream)
                o.run()
            if evs is not None:
                evs[len(ops)].record(stream)
            return
        fork = torch.cuda.Event()
        fork.record(stream)
        for s in lanes[1:]:
            s.wait_event(fork)
        for i, o in enumerate(ops):
            if evs is not None:
                evs[2 * i].record(o.stream)
            o.run()
            if evs is not None:
                evs[2 * i + 1].record(o.stream)
        for s in lanes[1:]:
            join = torch.cuda.Event()
            join.record(s)
            stream.wait_event(join)

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    assert api.vq_device_error() == 0
    if world > 1:
        dist.barrier()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank)
    time.sleep(0.1)
    torch.cuda.synchronize()
    # a GPU-side head start (a spin of ~20 ms on the stream, before the timed
    # region): the host queues launches meanwhile and stays ahead, as an
    # asynchronous caller does, so the events time the kernels, not the
    # host's launch latency (launch-bound workloads: see also --graph)
    torch.cuda._sleep(HEAD_START_CYCLES)
    t_start.record(stream)
    for k in range(K):
        step(evs[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    step_bytes = sum(o.nbytes for o in ops)
    step_elems = sum(o.nelem for o in ops)
    value = world * step_bytes * K / (elapsed_ms * 1e-3) / 1e9

    # the same step as one CUDA graph (no host work or launch gaps between kernels)
    graph = None
    if args.graph:
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            step()
        for _ in range(W):
            g.replay()
        torch.cuda.synchronize()
        assert api.vq_device_error() == 0
        if world > 1:
            dist.barrier()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(K):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        gms = max_over_ranks(g0.elapsed_time(g1), world, dev)
        graph = {"ms_per_step": round(gms / K, 5),
                 "eager_value": round(value, 2), "eager_ms_per_step": round(elapsed_ms / K, 5)}
        elapsed_ms = gms
        value = world * step_bytes * K / (elapsed_ms * 1e-3) / 1e9
    gelem = world * step_elems * K / (elapsed_ms * 1e-3) / 1e9

    # per-op average durations (events on the launching stream)
    per_ms, per_step = {}, {}
    for i, o in enumerate(ops):
        a, b = (i, i + 1) if lanes is None else (2 * i, 2 * i + 1)
        per_step[o.name] = [evs[k][a].elapsed_time(evs[k][b]) for k in range(K)]
        per_ms[o.name] = statistics.mean(per_step[o.name])
    by_kernel = {}
    for o in ops:
        d = by_kernel.setdefault(o.kernel, {"ms": 0.0, "bytes": 0, "launches": 0, "steps": [0.0] * K})
        d["ms"] += per_ms[o.name]
        d["bytes"] += o.nbytes
        d["launches"] += o.launches
        d["steps"] = [a + b for a, b in zip(d["steps"], per_step[o.name])]
    peak, peak_src = measured_peak()
    dom = max(by_kernel, key=lambda n: by_kernel[n]["ms"])
    dk = by_kernel[dom]
    avg_launch_ms = dk["ms"] / dk["launches"]
    ach = dk["bytes"] / dk["launches"] / (avg_launch_ms * 1e-3) / 1e9
    rec = recorded_traffic(dom)
    traffic = None
    if rec is not None:
        traffic = rec["dram_bytes_per_unit"] * dk["bytes"] / dk["launches"] / rec["alg_bytes_per_unit"]

    # end to end through the public API with host buffers: the step's chunks
    # (C5: one per batch, C3: one per layer) are pipelined over three streams,
    # host->device copy of chunk c+1 and device->host copy of chunk c-1
    # overlapping the kernels of chunk c
    e2e = None
    if not args.no_e2e:
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        for c in chunks:
            c["pin_in"] = [torch.from_numpy(np.ascontiguousarray(h)).pin_memory() for h, _ in c["inputs"]]
            c["pin_out"] = [torch.empty(r.shape, dtype=r.dtype, pin_memory=True) for r in c["results"]]
            c["ev_in"], c["ev_run"], c["ev_out"] = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
        h2d = sum(p.numel() * p.element_size() for c in chunks for p in c["pin_in"])
        d2h = sum(p.numel() * p.element_size() for c in chunks for p in c["pin_out"])
        assert sum(o.nbytes for c in chunks for o in c["ops"]) == step_bytes

        def e2e_step():
            for c in chunks:
                s_in.wait_event(c["ev_run"])  # the inputs' previous readers are done
                with torch.cuda.stream(s_in):
                    for p, (_, dv) in zip(c["pin_in"], c["inputs"]):
                        dv.copy_(p, non_blocking=True)
                c["ev_in"].record(s_in)
                s_run.wait_event(c["ev_in"])
                # the outputs' previous copy to the host is done (a no-op the first time)
                s_run.wait_event(c["ev_out"])
                if c.get("own_stream", True):
                    for o in c["ops"]:
                        o.run()
                else:  # the step's own ops run on the current stream: order it after the copies
                    stream.wait_event(c["ev_in"])
                    stream.wait_event(c["ev_out"])
                    for o in c["ops"]:
                        o.run()
                    s_run.wait_stream(stream)
                c["ev_run"].record(s_run)
                s_out.wait_event(c["ev_run"])
                with torch.cuda.stream(s_out):
                    for p, r in zip(c["pin_out"], c["results"]):
                        p.copy_(r, non_blocking=True)
                c["ev_out"].record(s_out)

        Ke = max(3, min(K, 20))
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for _ in range(Ke):
            e2e_step()
        s_out.wait_event(chunks[-1]["ev_run"])
        e1.record(s_out)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), world, dev)
        e2e = {"value": round(world * step_bytes * Ke / (ems * 1e-3) / 1e9, 2), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(ems / Ke, 4), "chunks_per_step": len(chunks),
               "overlap": "host copies of neighbouring chunks overlap the kernels (3 streams)"}
    assert api.vq_device_error() == 0

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rates, desc = oracle_sample_rates(args.workload)
        # (the oracle runs the step's parts one by one: the same bytes)
        cpu = {"value": round(step_rate_from_ops(reference_ops(args.workload), rates) / 1e9, 6), "unit": UNIT, "cores": 1,
               "host_cores": os.cpu_count(), "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": round(elapsed_ms / K, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded N(0,1) fp16 with per-head outlier channels)",
            "config": {"workload": args.workload + ": " + describe(args.workload),
                       "parallelism": "replicas (independent shards per GPU)" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (129 MB); no flush" if args.workload in ("c5", "c3", "c2", "attn", "kattn", "qjl", "gen")
                             else "inputs smaller than L2 (no flush: steps may reuse L2)",
                       "bytes_per_step": step_bytes, "elements_per_step": step_elems,
                       "timing": ("CUDA graph replays of the step" if args.graph else
                                  "CUDA events on the stream; the host queues ahead of the GPU "
                                  "(a 20 ms GPU spin before the timed region)"),
                       **({"streams": "the layers round-robin over %d streams; per-kernel times overlap "
                                      "(each measured on its own stream)" % args.streams} if lanes else {})},
            "pct_of_peak": round(100 * value / world / peak, 2),
            "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
            "gelem_per_s": round(gelem, 3),
            "per_kernel": {n: {"ms_per_launch": round(d["ms"] / d["launches"], 5),
                               "ms_per_launch_median": round(statistics.median(d["steps"]) / d["launches"], 5),
                               "ms_per_launch_min": round(min(d["steps"]) / d["launches"], 5),
                               "ms_per_launch_max": round(max(d["steps"]) / d["launches"], 5),
                               "GB_s": round(d["bytes"] / d["launches"] / (d["ms"] / d["launches"] * 1e-3) / 1e9, 1),
                               "frac_of_peak": round(d["bytes"] / d["launches"] / (d["ms"] / d["launches"] * 1e-3) / 1e9 / peak, 4),
                               "launches_per_step": d["launches"]} for n, d in by_kernel.items()},
            "roofline": {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": peak,
                         "peak_source": peak_src, "unit": "GB/s", "frac": round(ach / peak, 4),
                         "traffic": None if traffic is None else int(traffic),
                         "alg_bytes_per_launch": int(dk["bytes"] / dk["launches"])},
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clk, "graph": graph,
            "gpu_launches": sum(o.gpu_launches for o in ops) * K,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_reference(args, world):
    """The CPU oracle timed on bounded samples of the workload, one per step."""
    import oracle
    oracle.build()
    # op list without a GPU: sizes only
    ops = reference_ops(args.workload)
    W, K = max(args.warmup, 0), args.steps
    vals, t_total = [], 0.0
    # the same fixed samples every step, sized once (untimed) so that the
    # W + K steps take about two minutes in all
    per_step_target = min(2.0, 120.0 / max(W + K, 1))
    plan, desc = oracle_sample_plan(args.workload, target_s=max(per_step_target / 6, 0.05))
    for i in range(W + K):
        rates, dt = time_plan(plan)
        if i >= W:
            vals.append(step_rate_from_ops(ops, rates) / 1e9)
            t_total += dt
    value = statistics.median(vals)
    step_bytes = sum(o.nbytes for o in ops)
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(1e3 * step_bytes / (value * 1e9), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) fp16 with per-head outlier channels)",
        "config": {"workload": args.workload + ": " + describe(args.workload),
                   "bytes_per_step": step_bytes},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1, "host_cores": os.cpu_count(),
                         "kind": "oracle", "sample": desc + "; wall %.1f s over %d steps" % (t_total, K)},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def reference_ops(name):
    """Byte/element counts of the workload's ops (no device work)."""
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    cfgs = synth.CONFIGS
    ops = []
    noop = lambda: None
    if name == "c5":
        c = cfgs["c5_long_32k"]
        rows = c["B"] * c["H"] * c["S"]
        bh, s_q = c["B"] * c["H"], c["S"] - c["residual"]
        for n in ("rvq_encode", "rvq_decode"):
            ops.append(Op(n, n, noop, rvq_bytes(rows, 2), rows * D))
        for n, pc in (("kivi_quant_k", True), ("kivi_quant_v", False), ("kivi_dequant_k", True),
                      ("kivi_dequant_v", False)):
            ops.append(Op(n, n, noop, kivi_bytes(bh, s_q, 2, c["group"], pc), bh * s_q * D))
    elif name in ("c3", "c1"):
        c = cfgs["c3_rvq_b4_32L_8k"] if name == "c3" else cfgs["c1_rvq_b2_8x512"]
        rows = c["B"] * c["H"] * c["S"] * c.get("layers", 1)
        for n in ("rvq_encode", "rvq_decode"):
            ops.append(Op(n, n, noop, rvq_bytes(rows, c["bits"]), rows * D))
    elif name == "c2":
        c = cfgs["c2_kivi_b2_32x4096"]
        bh, s_q = c["B"] * c["H"], c["S"] - c["residual"]
        for n, pc in (("kivi_quant_k", True), ("kivi_quant_v", False), ("kivi_dequant_k", True),
                      ("kivi_dequant_v", False)):
            ops.append(Op(n, n, noop, kivi_bytes(bh, s_q, 2, c["group"], pc), bh * s_q * D))
    elif name in ("c4", "c4s"):
        c = cfgs["c4_decode_flush_64x8x128"]
        rows = c["B"] * c["H"] * c["S"]
        ops.append(Op("rvq_encode", "rvq_encode", noop, rvq_bytes(rows, 2), rows * D))
        for n, pc in (("kivi_quant_k", True), ("kivi_quant_v", False)):
            ops.append(Op(n, n, noop, kivi_bytes(c["B"] * c["H"], c["S"], 2, c["group"], pc), rows * D))
    elif name == "kattn":
        c = cfgs["kattn_decode_64x8x32_16k"]
        lens = (synth.cache_lengths(c["B"], c["seed"]) // 32 * 32).astype(np.int32)
        res = np.random.default_rng(c["seed"]).integers(0, c["R"] + 1, c["B"]).astype(np.int32)
        ops.append(Op("kivi_attend", "kivi_attend", noop,
                      kattend_bytes(lens, res, c["Hkv"], c["Hq"], c["bits"], c["group"]),
                      int(lens.sum() + res.sum()) * c["Hkv"] * D))
    elif name == "attn":
        c = cfgs["attn_decode_64x8x32_16k"]
        lens = synth.cache_lengths(c["B"], c["seed"])
        ops.append(Op("rvq_attend", "rvq_attend", noop, attend_bytes(lens, c["Hkv"], c["Hq"], c["bits"]),
                      int(lens.sum()) * c["Hkv"] * D))
    elif name == "qjl":
        c = cfgs["qjl_long_32k_m128"]
        rows = c["B"] * c["H"] * c["S"]
        ops.append(Op("qjl_encode", "qjl_encode", noop, qjl_bytes(rows, c["m"]), rows * D))
    elif name == "gen":
        for tag, (Bg, dg, bits) in (("D64b2_", (4, 64, 2)), ("D256b4_", (1, 256, 4)), ("D128b3_", (2, 128, 3))):
            rows = Bg * 32 * 32768
            for n in ("rvq_encode", "rvq_decode"):
                ops.append(Op(tag + n, tag + n, noop, rvq_bytes(rows, bits, dg), rows * dg))
    return ops


if __name__ == "__main__":
    sys.exit(main())
