"""Seeded synthetic KV-cache inputs.

This module only draws random numbers; it holds none of the codecs'
arithmetic.  Both the CUDA path and the CPU oracle receive its arrays, so
their inputs are identical bit for bit.

Recipe (numpy PCG64 ``default_rng(seed)``, ``standard_normal`` in float32,
cast to float16):

* base entries N(0, 1);
* optional per-(head, channel) scales drawn log-uniform in [lo, hi];
* optional outlier channels: per head, ``n_outliers`` distinct channels drawn
  without replacement, multiplied by ``outlier_scale`` for every token (the
  KIVI page's point that a few key channels carry much larger magnitudes);
* generation runs one (batch, head) slice at a time, so the stream of random
  numbers, and therefore the tensor, does not depend on chunking.

The named workloads below are the five configurations the library is
measured and checked on (shapes [B, H, S, D], fp16).
"""
from __future__ import annotations

import numpy as np

D = 128


def kv_tensor(B: int, H: int, S: int, D: int, seed: int, n_outliers: int = 0,
              outlier_scale: float = 1.0, channel_scale_range=None,
              heads=None) -> np.ndarray:
    """One fp16 tensor [B, H, S, D] (or [B, len(heads), S, D] when `heads`
    selects a subset; the subset equals the same slice of the full tensor)."""
    rng = np.random.default_rng(seed)
    # Per-head side information is drawn first, for all heads, so that it
    # does not depend on which heads are materialised.
    outl = [rng.choice(D, n_outliers, replace=False) if n_outliers else None
            for _ in range(H)]
    if channel_scale_range is not None:
        lo, hi = channel_scale_range
        cscale = np.exp(rng.uniform(np.log(lo), np.log(hi), (H, D))).astype(np.float32)
    else:
        cscale = None
    heads = list(range(H)) if heads is None else list(heads)
    out = np.empty((B, len(heads), S, D), np.float16)
    for b in range(B):
        for hi_, h in enumerate(range(H)):
            sub = np.random.default_rng([seed, b, h])
            if h not in heads:
                continue
            x = sub.standard_normal((S, D), dtype=np.float32)
            if cscale is not None:
                x *= cscale[h][None, :]
            if outl[h] is not None:
                x[:, outl[h]] *= np.float32(outlier_scale)
            out[b, heads.index(h)] = x.astype(np.float16)
    return out


def cache_lengths(n: int, seed: int, lo: int = 1024, hi: int = 16384, multiple: int = 128):
    """Per-sequence cache lengths uniform in [lo, hi], rounded down to a multiple."""
    rng = np.random.default_rng(seed)
    L = rng.integers(lo, hi + 1, n)
    return (L // multiple * multiple).astype(np.int32)


# Named workloads ------------------------------------------------------------

CONFIGS = {
    # RVQ b=2 on one key tensor, per-channel scales log-uniform in [0.5, 2].
    "c1_rvq_b2_8x512": dict(kind="rvq", B=1, H=8, S=512, bits=2, seed=101,
                            channel_scale_range=(0.5, 2.0)),
    # KIVI 2-bit flush on K and V, 4 key outlier channels per head at 20x,
    # G = 32, residual 128.
    "c2_kivi_b2_32x4096": dict(kind="kivi", B=1, H=32, S=4096, bits=2, group=32,
                               residual=128, seed=102, k_outliers=(4, 20.0)),
    # RVQ b=4 over 32 layers of [1, 32, 8192, 128] keys with 4x20 outliers,
    # then unpack+dequant.
    "c3_rvq_b4_32L_8k": dict(kind="rvq", B=1, H=32, S=8192, bits=4, layers=32, seed=1030,
                             k_outliers=(4, 20.0)),
    # Decode-time flush: 64 sequences x 8 heads x 128 new tokens into caches of
    # random lengths; RVQ b in {1,2,4}, KIVI b in {2,4}, G = 32, residual 0.
    "c4_decode_flush_64x8x128": dict(kind="decode", B=64, H=8, S=128, seed=104,
                                     k_outliers=(4, 20.0), s_dst=16384 + 128,
                                     rvq_bits=(1, 2, 4), kivi_bits=(2, 4), group=32),
    # Long context: K, V [4, 32, 32768, 128], outliers 4 per head at 40x in K
    # and V; RVQ b=2 on K, KIVI 2-bit G=64 residual 128 on K and V, then
    # unpack+dequant of both.
    "c5_long_32k": dict(kind="long", B=4, H=32, S=32768, rvq_bits=2, kivi_bits=2, group=64,
                        residual=128, seed=105, k_outliers=(4, 40.0), v_outliers=(4, 40.0)),
    # Decode-time attention over the flushed cache: 64 sequences, 8 kv heads
    # and 32 query heads (GQA 4), RVQ b=2 keys and fp16 values in caches of
    # capacity 16384 holding random lengths in [1k, 16k].
    "attn_decode_64x8x32_16k": dict(kind="attend", B=64, Hkv=8, Hq=32, S_cap=16384, bits=2, seed=110),
    # The same decode batch over a KIVI 2-bit (G = 32) cache with dequantization
    # inside the attention, plus a 128-token fp16 residual window holding
    # random fill levels in [0, 128].
    "kattn_decode_64x8x32_16k": dict(kind="kattend", B=64, Hkv=8, Hq=32, S_cap=16384, R=128, bits=2,
                                     group=32, seed=111),
    # QJL encode of the long-context keys: m = 128 sketch rows (the 16x
    # compression the pages quote for QJL: 128 fp16 values -> 128 bits), a
    # seeded N(0, 1) fp16 sketch.
    "qjl_long_32k_m128": dict(kind="qjl", B=4, H=32, S=32768, m=128, seed=112, k_outliers=(4, 40.0)),
}


def keys_for(cfg: dict, layer: int = 0, heads=None, B=None) -> np.ndarray:
    Bv = cfg["B"] if B is None else B
    n, sc = cfg.get("k_outliers", (0, 1.0))
    return kv_tensor(Bv, cfg["H"], cfg["S"], D, cfg["seed"] + layer, n, sc,
                     cfg.get("channel_scale_range"), heads=heads)


def values_for(cfg: dict, heads=None, B=None) -> np.ndarray:
    Bv = cfg["B"] if B is None else B
    n, sc = cfg.get("v_outliers", (0, 1.0))
    return kv_tensor(Bv, cfg["H"], cfg["S"], D, cfg["seed"] + 7919, n, sc, heads=heads)
