"""Whole-configuration parity: every code of a configuration against the oracle.

Test infrastructure.  The GPU outputs of a full-size configuration are cut
into slices (a (batch, head) slice or a few of them); each slice is checked in
a worker process that runs the oracle on the slice's input and returns counts,
so the single-threaded oracle covers every row on all host cores.  The pool is
started with the ``spawn`` method (a process forked after CUDA is initialised
can hang); workers import only numpy, the oracle and ``parity``.

Per slice the checks are the parity rule itself:
* codes: a code may differ from the oracle's only where the oracle flags it
  as a tie (counted per stream; the caller holds the total to 1e-6 of codes);
* RVQ norms within NORM_RTOL; RVQ words equal wherever no code in them is
  tie-flagged; KIVI scale and zero bit-exact, pad slots of a ragged key group 0;
* dequant of the GPU's own storage: KIVI bit-exact against the oracle's
  dequant of that storage, RVQ within 1e-3 * ||x|| of the oracle's binary64
  decode of it.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

from parity import NORM_RTOL, unpack_kivi_keys, unpack_rows

D = 128


def _code_stats(got, ref, tie, prefix):
    tie = np.asarray(tie).astype(bool)
    mis = np.asarray(got) != np.asarray(ref)
    return {prefix + "codes": int(mis.size), prefix + "mismatch": int(mis.sum()),
            prefix + "untied_mismatch": int((mis & ~tie).sum()), prefix + "tie": int(tie.sum())}


def rvq_slice(task):
    """task: dict(x [n, D] fp16, p1, p2 [n, W] uint32, norms [n] fp32,
    dec [n, D] fp16 or None, bits, cb = (c1, b1, c2, b2))."""
    import oracle
    x, bits = task["x"], task["bits"]
    c1, b1, c2, b2 = task["cb"]
    n = x.shape[0]
    E = 32 // bits
    W = -(-D // E)
    p1 = np.asarray(task["p1"]).view(np.uint32).reshape(n, W)
    p2 = np.asarray(task["p2"]).view(np.uint32).reshape(n, W)
    gn = np.asarray(task["norms"], np.float32).reshape(n)
    ora = oracle.rvq_encode(x, bits, c1, b1, c2, b2)
    st = {"rows": n}
    st.update(_code_stats(unpack_rows(p1, bits), ora["idx1"], ora["tie1"], "s1_"))
    st.update(_code_stats(unpack_rows(p2, bits), ora["idx2"], ora["tie2"], "s2_"))
    rn = ora["norms"].astype(np.float64)
    rel = np.abs(gn.astype(np.float64) - rn) / np.maximum(rn, 1e-30)
    st["norm_bad"] = int(np.sum(~((rel <= NORM_RTOL) | (rn == gn.astype(np.float64)))))
    pad = W * E - D
    t1 = np.pad(ora["tie1"], ((0, 0), (0, pad))).reshape(n, W, E).any(-1)
    t2 = np.pad(ora["tie2"], ((0, 0), (0, pad))).reshape(n, W, E).any(-1)
    st["word_bad"] = int(np.sum((p1 != ora["packed1"]) & ~t1) + np.sum((p2 != ora["packed2"]) & ~t2))
    if task.get("dec") is not None:
        got = np.asarray(task["dec"], np.float16).reshape(n, D)
        ref16, ref64 = oracle.rvq_decode(p1, p2, gn, D, bits, c1, c2, want_f64=True)
        err = np.abs(got.astype(np.float64) - ref64)
        nrm = gn.astype(np.float64)[:, None]
        st["dec_values"] = int(got.size)
        st["dec_bad"] = int(np.sum(err > 1e-3 * nrm))
        st["dec_max_rel"] = float(np.max(err / np.maximum(nrm, 1e-30))) if n else 0.0
        st["dec_same_fp16"] = int(np.sum(got.view(np.uint16) == ref16.view(np.uint16)))
    return st


def kivi_slice(task):
    """task: dict(x [1, H, S, D] fp16 (tokens [0, S - R) are quantized),
    per_channel, bits, G, R, packed, scale, zero (the GPU storage of these H
    heads, trimmed to their S_q tokens or NG groups), dec [H, S_q, D] fp16 or
    None)."""
    import oracle
    x, bits, G, R, pc = task["x"], task["bits"], task["G"], task["R"], task["per_channel"]
    BH = x.shape[0] * x.shape[1]
    ora = oracle.kivi_quant(x, bits, G, R, pc)
    S_q, NG = ora["S_q"], ora["NG"]
    packed = np.asarray(task["packed"]).view(np.uint32)
    scale = np.asarray(task["scale"], np.float16)
    zero = np.asarray(task["zero"], np.float16)
    if pc:
        packed = packed.reshape(BH, NG, G * bits // 32, D)
        codes = unpack_kivi_keys(packed, bits, G, S_q)
        full = unpack_kivi_keys(packed, bits, G, NG * G)
        st = {"pad_bad": int(np.sum(full[:, S_q:] != 0))}
        scale = scale.reshape(BH, NG, D)
        zero = zero.reshape(BH, NG, D)
    else:
        packed = packed.reshape(BH, S_q, D * bits // 32)
        codes = unpack_rows(packed, bits)
        st = {"pad_bad": 0}
        scale = scale.reshape(BH, S_q, D // G)
        zero = zero.reshape(BH, S_q, D // G)
    st.update(_code_stats(codes, ora["codes"], ora["tie"], ""))
    st["scale_bad"] = int(np.sum(scale.view(np.uint16) != ora["scale"].view(np.uint16)))
    st["zero_bad"] = int(np.sum(zero.view(np.uint16) != ora["zero"].view(np.uint16)))
    if task.get("dec") is not None:
        got = np.asarray(task["dec"], np.float16).reshape(BH, S_q, D)
        ref = oracle.kivi_dequant(packed, scale, zero, BH, S_q, D, bits, G, pc)
        st["dec_values"] = int(got.size)
        st["dec_bad"] = int(np.sum(got.view(np.uint16) != ref.view(np.uint16)))
    return st


def merge(stats):
    out = {}
    for s in stats:
        for k, v in s.items():
            if k.endswith("_max_rel"):
                out[k] = max(out.get(k, 0.0), v)
            else:
                out[k] = out.get(k, 0) + v
    return out


class Pool:
    """A spawn-method process pool over the host's cores."""

    def __init__(self, procs=None):
        self.procs = procs or max(1, min(os.cpu_count() or 1, 32))
        self._pool = mp.get_context("spawn").Pool(self.procs)

    def map(self, fn, tasks):
        return self._pool.map(fn, tasks, chunksize=1)

    def submit(self, fn, tasks):
        return self._pool.map_async(fn, tasks, chunksize=1)

    def close(self):
        self._pool.close()
        self._pool.join()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        if exc[0] is not None:
            self._pool.terminate()
        self.close()


def assert_rule(st, streams, what, rate=1e-6):
    """The parity rule over a whole configuration; returns a one-line report."""
    parts = []
    for p in streams:
        n, mis, untied, tie = st[p + "codes"], st[p + "mismatch"], st[p + "untied_mismatch"], st[p + "tie"]
        assert untied == 0, "%s %s: %d mismatches outside the tie band" % (what, p or "codes", untied)
        assert mis <= np.floor(rate * n), "%s %s: %d tie mismatches of %d codes" % (what, p or "codes", mis, n)
        parts.append("%s%d codes, %d mismatches, %d tie-flagged" % (p, n, mis, tie))
    for k in ("norm_bad", "word_bad", "pad_bad", "scale_bad", "zero_bad", "dec_bad"):
        if k in st:
            assert st[k] == 0, "%s: %s = %d" % (what, k, st[k])
    if "dec_values" in st:
        parts.append("dequant %d values checked" % st["dec_values"])
    return "%s: %s" % (what, "; ".join(parts))
