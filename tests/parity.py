"""Comparison rules for CUDA-vs-oracle parity (test infrastructure).

Codes: bit-exact, except that a code may differ when the oracle flags it as a
tie (its pre-quantization value within 1e-5 of an RVQ boundary, or within
1e-4*scale of a KIVI rounding tie); such mismatches are counted and must stay
below 1e-6 of all codes.
Norms: relative error <= 4e-7.  The fast path sums 128 squares in fp32 with 16
partial sums (depth 8 + 4, error <= 12 u), takes an IEEE square root (0.5 u
after halving the sum's error: <= 6.5 u total) - about 3.9e-7 with
u = 2^-24; rows recomputed exactly are within 0.5 u.
RVQ dequant: |x_gpu - x_oracle| <= 1e-3 * ||x|| (unit-norm rows: 1e-3).
KIVI dequant: bit-exact (both sides round q*scale + zero once).
"""
import numpy as np

TIE_RATE = 1e-6
NORM_RTOL = 4e-7


def unpack_rows(words, bits, D=128):
    """[..., W] uint32 (LSB first) -> [..., D] uint8 codes."""
    w = np.asarray(words).view(np.uint32)
    E = 32 // bits
    sh = (np.arange(D) % E) * bits
    idx = np.arange(D) // E
    return ((w[..., idx] >> sh.astype(np.uint32)) & ((1 << bits) - 1)).astype(np.uint8)


def check_codes(got, ref, tie, what, allow_rate=TIE_RATE, strict=True):
    """Assert the mismatch rule; returns (n_mismatch, n_codes, n_tie)."""
    got = np.asarray(got)
    ref = np.asarray(ref)
    tie = np.asarray(tie).astype(bool)
    mis = got != ref
    n = mis.sum()
    bad = mis & ~tie
    assert not bad.any(), "%s: %d mismatches outside the tie band (first at %s)" % (
        what, bad.sum(), np.argwhere(bad)[0].tolist())
    if strict:
        assert n <= np.floor(allow_rate * got.size), "%s: %d tie mismatches of %d codes" % (
            what, n, got.size)
    return int(n), int(got.size), int(tie.sum())


def check_rvq(gpu_p1, gpu_p2, gpu_norms, ora, bits, strict=True, D=128):
    E = 32 // bits
    W = -(-D // E)
    g1 = unpack_rows(np.asarray(gpu_p1).reshape(-1, W), bits, D)
    g2 = unpack_rows(np.asarray(gpu_p2).reshape(-1, W), bits, D)
    s1 = check_codes(g1, ora["idx1"], ora["tie1"], "stage-1 codes", strict=strict)
    s2 = check_codes(g2, ora["idx2"], ora["tie2"], "stage-2 codes", strict=strict)
    gn = np.asarray(gpu_norms, dtype=np.float32).reshape(-1).astype(np.float64)
    rn = ora["norms"].astype(np.float64)
    rel = np.abs(gn - rn) / np.maximum(rn, 1e-30)
    assert np.all((rel <= NORM_RTOL) | (rn == gn)), "norm rel err %g" % rel.max()
    # words equal wherever no code in them is tie-flagged
    pad = W * E - D
    t1 = np.pad(ora["tie1"].reshape(-1, D), ((0, 0), (0, pad))).reshape(-1, W, E).any(-1)
    t2 = np.pad(ora["tie2"].reshape(-1, D), ((0, 0), (0, pad))).reshape(-1, W, E).any(-1)
    w1 = np.asarray(gpu_p1).view(np.uint32).reshape(-1, W)
    w2 = np.asarray(gpu_p2).view(np.uint32).reshape(-1, W)
    assert np.array_equal(w1[~t1], ora["packed1"][~t1])
    assert np.array_equal(w2[~t2], ora["packed2"][~t2])
    return s1, s2


def unpack_kivi_keys(k_packed, bits, G, S_q):
    """[BH, NG, G*b/32, D] words -> codes [BH, S_q, D]."""
    w = np.asarray(k_packed).view(np.uint32)
    BH, NG, WG, D = w.shape
    E = 32 // bits
    j = np.arange(E, dtype=np.uint32) * bits
    c = (w[:, :, :, None, :] >> j[None, None, None, :, None]) & ((1 << bits) - 1)
    c = c.reshape(BH, NG * G, D)[:, :S_q]
    return c.astype(np.uint8)
