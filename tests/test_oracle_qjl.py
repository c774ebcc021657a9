"""Pins of the oracle's QJL encode (turboquant page, "Kernel 4: QJL Encode -
Simdgroup Sign Packing") against things other than itself: exact rational
arithmetic, a sketch whose sign pattern is known by construction, and
invariants."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle


def _exact(v):
    return Fraction(float(v))  # fp16 -> float64 is exact, and so is Fraction(float)


@pytest.mark.parametrize("seed", [0, 1])
def test_signs_and_packing_match_exact_rationals(seed):
    rng = np.random.default_rng(seed)
    N, d, m = 3, 16, 64
    x = rng.standard_normal((N, d)).astype(np.float16)
    S = rng.standard_normal((m, d)).astype(np.float16)
    r = oracle.qjl_encode(x, S)
    for n in range(N):
        bits = 0
        for j in range(m):
            dot = sum(_exact(S[j, k]) * _exact(x[n, k]) for k in range(d))
            if dot >= 0:
                bits |= 1 << j
        words = [(bits >> (32 * w)) & 0xFFFFFFFF for w in range(m // 32)]
        assert list(r["packed"][n]) == words
        # bytes LSB-first: byte k bit j is sketch row 8k + j (little-endian words)
        by = r["packed"][n].astype("<u4").tobytes()
        for j in range(m):
            assert ((by[j // 8] >> (j % 8)) & 1) == ((bits >> j) & 1)


def test_known_pattern_and_zero_dot():
    """Sketch row j is +e0 or -e0 by bit j of a pattern; x = e0 gives that
    pattern.  Rows orthogonal to x give a zero dot product: bit 1 (>= 0)."""
    d, m = 128, 96
    pattern = 0x9E3779B97F4A7C15F39CC060 & ((1 << m) - 1)
    S = np.zeros((m, d), np.float16)
    for j in range(m):
        S[j, 0] = 1.0 if (pattern >> j) & 1 else -1.0
    S[:, 2] = 1.0           # and every row has +1 at coordinate 2
    x = np.zeros((3, d), np.float16)
    x[0, 0] = 0.5
    x[1, 1] = 3.0           # orthogonal to every row: all products 0, dots exactly 0
    x[2, 0] = 0.25          # +-0.25 from coordinate 0 ...
    x[2, 2] = 0.25          # ... +0.25 from coordinate 2: dot 0.5 or exactly 0 (cancelling)
    r = oracle.qjl_encode(x, S)
    got = sum(int(w) << (32 * i) for i, w in enumerate(r["packed"][0]))
    assert got == pattern
    assert all(int(w) == 0xFFFFFFFF for w in r["packed"][1])
    assert all(int(w) == 0xFFFFFFFF for w in r["packed"][2])  # 0 counts as >= 0
    # ties: only the dots that cancel nonzero terms (rows with a -1 at coordinate 0)
    assert not r["tie"][0].any() and not r["tie"][1].any()
    assert np.array_equal(r["tie"][2], np.array([not (pattern >> j) & 1 for j in range(m)]))


def test_norms_are_fp16_of_the_exact_norm():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((20, 128)) * rng.uniform(0.01, 100, (20, 1))).astype(np.float16)
    x[0] = 0
    x[1, :] = np.float16(2.0 ** -24)     # subnormals
    x[2, :3] = [3, 4, 12]                # 13 exactly
    x[2, 3:] = 0
    r = oracle.qjl_encode(x, np.ones((32, 128), np.float16))
    for n in range(20):
        q = sum(_exact(v) ** 2 for v in x[n])
        want = np.float16(math.sqrt(q))   # float64 sqrt of the exact (representable) sum, then fp16
        if not r["norm_tie"][n]:
            assert r["norms"][n] == want, n
    assert r["norms"][0] == 0 and r["norms"][2] == 13


def test_sign_pattern_is_scale_invariant():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 128)).astype(np.float16)
    S = rng.standard_normal((128, 128)).astype(np.float16)
    a = oracle.qjl_encode(x, S)
    b = oracle.qjl_encode((x.astype(np.float32) * 8).astype(np.float16), S)  # exact power-of-two scaling
    assert np.array_equal(a["packed"], b["packed"])
    assert np.all(b["norms"].astype(np.float64) == 8 * a["norms"].astype(np.float64))
