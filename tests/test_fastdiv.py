"""Host test of the multiply-shift division the kernels use for per-block
index arithmetic (FastDiv in csrc/launch.h): for numerators below 2^31 the
device computes umulhi(n, m) >> s, which must equal n // d exactly."""
import os
import random
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "kv_cache_quantization_turboquantrvq_gb300", "csrc")


@pytest.fixture(scope="module")
def constants(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path_factory.mktemp("fastdiv") / "fastdiv_harness")
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                           "-I", "/usr/local/cuda/include", os.path.join(ROOT, "tests", "fastdiv_harness.cpp"),
                           "-o", exe])
    rng = random.Random(5)
    ds = (list(range(1, 3000)) + [rng.randrange(1, 2 ** 31) for _ in range(3000)] +
          [2 ** k for k in range(31)] + [2 ** k - 1 for k in range(2, 32)] + [2 ** k + 1 for k in range(1, 31)] +
          [32640, 32768, 510, 2040, 8192, 16512, 4096])
    out = {}
    for i in range(0, len(ds), 1000):
        r = subprocess.run([exe] + [str(d) for d in ds[i:i + 1000]], capture_output=True, text=True, check=True)
        for line in r.stdout.split("\n"):
            if line.strip():
                d, m, s, one = map(int, line.split())
                out[d] = (m, s, one)
    return out


def _div(c, n):
    m, s, one = c
    return n if one else ((n * m) >> 32) >> s


def test_quotients_exact(constants):
    rng = random.Random(6)
    for d, c in constants.items():
        assert c[0] < 2 ** 32
        ns = [0, 1, d - 1, d, d + 1, 2 ** 31 - 1, 2 ** 31 - 2] + [rng.randrange(0, 2 ** 31) for _ in range(20)]
        k = (2 ** 31 - 1) // d
        ns += [d * k, d * k - 1] + [d * j + r for j in (2, 1000) for r in (-1, 0, 1)]
        for n in ns:
            if 0 <= n < 2 ** 31:
                assert _div(c, n) == n // d, (d, n)
