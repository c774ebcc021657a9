"""Host tests of the shuffle-table boundary count used by the RVQ encoder
(csrc/grid.cpp): a table must exist for the library's codebooks and must
reproduce the plain boundary count exactly (no GPU needed)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "kv_cache_quantization_turboquantrvq_gb300", "csrc")
GUARD = "2.5e-7"  # the library's guard band


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path_factory.mktemp("grid") / "grid_harness")
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                           "-I", "/usr/local/cuda/include", os.path.join(ROOT, "tests", "grid_harness.cpp"),
                           os.path.join(CSRC, "grid.cpp"), "-o", exe])
    return exe


def _run(exe, b):
    r = subprocess.run([exe, GUARD] + ["%.9g" % float(v) for v in np.asarray(b, np.float32)],
                       capture_output=True, text=True)
    return r.returncode, r.stdout.strip()


@pytest.mark.parametrize("bits", [1, 2, 4])
def test_tables_for_library_codebooks(harness, bits):
    from kv_cache_quantization_turboquantrvq_gb300 import api, build
    build.build()
    c1, b1, c2, b2 = api.vq_rvq_codebook(128, bits)
    for b in (b1, b2):
        rc, out = _run(harness, b)
        assert rc == 0, out


def test_tables_for_random_codebooks(harness):
    rng = np.random.default_rng(0)
    built = 0
    for trial in range(40):
        nb = int(rng.choice([1, 3, 7, 15]))
        b = np.sort(rng.normal(0, rng.uniform(0.01, 3), nb).astype(np.float32))
        if np.any(np.diff(b) <= 0):
            continue
        rc, out = _run(harness, b)
        if out == "NOTABLE":
            continue  # the encoder then uses its plain-count fallback
        assert rc == 0, out
        built += 1
    assert built >= 30


def test_no_table_when_boundaries_too_close(harness):
    b = np.array([-1.0, 0.0, 1e-7, 1.0], np.float32)  # two boundaries inside one guard band
    rc, out = _run(harness, b)
    assert out == "NOTABLE"
