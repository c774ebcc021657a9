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


def _pair_args(c1, b1, c2, b2):
    return ["pair", GUARD] + ["%.9g" % float(x) for a in (c1, b1, c2, b2) for x in np.asarray(a, np.float32)]


def test_pair_table_for_library_4bit_codebook(harness):
    """The one-lookup two-stage table of the 4-bit encoder: every looked-up
    pair outside the guard band equals the exact pair, and no step of the pair
    function is within the guard band of a value in another cell."""
    from kv_cache_quantization_turboquantrvq_gb300 import api, build
    build.build()
    c1, b1, c2, b2 = api.vq_rvq_codebook(128, 4)
    r = subprocess.run([harness] + _pair_args(c1, b1, c2, b2), capture_output=True, text=True)
    assert r.returncode == 0, r.stdout
    assert r.stdout.startswith("OK") and "steps 163" in r.stdout


def test_pair_table_for_scaled_and_perturbed_codebooks(harness):
    """Other 16-level books (the library's at other dimensions, and randomly
    perturbed ones): a table is either built and exact, or refused.  The
    library's books at D = 64 and 256 must get one; perturbed books whose
    steps crowd closer than a 512-cell grid can separate are refused (the
    encoder then uses the two-table quantizer)."""
    from kv_cache_quantization_turboquantrvq_gb300 import api, build
    build.build()
    rng = np.random.default_rng(5)
    built = 0
    books = [api.vq_rvq_codebook(d, 4) for d in (64, 256)]
    c1, b1, c2, b2 = api.vq_rvq_codebook(128, 4)
    for _ in range(6):
        j1 = np.sort(c1 * rng.uniform(0.97, 1.03, 16)).astype(np.float32)
        j2 = np.sort(c2 * rng.uniform(0.95, 1.05, 16)).astype(np.float32)
        books.append((j1, (0.5 * (j1[1:] + j1[:-1])).astype(np.float32), j2,
                      (0.5 * (j2[1:] + j2[:-1])).astype(np.float32)))
    for i, book in enumerate(books):
        r = subprocess.run([harness] + _pair_args(*book), capture_output=True, text=True)
        if r.stdout.strip() == "NOTABLE":
            assert i >= 2, "no table for the library's book"
            continue  # the encoder then uses the two-table quantizer
        assert r.returncode == 0, r.stdout
        built += 1
    assert built >= 4
