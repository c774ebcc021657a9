"""The whole-configuration parity harness (tests/full_parity.py) on the CPU:
fed the oracle's own outputs it reports nothing; fed outputs with a planted
fault it reports exactly that fault.  The faults are planted in copies of the
oracle's outputs here, never in a kernel."""
import numpy as np
import pytest

import full_parity as fp

D = 128


@pytest.fixture(scope="module")
def pool():
    with fp.Pool(2) as p:
        yield p


def _rvq_task(oracle_mod, bits, seed, n=300):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    x = synth.kv_tensor(1, 1, n, D, seed, 4, 20.0).reshape(n, D)
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    o = oracle_mod.rvq_encode(x, bits, *cb)
    dec = oracle_mod.rvq_decode(o["packed1"], o["packed2"], o["norms"], D, bits, cb[0], cb[2])
    return dict(x=x, p1=o["packed1"].copy(), p2=o["packed2"].copy(), norms=o["norms"].copy(),
                dec=dec, bits=bits, cb=cb), o


def test_rvq_clean_and_planted(oracle_mod, pool):
    t_clean, _ = _rvq_task(oracle_mod, 2, 5)
    t_code, _ = _rvq_task(oracle_mod, 2, 5)
    t_code["p2"][7, 3] ^= 0x3 << 4          # one stage-2 code changed
    t_norm, _ = _rvq_task(oracle_mod, 2, 5)
    t_norm["norms"][11] *= np.float32(1 + 1e-5)
    t_dec, _ = _rvq_task(oracle_mod, 2, 5)
    t_dec["dec"][2, 9] = np.float16(float(t_dec["dec"][2, 9]) + 0.5)
    st = pool.map(fp.rvq_slice, [t_clean, t_code, t_norm, t_dec])
    fp.assert_rule(st[0], ["s1_", "s2_"], "clean")
    assert st[0]["s1_codes"] == 300 * D and st[0]["dec_values"] == 300 * D
    assert st[1]["s2_mismatch"] == 1 and st[1]["s1_mismatch"] == 0
    with pytest.raises(AssertionError):
        fp.assert_rule(st[1], ["s1_", "s2_"], "planted code")
    assert st[2]["norm_bad"] == 1
    assert st[3]["dec_bad"] == 1
    merged = fp.merge(st)
    assert merged["rows"] == 1200 and merged["s2_mismatch"] == 1


def test_rvq_tie_mismatch_is_forgiven_but_counted(oracle_mod, pool):
    """A code that differs where the oracle flags a tie passes the rule as long
    as the count stays under 1e-6 of codes (here: the rate is raised)."""
    bits = 2
    cb = oracle_mod.rvq_codebooks(D, bits)[:4]
    x = np.zeros((1, D), np.float16)
    x[0, 0] = 1.0  # rotates to the constant 1/sqrt(D)
    c1, b1, c2, b2 = [a.copy() for a in cb]
    b1 = np.array([b1[0], np.float32(1 / np.sqrt(128.0)), b1[2]], np.float32)  # every y on a boundary
    c1[2] = np.float32(0.5 * (float(b1[1]) + float(b1[2])))
    o = oracle_mod.rvq_encode(x, bits, c1, b1, c2, b2)
    assert o["tie1"].all()
    t = dict(x=x, p1=o["packed1"].copy(), p2=o["packed2"].copy(), norms=o["norms"].copy(), dec=None,
             bits=bits, cb=(c1, b1, c2, b2))
    t["p1"][0, 0] ^= 0x3  # code 0 flipped: tie-flagged
    st = pool.map(fp.rvq_slice, [t])[0]
    assert st["s1_mismatch"] == 1 and st["s1_untied_mismatch"] == 0
    fp.assert_rule(st, ["s1_", "s2_"], "tie", rate=1.0)
    with pytest.raises(AssertionError):
        fp.assert_rule(st, ["s1_", "s2_"], "tie")  # 1 of 128 codes is above 1e-6


@pytest.mark.parametrize("per_channel", [True, False])
def test_kivi_clean_and_planted(oracle_mod, pool, per_channel):
    from kv_cache_quantization_turboquantrvq_gb300 import synth
    bits, G, R, S = 2, 32, 10, 150
    x = synth.kv_tensor(1, 1, S, D, 9, 4, 20.0)
    o = oracle_mod.kivi_quant(x, bits, G, R, per_channel)
    S_q = o["S_q"]
    dec = oracle_mod.kivi_dequant(o["packed"], o["scale"], o["zero"], 1, S_q, D, bits, G, per_channel)

    def task():
        return dict(x=x, per_channel=per_channel, bits=bits, G=G, R=R, packed=o["packed"][0].copy(),
                    scale=o["scale"][0].copy(), zero=o["zero"][0].copy(), dec=dec[0].copy())
    clean, bad_scale, bad_dec, bad_code = task(), task(), task(), task()
    bad_scale["scale"].reshape(-1)[5] = np.float16(float(bad_scale["scale"].reshape(-1)[5]) * 2 + 1)
    bad_dec["dec"][3, 4] = np.float16(float(bad_dec["dec"][3, 4]) + 1.0)
    bad_code["packed"].reshape(-1)[0] ^= np.uint32(0x3)
    st = pool.map(fp.kivi_slice, [clean, bad_scale, bad_dec, bad_code])
    fp.assert_rule(st[0], [""], "clean")
    assert st[0]["codes"] == S_q * D and st[0]["dec_values"] == S_q * D
    assert st[1]["scale_bad"] == 1
    assert st[2]["dec_bad"] == 1
    assert st[3]["mismatch"] == 1
    with pytest.raises(AssertionError):
        fp.assert_rule(st[3], [""], "planted")
