"""The seeded input generators: shapes, determinism, routing contract, skew."""
import json
import os

import numpy as np
import pytest

import moe_workloads as mw

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.mark.parametrize("name", sorted(mw.WORKLOADS))
def test_ids_shape_range_distinct_deterministic(name):
    w = mw.WORKLOADS[name]
    ids = mw.gen_ids(w)
    assert ids.shape == (w.T, w.k) and ids.dtype == np.int32
    assert ids.min() >= 0 and ids.max() < w.E
    s = np.sort(ids, axis=1)
    assert np.all(s[:, 1:] != s[:, :-1])
    assert np.array_equal(ids, mw.gen_ids(w))
    g = mw.gen_gates(w)
    assert g.shape == (w.T, w.k) and np.allclose(g.sum(axis=1), 1.0, atol=1e-6)


def test_x_generators():
    w = mw.scaled(mw.WORKLOADS["prefill-fp8"], T=64)
    q, sc = mw.gen_x_fp8(w)
    assert q.shape == (64, w.h) and sc.shape == (64, w.h // 128)
    deq = mw.fp8_codes_to_f32(q).reshape(64, -1, 128) * sc[:, :, None]
    x = np.random.default_rng([w.seed, 3, 0]).standard_normal((64, w.h), dtype=np.float32)
    assert np.all(np.abs(deq.reshape(64, -1) - x) <= np.abs(x) * 2 ** -3 + sc.repeat(128, 1) * 2 ** -9 * 1.01)
    xb = mw.gen_x_bf16(mw.WORKLOADS["tiny"])
    assert xb.dtype == np.uint16 and xb.shape == (256, 1024)


def test_calibrated_skew_hits_targets(oracle_mod):
    """The stored Zipf exponents give the stated imbalance ratios (oracle)."""
    cal = json.load(open(os.path.join(GOLDEN, "zipf_calibration.json")))
    w = mw.WORKLOADS["decode-EP32-r8"]
    assert w.zipf_s == cal["decode-EP32-r8"]["s"]
    prob, keep = oracle_mod.make_problem(w.T, w.h, w.k, w.E, w.R, w.P, w.R_src)
    assert abs(oracle_mod.stats(prob, mw.gen_ids(w))["imbalance_ratio"] - 8.0) < 0.25
    wa = mw.WORKLOADS["decode-EP32-alt"]
    proba, keepa = oracle_mod.make_problem(wa.T, wa.h, wa.k, wa.E, wa.R, wa.P, wa.R_src)
    for st in cal["decode-EP32-alt"]:
        i = st["step"]
        assert wa.s_for_step(i) == st["s"]
        r = oracle_mod.stats(proba, mw.gen_ids(wa, step=i))["imbalance_ratio"]
        assert abs(r - st["target"]) <= 0.02 * st["target"]
