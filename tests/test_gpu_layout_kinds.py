"""The three forms of moe_layout's kernels -- split (position blocks wait only
for the expert histograms while other blocks count tokens for the
statistics), fused (one cooperative kernel, one barrier) and two kernels --
give the same layout and statistics record, equal to the oracle's, bit for
bit: seeded random problems (several source ranks inside one block, random
placements with empty ranks, k up to 32, E = R = 1024 with 64 hosts), the
record written by the layout itself and by moe_stats_device, and the same
status bits for bad ids."""
import numpy as np
import pytest

import moe_workloads as mw
from harness import Case, oracle_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__ as ge
    ge.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _kinds():
    import combine_moe_layout_04_gb300 as moe
    return [moe.MOE_LAYOUT_SPLIT, moe.MOE_LAYOUT_FUSED, moe.MOE_LAYOUT_TWO_KERNELS]


def _draw(seed):
    rng = np.random.default_rng(5000 + seed)
    P = int(rng.choice([1, 2, 4, 8]))
    H = int(rng.choice([1, 2, 3, 4, 8]))
    R = P * H
    E = R * int(rng.choice([1, 2, 4, 8]))
    k = int(rng.integers(1, min(E, 32) + 1))
    R_src = int(rng.integers(1, R + 1))
    T = max(int(rng.integers(1, 3000)) // R_src, 1) * R_src
    w = mw.Workload(f"kinds{seed}", T=T, h=8, k=k, E=E, R=R, P=P, R_src=R_src,
                    routing="zipf" if rng.random() < 0.5 else "uniform",
                    zipf_s=float(rng.uniform(0.2, 1.5)), seed=seed)
    e2r = None
    if rng.random() < 0.4:
        e2r = rng.integers(0, R, size=E).astype(np.int32)
        e2r[rng.integers(0, E)] = R - 1
    return w, e2r


CASES = [_draw(s) for s in range(24)] + [
    (mw.Workload("one-token", T=1, h=8, k=3, E=8, R=4, P=2, R_src=1), None),
    (mw.Workload("ragged", T=1000, h=8, k=8, E=256, R=32, P=8, R_src=8), None),
    (mw.Workload("wide", T=640, h=8, k=8, E=1024, R=1024, P=16, R_src=64, routing="zipf", zipf_s=0.9), None),
    (mw.Workload("k32", T=384, h=8, k=32, E=64, R=8, P=4, R_src=3), None),
]


def _run(case, kind, with_stats):
    import combine_moe_layout_04_gb300 as moe
    case.prob.tuning = moe.Tuning(layout_kind=kind)
    case.poison()
    lay = moe.Layout(case.prob, case.dev, with_stats=with_stats)
    if with_stats:
        lay.stats.fill_(-1)
    moe.moe_layout(case.prob, case.ids_d, case.ws, lay)
    case.stats.fill_(-1)
    moe.moe_stats_device(case.prob, case.ws, case.stats)
    return lay


@pytest.mark.parametrize("w,e2r", CASES, ids=[c[0].name for c in CASES])
def test_every_layout_kind_matches_oracle(dev, oracle_mod, w, e2r):
    import combine_moe_layout_04_gb300 as moe
    case = Case(w, dev, expert_to_rank=e2r, y_on_device=False)
    prob, keep = oracle_problem(oracle_mod, w, None, e2r)
    ref = oracle_mod.layout(prob, case.ids)
    ref_stats = oracle_mod.stats(prob, case.ids)
    for kind in _kinds():
        for with_stats in (True, False):
            lay = _run(case, kind, with_stats)
            rc, bits = moe.moe_status(case.ws)
            assert rc == 0 and bits == 0, (kind, rc, bits)
            got = lay.to_host()
            for name, val in ref.items():
                assert np.array_equal(got[name], val), (kind, with_stats, name)
            records = [case.stats.cpu().numpy()]
            if with_stats:
                records.append(lay.stats.cpu().numpy())
            for rec in records:
                st = moe.decode_stats(case.prob, rec)
                assert st["status"] == 0
                for name, val in ref_stats.items():
                    assert np.array_equal(np.asarray(st[name]), np.asarray(val)), (kind, with_stats, name)
    assert moe.moe_move_faults() == 0


def test_every_layout_kind_reports_bad_ids(dev):
    """Out-of-range and repeated ids set the same status bits in every form;
    positions stay a permutation of the receive rows."""
    import combine_moe_layout_04_gb300 as moe
    w = mw.Workload("bad", T=700, h=8, k=4, E=16, R=4, P=2, R_src=2)
    ids = mw.gen_ids(w)
    ids[7, 2] = 99
    ids[650, 3] = ids[650, 0]
    case = Case(w, dev, ids=ids, y_on_device=False)
    for kind in _kinds():
        lay = _run(case, kind, True)
        rc, bits = moe.moe_status(case.ws)
        assert rc == moe.MOE_ERR_BAD_IDS, kind
        assert bits == moe.MOE_STATUS_ID_RANGE | moe.MOE_STATUS_ID_REPEAT, kind
        pos = lay.pos.cpu().numpy().ravel()
        assert np.array_equal(np.sort(pos), np.arange(w.slots)), kind
        assert moe.decode_stats(case.prob, lay.stats.cpu().numpy())["status"] == bits
