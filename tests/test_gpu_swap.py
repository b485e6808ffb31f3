"""Per-step intra-host expert swap planning on the GPU vs the oracle."""
import numpy as np
import pytest

import moe_workloads as mw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__ as ge
    ge.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _plan(dev, w, ids, tau, e2r=None):
    import torch
    import combine_moe_layout_04_gb300 as moe
    e2r_d = None if e2r is None else torch.from_numpy(np.asarray(e2r, np.int32)).to(dev)
    prob = moe.Problem(w.T, w.h, w.k, w.E, w.R, w.P, w.R_src, moe.MOE_DTYPE_BF16, e2r_d)
    lay = moe.Layout(prob, dev)
    ws = moe.alloc_workspace(prob, dev)
    moe.moe_layout(prob, torch.from_numpy(np.ascontiguousarray(ids, np.int32)).to(dev), ws, lay)
    new = torch.full((w.E,), -5, dtype=torch.int32, device=dev)
    swaps = torch.full((w.H, w.P // 2, 6), -9, dtype=torch.int32, device=dev)
    moe.moe_swap_plan(prob, lay, tau, new, swaps)
    rc, bits = moe.moe_status(ws)
    assert rc == moe.MOE_OK
    return lay.expert_count.cpu().numpy(), new.cpu().numpy(), swaps.cpu().numpy()


def test_swap_worked_example(dev):
    """160 / 100 -> 130 / 130 by exchanging e0 (60 tokens) and e1 (30)."""
    w = mw.Workload("swap", T=260, h=8, k=1, E=6, R=2, P=2, R_src=1)
    e2r = np.array([0, 1, 0, 1, 0, 1], np.int32)
    counts = [60, 30, 50, 35, 50, 35]
    ids = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)])[:, None]
    cnt, new, swaps = _plan(dev, w, ids, 30, e2r)
    assert list(cnt) == counts
    assert tuple(swaps[0, 0]) == (0, 1, 0, 1, 160, 130)
    assert list(new) == [1, 0, 0, 1, 0, 1]


def _oracle_counts(oracle_mod, w, ids, e2r=None):
    """Expert counts from the oracle's own layout of the same ids: the swap
    plan's expected values never take an input from the CUDA path."""
    prob, keep = oracle_mod.make_problem(w.T, w.h, w.k, w.E, w.R, w.P, w.R_src,
                                         expert_to_rank=None if e2r is None else np.asarray(e2r, np.int32))
    return prob, keep, oracle_mod.layout(prob, np.ascontiguousarray(ids, np.int32))["expert_count"]


@pytest.mark.parametrize("name", ["decode-EP32-r8", "decode-EP32-s1.1", "prefill-fp8"])
def test_swap_plan_parity(dev, oracle_mod, name):
    """"Balancing and Beyond", section 3.1 and Figure 2(b): the plan from the
    layout's expert counts, against the oracle's plan from the oracle's counts."""
    w = mw.WORKLOADS[name]
    ids = mw.gen_ids(w)
    prob, keep, want_cnt = _oracle_counts(oracle_mod, w, ids)
    for tau in (0, 5, 200):
        cnt, new, swaps = _plan(dev, w, ids, tau)
        assert np.array_equal(cnt, want_cnt), "GPU expert counts differ from the oracle layout's"
        want_new, want_swaps = oracle_mod.swap_plan(prob, want_cnt, tau)
        assert np.array_equal(new, want_new)
        assert np.array_equal(swaps, want_swaps)


def test_swap_plan_custom_placement_and_next_layout(dev, oracle_mod):
    """With a custom placement, and the plan fed to the next layout: the
    heaviest rank of each host gets lighter by the planned amount."""
    w = mw.scaled(mw.WORKLOADS["decode-EP32-r8"], T=2048, R_src=16)
    rng = np.random.default_rng(12)
    e2r = rng.permutation(np.repeat(np.arange(w.R), w.E // w.R)).astype(np.int32)
    ids = mw.gen_ids(w)
    prob, keep, want_cnt = _oracle_counts(oracle_mod, w, ids, e2r)
    cnt, new, swaps = _plan(dev, w, ids, 1, e2r)
    assert np.array_equal(cnt, want_cnt), "GPU expert counts differ from the oracle layout's"
    want_new, want_swaps = oracle_mod.swap_plan(prob, want_cnt, 1)
    assert np.array_equal(new, want_new) and np.array_equal(swaps, want_swaps)
    # the next step's layout under the new placement, against the oracle's
    prob2, keep2, want_cnt2 = _oracle_counts(oracle_mod, w, ids, want_new)
    cnt2, _, _ = _plan(dev, w, ids, 1, new)
    assert np.array_equal(cnt2, want_cnt2)
    load_after = np.bincount(want_new, weights=want_cnt2, minlength=w.R)
    for hh in range(w.H):
        for a, b, x, y, old, best in want_swaps[hh]:
            if old - best >= 1:
                assert max(load_after[a], load_after[b]) == best
