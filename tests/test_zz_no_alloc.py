"""moe_layout_noalloc: the layout entry point for callers that cannot allocate
device memory (an engine plugin whose device memory the engine plans and
owns, or a plain C caller with no device allocator).  It must give exactly what
the oracle's layout gives -- and what moe_layout gives with a caller
workspace -- call after call, although every call reuses the same fixed
scratch inside the library.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import numpy as np
import pytest

import moe_workloads as mw

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import torch
    import __graft_entry__ as ge
    ge.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import combine_moe_layout_04_gb300 as m
    return m


def _problem(moe, w, dev):
    return moe.Problem(w.T, w.h, w.k, w.E, w.R, w.P, w.R_src,
                       moe.MOE_DTYPE_FP8_E4M3 if w.dtype == "fp8" else moe.MOE_DTYPE_BF16)


def _oracle_problem(oracle_mod, w):
    return oracle_mod.make_problem(w.T, w.h, w.k, w.E, w.R, w.P, w.R_src,
                                   1 if w.dtype == "fp8" else 2, w.scale_group)


CASES = [("prefill-fp8", 0), ("decode-EP32-alt", 15), ("tiny", 0)]


@pytest.mark.parametrize("name,step", CASES, ids=[c[0] for c in CASES])
def test_noalloc_layout_matches_oracle_and_workspace_layout(moe, oracle_mod, name, step):
    import torch
    dev = torch.device("cuda:0")
    w = mw.WORKLOADS[name]
    prob = _problem(moe, w, dev)
    ids_h = mw.gen_ids(w, step=step)
    ids = torch.from_numpy(ids_h).to(dev)
    oprob, keep = _oracle_problem(oracle_mod, w)
    want = oracle_mod.layout(oprob, ids_h)
    want_stats = oracle_mod.stats(oprob, ids_h)
    ref = moe.Layout(prob, dev, with_stats=True)
    ws = moe.alloc_workspace(prob, dev)
    moe.moe_layout(prob, ids, ws, ref)
    rc, bits = moe.moe_status(ws)
    assert rc == moe.MOE_OK and bits == 0
    # two calls in a row on the shared scratch, each checked on its own
    for _ in range(2):
        got = moe.Layout(prob, dev, with_stats=True)
        for n in ("pos", "recv_src", "expert_offset"):
            getattr(got, n).fill_(-3)
        got.stats.fill_(-3)
        moe.moe_layout_noalloc(prob, ids, got)
        torch.cuda.synchronize()
        out = got.to_host()
        for field, val in want.items():
            assert np.array_equal(out[field], val), f"{w.name}: {field} differs from the oracle"
        # the statistics record: word for word as the workspace call's, every
        # field as the oracle's; moe_stats reads it without a workspace
        assert torch.equal(got.stats, ref.stats)
        rc, rec = moe.moe_stats(prob, got, None)
        assert rc == moe.MOE_OK
        st = moe.decode_stats(prob, rec)
        assert st["status"] == 0
        for field, val in want_stats.items():
            assert np.array_equal(np.asarray(st[field]), np.asarray(val)), f"{w.name}: stats {field} differs"


def test_noalloc_reports_bad_ids_through_the_record(moe):
    """An id out of range: the status bit reaches the caller in the record's
    MOE_ST_STATUS word, and every output equals the workspace call's (the bad
    slot is placed as expert 0, in bounds)."""
    import torch
    dev = torch.device("cuda:0")
    w = mw.scaled(mw.WORKLOADS["tiny"], T=256)
    ids_h = mw.gen_ids(w)
    ids_h[17, 1] = w.E + 5
    ids = torch.from_numpy(ids_h).to(dev)
    prob = _problem(moe, w, dev)
    ref = moe.Layout(prob, dev, with_stats=True)
    ws = moe.alloc_workspace(prob, dev)
    moe.moe_layout(prob, ids, ws, ref)
    rc, bits = moe.moe_status(ws)
    assert rc == moe.MOE_ERR_BAD_IDS and bits == moe.MOE_STATUS_ID_RANGE
    for _ in range(2):
        got = moe.Layout(prob, dev, with_stats=True)
        moe.moe_layout_noalloc(prob, ids, got)
        rc, rec = moe.moe_stats(prob, got, None)
        assert rc == moe.MOE_ERR_BAD_IDS and rec[moe.MOE_ST_STATUS] == moe.MOE_STATUS_ID_RANGE
        for field, val in ref.to_host().items():
            assert np.array_equal(got.to_host()[field], val), field
        assert torch.equal(got.stats, ref.stats)
    # a clean call afterwards clears the bit: each call starts from zeroed counters
    good = torch.from_numpy(mw.gen_ids(w)).to(dev)
    got = moe.Layout(prob, dev, with_stats=True)
    moe.moe_layout_noalloc(prob, good, got)
    rc, rec = moe.moe_stats(prob, got, None)
    assert rc == moe.MOE_OK and rec[moe.MOE_ST_STATUS] == 0


def test_noalloc_rejects_problems_beyond_its_scratch(moe):
    import torch
    dev = torch.device("cuda:0")
    w = mw.Workload("big", T=1 << 20, h=128, k=8, E=1024, R=64, P=8, R_src=1)
    prob = _problem(moe, w, dev)
    assert moe.moe_workspace_bytes(prob) > moe.MOE_NOALLOC_SCRATCH_BYTES
    lay = moe.Layout.__new__(moe.Layout)
    for n in moe._LAYOUT_FIELDS:   # never touched: the size check comes first
        setattr(lay, n, torch.empty(1, dtype=torch.int32, device=dev))
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layout_noalloc(prob, torch.empty(1, dtype=torch.int32, device=dev), lay)
    assert ei.value.code == moe.MOE_ERR_CAPACITY
