"""moe_layout_noalloc: the layout entry point for callers that cannot allocate
device memory (an engine plugin whose device memory the engine plans and
owns, or a plain C caller with no device allocator).  It must give exactly what
moe_layout gives with a caller workspace, call after call, although every call
reuses the same fixed scratch inside the library.

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


def test_noalloc_layout_matches_workspace_layout(moe):
    import torch
    dev = torch.device("cuda:0")
    cases = [(mw.WORKLOADS["prefill-fp8"], 0), (mw.WORKLOADS["decode-EP32-alt"], 15),
             (mw.WORKLOADS["tiny"], 0)]
    for w, step in cases:
        prob = _problem(moe, w, dev)
        ids = torch.from_numpy(mw.gen_ids(w, step=step)).to(dev)
        ref = moe.Layout(prob, dev)
        ws = moe.alloc_workspace(prob, dev)
        moe.moe_layout(prob, ids, ws, ref)
        rc, bits = moe.moe_status(ws)
        assert rc == moe.MOE_OK and bits == 0
        want = ref.to_host()
        # two calls in a row on the shared scratch, each checked on its own
        for _ in range(2):
            got = moe.Layout(prob, dev)
            for n in ("pos", "recv_src", "expert_offset"):
                getattr(got, n).fill_(-3)
            moe.moe_layout_noalloc(prob, ids, got)
            torch.cuda.synchronize()
            out = got.to_host()
            for name, val in want.items():
                assert np.array_equal(out[name], val), f"{w.name}: {name} differs"


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
