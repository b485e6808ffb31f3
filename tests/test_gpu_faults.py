"""Failure handling on the GPU without faulting it: bounded waits that give
up, data faults reported through the status word, and a context that stays
usable afterwards."""
import time

import numpy as np
import pytest

import moe_workloads as mw
from harness import Case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import torch
    import __graft_entry__ as ge
    ge.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import combine_moe_layout_04_gb300 as m
    return m


def test_bounded_waits_give_up_and_succeed(moe):
    """An mbarrier and a grid barrier that can never complete give up (10 ms
    limit); ones that complete succeed.  The whole test takes well under a
    second and leaves the context usable."""
    t0 = time.time()
    bits = moe.moe_selftest_bounded_waits()
    assert bits == 0xF, hex(bits)
    assert time.time() - t0 < 5.0
    # the context still works: a full layout / dispatch / combine afterwards
    import torch
    w = mw.WORKLOADS["tiny"]
    case = Case(w, torch.device("cuda:0"), y_on_device=False)
    rc, status = case.run()
    assert rc == moe.MOE_OK and status == 0
    assert moe.moe_move_faults() == 0


def test_repeated_selftest_is_stable(moe):
    for _ in range(3):
        assert moe.moe_selftest_bounded_waits() == 0xF
