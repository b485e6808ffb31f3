"""Launch shapes (moe_tuning) change speed, never bytes: the flat, relay and
expert-group calls under non-default shapes -- bulk or vector movers, few SMs,
one CTA per SM, small and odd chunk sizes, few or many warps and stages --
against the oracle, bit for bit, through the C-ABI.  The knobs are this
library's counterparts of the HybridEP issue's NUM_OF_TOKENS_PER_CHUNK_*,
NUM_SMS_DISPATCH / NUM_SMS_COMBINE and NUM_BLOCKS_* ("Poor HybridEP
performance on dual-node 16x B300 GPUs")."""
import numpy as np
import pytest

import moe_workloads as mw
from harness import Case, dev_to_bits, oracle_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__ as ge
    ge.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _shapes():
    import combine_moe_layout_04_gb300 as moe
    V, B = moe.MOE_MOVE_VECTOR, moe.MOE_MOVE_BULK
    return [
        dict(dispatch_kind=B),
        dict(dispatch_kind=B, dispatch_warps=2, dispatch_stages=3, dispatch_chunk_bytes=2048),
        dict(dispatch_kind=B, dispatch_warps=16, dispatch_stages=1, dispatch_chunk_bytes=256, dispatch_sms=5),
        dict(dispatch_kind=B, dispatch_warps=5, dispatch_stages=8, dispatch_chunk_bytes=4112),
        dict(dispatch_kind=V, dispatch_sms=7, dispatch_ctas_per_sm=1),
        dict(combine_kind=V),
        dict(combine_kind=B, combine_sms=3, combine_ctas_per_sm=1),
        dict(dispatch_kind=V, dispatch_sms=1, combine_kind=V, combine_sms=2),
    ]


WORKLOADS = [
    ("prefill-fp8", dict(T=600)),                 # fp8 rows + staged scale rows
    ("decode-EP32-r8", dict(T=640, R_src=8)),     # bf16, two spans per row
    ("tiny", {}),                                 # 2 KB rows, k = 2
]


@pytest.mark.parametrize("name,changes", WORKLOADS, ids=[w[0] for w in WORKLOADS])
def test_flat_calls_under_every_shape(dev, oracle_mod, name, changes):
    import combine_moe_layout_04_gb300 as moe
    w = mw.scaled(mw.WORKLOADS[name], **changes)
    case = Case(w, dev, y_on_device=False)
    prob, keep = oracle_problem(oracle_mod, w)
    ref = oracle_mod.layout(prob, case.ids)
    if w.dtype == "fp8":
        want_recv, want_rs = oracle_mod.dispatch(prob, ref["pos"], case.xq, case.xs)
    else:
        want_recv, want_rs = oracle_mod.dispatch(prob, ref["pos"], case.x), None
    want_out = oracle_mod.combine(prob, ref["pos"], case.y_host, case.gates)
    for shape in _shapes():
        case.prob.tuning = moe.Tuning(**shape)
        case.poison()
        rc, bits = case.run()
        assert rc == 0 and bits == 0, shape
        got = case.lay.to_host()
        for field, val in ref.items():
            assert np.array_equal(got[field], val), (shape, field)
        if want_rs is not None:
            assert np.array_equal(case.recv.cpu().numpy(), want_recv), shape
            assert np.array_equal(case.recv_s.cpu().numpy().view(np.uint32), want_rs.view(np.uint32)), shape
        else:
            assert np.array_equal(dev_to_bits(case.recv), want_recv), shape
        assert np.array_equal(dev_to_bits(case.out), want_out), shape
    assert moe.moe_move_faults() == 0


def test_relay_and_group_calls_under_shapes(dev, oracle_mod):
    import torch
    import combine_moe_layout_04_gb300 as moe
    w = mw.scaled(mw.WORKLOADS["decode-EP32-r8"], T=512, R_src=8)
    case = Case(w, dev, y_on_device=False)
    prob, keep = oracle_problem(oracle_mod, w)
    ref = oracle_mod.layout(prob, case.ids)
    rp = oracle_mod.relay_layout(prob, case.ids)
    n = int((rp >= 0).sum())
    want_relay, _, want_recv, _ = oracle_mod.relay_dispatch(prob, case.ids, ref["pos"], rp, case.x)
    want_part, want_out = oracle_mod.relay_combine(prob, case.ids, ref["pos"], rp, case.y_host, case.gates)
    G = 4
    grp_ref = oracle_mod.expert_groups(prob, G)
    _, want_gout = oracle_mod.combine_groups(prob, case.ids, ref["pos"], grp_ref, G, case.y_host, case.gates)
    for shape in _shapes():
        case.prob.tuning = moe.Tuning(**shape)
        case.poison()
        case.run(dispatch=False, combine=False)
        rel = moe.Relay(case.prob, dev)
        rows = torch.empty((rel.capacity, w.h), dtype=torch.bfloat16, device=dev)
        part = torch.empty((rel.capacity, w.h), dtype=torch.bfloat16, device=dev)
        moe.moe_relay_layout(case.prob, case.lay, case.ws, rel)
        moe.moe_dispatch_relay(case.prob, case.lay, rel, case.x_d, None, rows, None, case.recv, None)
        moe.moe_combine_relay(case.prob, case.lay, rel, case.y_d, case.gates_d, part, case.out)
        assert np.array_equal(dev_to_bits(rows[:n]), want_relay), shape
        assert np.array_equal(dev_to_bits(case.recv), want_recv), shape
        assert np.array_equal(dev_to_bits(part[:n]), want_part), shape
        assert np.array_equal(dev_to_bits(case.out), want_out), shape
        grp = torch.empty(w.E, dtype=torch.int32, device=dev)
        moe.moe_expert_groups(case.prob, G, grp)
        acc = torch.empty((w.T, w.h), dtype=torch.float32, device=dev)
        case.recv.view(torch.uint8).fill_(0xFF)
        for g in range(G):
            moe.moe_dispatch_group(case.prob, case.lay, case.ids_d, grp, g, case.x_d, None, case.recv, None)
            moe.moe_combine_group(case.prob, case.lay, case.ids_d, grp, g, G, case.y_d, case.gates_d, acc, case.out)
        assert np.array_equal(dev_to_bits(case.recv), want_recv), shape
        assert np.array_equal(dev_to_bits(case.out), want_gout), shape
        rc, bits = moe.moe_status(case.ws)
        assert rc == 0 and bits == 0
    assert moe.moe_move_faults() == 0
