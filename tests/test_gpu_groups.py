"""Per-expert-group calls ("Balancing and Beyond", section 3.3): expert groups,
group dispatch and the group combine chain on the GPU vs the oracle, through
the C-ABI.

Group tables and moved bytes are bit-exact; the fp32 accumulator after every
group but the last and the bf16 output are compared bit for bit (both sides
run the same chain: groups ascending, slots ascending inside a group).
"""
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


def _groups(case, G):
    import torch
    grp = torch.empty(case.w.E, dtype=torch.int32, device=case.dev)
    case.moe.moe_expert_groups(case.prob, G, grp)
    return grp


def _run_groups(case, G, grp, check=None, streams=None, acc_offset=0):
    """Layout, then per group: dispatch, combine.  `check(g, acc)` runs after
    each group's combine when given.  With `streams` = (a, b), dispatches run
    on a and combines on b, each combine after its group's dispatch.  The fp32
    chain starts acc_offset floats into its allocation (4: 16-byte but not
    32-byte aligned, the smallest alignment the call accepts)."""
    import torch
    m, c, w = case.moe, case, case.w
    acc = None
    if G > 1:
        buf = torch.empty(w.T * w.h + acc_offset, dtype=torch.float32, device=case.dev)
        acc = buf[acc_offset:].view(w.T, w.h)
    m.moe_layout(c.prob, c.ids_d, c.ws, c.lay)
    if streams is not None:
        sa, sb = streams
        sa.wait_stream(torch.cuda.current_stream())
        sb.wait_stream(torch.cuda.current_stream())
    for g in range(G):
        if streams is None:
            m.moe_dispatch_group(c.prob, c.lay, c.ids_d, grp, g, c.x_d, c.xs_d, c.recv, c.recv_s)
            m.moe_combine_group(c.prob, c.lay, c.ids_d, grp, g, G, c.y_d, c.gates_d, acc, c.out)
        else:
            m.moe_dispatch_group(c.prob, c.lay, c.ids_d, grp, g, c.x_d, c.xs_d, c.recv, c.recv_s, stream=sa)
            ev = torch.cuda.Event()
            ev.record(sa)
            sb.wait_event(ev)
            m.moe_combine_group(c.prob, c.lay, c.ids_d, grp, g, G, c.y_d, c.gates_d, acc, c.out, stream=sb)
        if check is not None:
            torch.cuda.synchronize()
            check(g, acc)
    if streams is not None:
        torch.cuda.current_stream().wait_stream(streams[0])
        torch.cuda.current_stream().wait_stream(streams[1])
    return m.moe_status(c.ws)


def _group_parity(oracle, case, G, e2r=None, streams=None, acc_offset=0):
    import torch
    w = case.w
    prob, keep = oracle_problem(oracle, w, case.src_off, e2r)
    ref = oracle.layout(prob, case.ids)
    grp_ref = oracle.expert_groups(prob, G)
    grp = _groups(case, G)
    assert np.array_equal(grp.cpu().numpy(), grp_ref)
    y = case.y_host
    accs, out = oracle.combine_groups(prob, case.ids, ref["pos"], grp_ref, G, y, case.gates)
    slot_group = grp_ref[case.ids].reshape(-1)
    row_group = np.empty(w.slots, np.int32)
    row_group[ref["pos"].reshape(-1)] = slot_group
    if w.dtype == "fp8":
        want_recv, want_rs = oracle.dispatch(prob, ref["pos"], case.xq, case.xs)
    else:
        want_recv, want_rs = oracle.dispatch(prob, ref["pos"], case.x), None

    def check(g, acc):
        if streams is not None:
            return
        got = case.recv.view(torch.uint8).cpu().numpy().reshape(w.slots, -1)
        want = np.ascontiguousarray(want_recv).view(np.uint8).reshape(w.slots, -1)
        done = row_group <= g
        assert np.array_equal(got[done], want[done]), f"group {g}: dispatched rows differ"
        assert np.all(got[~done] == 0xFF), f"group {g}: a later group's row was written"
        if g < G - 1:
            assert np.array_equal(acc.cpu().numpy().view(np.uint32), accs[g].view(np.uint32)), \
                f"group {g}: fp32 accumulator differs"

    case.poison()
    code, bits = _run_groups(case, G, grp, check, streams, acc_offset)
    assert code == 0 and bits == 0
    got = case.recv.view(torch.uint8).cpu().numpy()
    assert np.array_equal(got.reshape(-1), np.ascontiguousarray(want_recv).view(np.uint8).reshape(-1))
    if want_rs is not None:
        assert np.array_equal(case.recv_s.cpu().numpy().view(np.uint32), want_rs.view(np.uint32))
    assert np.array_equal(dev_to_bits(case.out), out), "group combine output differs"


def _small(**kw):
    base = dict(name="groups", T=300, h=256, k=8, E=64, R=8, P=4, R_src=1)
    base.update(kw)
    return mw.Workload(**base)


GROUP_CASES = [
    (mw.scaled(mw.WORKLOADS["tiny"]), 2),
    (mw.scaled(mw.WORKLOADS["decode-EP32-r8"], T=1000, R_src=8), 2),
    (mw.scaled(mw.WORKLOADS["decode-EP32-r8"], T=640, R_src=8), 4),
    (mw.scaled(mw.WORKLOADS["prefill"], T=700), 3),                    # a middle group
    (mw.scaled(mw.WORKLOADS["prefill-fp8"], T=500), 2),                # fp8 rows + scales
    (_small(T=1), 4),
    (_small(T=257, h=8, k=2, E=16), 2),                                # smallest row, 2-partner stages
    (_small(T=333, k=4, E=32), 4),                                     # 4-partner stages
    (_small(T=200, k=16, E=128, R=16), 4),                             # k > 8: LSU chain
    (_small(T=96, k=32, E=64, R=8), 2),                                # largest top-k
    (_small(T=400, k=8, E=64, R=8), 1),                                # one group: plain combine
    (_small(T=150, k=4, E=16, R=8), 8),                                # more groups than experts per rank
    (_small(T=24, h=76800, k=4, E=16, R=8, P=2, dtype="fp8"), 2),      # 600 scale groups: plain copies
    (_small(T=200, k=8, E=1024, R=16, P=4), 64),                       # the largest E and group count
    (_small(T=128, k=32, E=1024, R=16, P=4), 64),                      # ... with the largest top-k (LSU chain)
]


@pytest.mark.parametrize("w,G", GROUP_CASES,
                         ids=[f"{w.name}_T{w.T}_h{w.h}_k{w.k}_E{w.E}_G{G}_{w.dtype}" for w, G in GROUP_CASES])
def test_group_parity(dev, oracle_mod, w, G):
    _group_parity(oracle_mod, Case(w, dev, y_on_device=False), G)


def test_group_custom_placement(dev, oracle_mod):
    """Random placement with empty ranks: uneven expert counts per rank."""
    w = _small(T=600, k=4, E=48, R=12, P=3, R_src=4)
    rng = np.random.default_rng(21)
    e2r = rng.integers(0, w.R - 2, size=w.E).astype(np.int32)
    _group_parity(oracle_mod, Case(w, dev, expert_to_rank=e2r, y_on_device=False), 3, e2r=e2r)


@pytest.mark.parametrize("kind", ["auto", "bulk"])
@pytest.mark.parametrize("acc_offset", [4, 8])
def test_group_chain_alignment(dev, oracle_mod, acc_offset, kind):
    """The fp32 chain moves as 32-byte accesses when its rows are 32-byte
    aligned and as 16-byte halves otherwise: a chain 16 bytes (and 32 bytes)
    into its allocation gives the same accumulators and output, in the
    register combine (the default) and in the packed shared-memory one."""
    import combine_moe_layout_04_gb300 as moe
    w = mw.scaled(mw.WORKLOADS["decode-EP32-r8"], T=640, R_src=8)
    case = Case(w, dev, y_on_device=False)
    if kind == "bulk":
        case.prob.tuning = moe.Tuning(combine_kind=moe.MOE_MOVE_BULK)
    _group_parity(oracle_mod, case, 4, acc_offset=acc_offset)


def test_group_overlap_on_two_streams(dev, oracle_mod):
    """Dispatches on one stream, combines on another (each after its group's
    dispatch): the per-expert-overlap schedule gives the same bytes."""
    import torch
    w = mw.scaled(mw.WORKLOADS["decode-EP32-r8"], T=1024, R_src=8)
    case = Case(w, dev, y_on_device=False)
    _group_parity(oracle_mod, case, 4, streams=(torch.cuda.Stream(dev), torch.cuda.Stream(dev)))


def test_group_empty_batch(dev):
    import combine_moe_layout_04_gb300 as moe
    w = _small(T=0)
    case = Case(w, dev, ids=np.zeros((0, w.k), np.int32), gates=np.zeros((0, w.k), np.float32),
                y_on_device=False)
    grp = _groups(case, 2)
    code, bits = _run_groups(case, 2, grp)
    assert code == moe.MOE_OK and bits == 0


@pytest.mark.parametrize("name,G", [("decode-EP32-r8", 4), ("prefill-fp8", 2)])
def test_group_full_size(dev, oracle_mod, name, G):
    """Full workload sizes: every receive row compared on the device with the
    row the layout names; the output on sampled tokens against the oracle run
    on those tokens alone (a token's chain depends on its own slots only)."""
    import torch
    w = mw.WORKLOADS[name]
    case = Case(w, dev, y_on_device=True)
    grp = _groups(case, G)
    case.poison()
    code, bits = _run_groups(case, G, grp)
    assert code == 0 and bits == 0
    prob, keep = oracle_problem(oracle_mod, w)
    ref = oracle_mod.layout(prob, case.ids)
    grp_ref = oracle_mod.expert_groups(prob, G)
    assert np.array_equal(grp.cpu().numpy(), grp_ref)
    src_tok = torch.from_numpy((ref["recv_src"] // w.k).astype(np.int64)).to(dev)
    assert torch.equal(case.recv.view(torch.uint8), case.x_d.view(torch.uint8).index_select(0, src_tok))
    if case.recv_s is not None:
        assert torch.equal(case.recv_s.view(torch.int32), case.xs_d.view(torch.int32).index_select(0, src_tok))
    sel = np.sort(np.random.default_rng(9).choice(w.T, size=256, replace=False))
    rows = torch.from_numpy(ref["pos"][sel].reshape(-1).astype(np.int64)).to(dev)
    y_sel = dev_to_bits(case.y_d.index_select(0, rows))
    sub, keep2 = oracle_mod.make_problem(len(sel), w.h, w.k, w.E, w.R, w.P, 1)
    ids_sub = case.ids[sel]
    lay_sub = oracle_mod.layout(sub, ids_sub)
    y_sub = np.empty_like(y_sel)
    y_sub[lay_sub["pos"].reshape(-1)] = y_sel
    _, out_sub = oracle_mod.combine_groups(sub, ids_sub, lay_sub["pos"], grp_ref, G, y_sub, case.gates[sel])
    assert np.array_equal(dev_to_bits(case.out[torch.from_numpy(sel).to(dev)]), out_sub)
