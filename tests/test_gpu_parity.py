"""GPU path vs the CPU oracle, through the C-ABI, on seeded inputs.

Integer outputs (counts, offsets, mask, pos, recv_src, statistics) and moved
bytes must be bit-exact.  Combined outputs must satisfy |gpu - ref| <=
2^-7 |ref| elementwise (exact where ref is 0); both sides run the same
ascending-slot fp32 fma chain, so bit-exact equality is asserted too.
"""
import numpy as np
import pytest

import moe_workloads as mw
from harness import Case, bf16_to_dev, dev_to_bits, oracle_problem

pytestmark = pytest.mark.gpu

TOL = 2.0 ** -7


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__ as ge
    ge.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _check_layout(oracle, case, src_off=None, e2r=None):
    prob, keep = oracle_problem(oracle, case.w, src_off, e2r)
    ref = oracle.layout(prob, case.ids)
    got = case.lay.to_host()
    for name, val in ref.items():
        assert np.array_equal(got[name], val), f"layout {name} differs"
    return prob, ref


def _check_stats(oracle, case, prob):
    ref = oracle.stats(prob, case.ids)
    got = case.stats_host()
    assert got["status"] == 0
    for name, val in ref.items():
        assert np.array_equal(np.asarray(got[name]), np.asarray(val)), f"stats {name} differs"
    assert got["num_hosts"] == case.w.H


def _check_dispatch(oracle, case, prob, ref, sample=None):
    w = case.w
    if sample is None:
        if w.dtype == "fp8":
            rq, rs = oracle.dispatch(prob, ref["pos"], case.xq, case.xs)
            assert np.array_equal(case.recv.cpu().numpy(), rq)
            assert np.array_equal(case.recv_s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
        else:
            assert np.array_equal(dev_to_bits(case.recv), oracle.dispatch(prob, ref["pos"], case.x))
        return
    rows = np.random.default_rng(5).choice(w.slots, size=min(sample, w.slots), replace=False)
    src_tok = ref["recv_src"][rows] // w.k
    if w.dtype == "fp8":
        assert np.array_equal(case.recv[rows].cpu().numpy(), case.xq[src_tok])
        assert np.array_equal(case.recv_s[rows].cpu().numpy().view(np.uint32), case.xs[src_tok].view(np.uint32))
    else:
        assert np.array_equal(dev_to_bits(case.recv[rows]), case.x[src_tok])


def _assert_combine_close(got_bits, ref_bits):
    g = mw.bf16_bits_to_f32(got_bits).astype(np.float64)
    r = mw.bf16_bits_to_f32(ref_bits).astype(np.float64)
    assert np.all(np.abs(g - r) <= TOL * np.abs(r)), "combine outside 2^-7 |ref|"
    assert np.array_equal(got_bits, ref_bits), "combine not bit-exact"


def _check_combine(oracle, case, prob, ref, sample=None):
    w = case.w
    if sample is None:
        y = case.y_host if case.y_host is not None else dev_to_bits(case.y_d)
        _assert_combine_close(dev_to_bits(case.out), oracle.combine(prob, ref["pos"], y, case.gates))
        return
    toks = np.sort(np.random.default_rng(6).choice(w.T, size=min(sample, w.T), replace=False))
    import torch
    rows = torch.from_numpy(ref["pos"][toks].reshape(-1).astype(np.int64)).to(case.dev)
    y_sub = dev_to_bits(case.y_d.index_select(0, rows))
    sub, keep = oracle.make_problem(len(toks), w.h, w.k, w.E, w.R, w.P, 1)
    pos_sub = np.arange(len(toks) * w.k, dtype=np.int32).reshape(len(toks), w.k)
    want = oracle.combine(sub, pos_sub, y_sub, case.gates[toks])
    _assert_combine_close(dev_to_bits(case.out[torch.from_numpy(toks).to(case.dev)]), want)


def _full_check(oracle, case, src_off=None, e2r=None, sample=None):
    case.poison()
    rc, bits = case.run()
    assert rc == 0 and bits == 0, (rc, bits)
    prob, ref = _check_layout(oracle, case, src_off, e2r)
    _check_stats(oracle, case, prob)
    _check_dispatch(oracle, case, prob, ref, sample)
    _check_combine(oracle, case, prob, ref, sample)
    return prob, ref


# ------------------------------------------------------------ moderate sizes

MODERATE = [
    ("tiny", {}),
    ("decode-EP32-r8", dict(T=1000, R_src=8)),          # ragged last block (1000 = 7*128 + 104)
    ("decode-EP32-s1.1", dict(T=640, R_src=20)),
    ("decode-EP32-alt", dict(T=777, R_src=7)),
    ("prefill", dict(T=1000)),
    ("prefill-fp8", dict(T=900)),
]


@pytest.mark.parametrize("name,changes", MODERATE, ids=[m[0] for m in MODERATE])
def test_parity_moderate(dev, oracle_mod, name, changes):
    w = mw.scaled(mw.WORKLOADS[name], **changes)
    steps = [0, w.steps - 1] if w.steps > 1 else [0]
    for step in steps:
        case = Case(w, dev, step=step, y_on_device=False)
        _full_check(oracle_mod, case)


# ------------------------------------------------------------ full sizes

@pytest.mark.parametrize("name", ["decode-EP32-r8", "decode-EP32-s1.1", "decode-EP32-alt", "prefill",
                                  "prefill-fp8"])
def test_parity_full_size(dev, oracle_mod, name):
    """Full workload sizes: layout and statistics compared in full, dispatch
    and combine on sampled rows / tokens."""
    w = mw.WORKLOADS[name]
    for step in ([0, 15] if w.steps > 1 else [0]):
        case = Case(w, dev, step=step, y_on_device=True)
        prob, ref = _full_check(oracle_mod, case, sample=384)
        # every receive row, compared on the device with the row the oracle's
        # inverse map names
        import torch
        src_tok = torch.from_numpy((ref["recv_src"] // w.k).astype(np.int64)).to(dev)
        assert torch.equal(case.recv.view(torch.uint8), case.x_d.view(torch.uint8).index_select(0, src_tok))
        if case.recv_s is not None:
            assert torch.equal(case.recv_s.view(torch.int32), case.xs_d.view(torch.int32).index_select(0, src_tok))


# ------------------------------------------------------------ edge cases

def _small(**kw):
    base = dict(name="edge", T=64, h=256, k=2, E=8, R=4, P=2, R_src=1)
    base.update(kw)
    return mw.Workload(**base)


@pytest.mark.parametrize("w", [
    _small(T=1),
    _small(T=129, k=1),
    _small(T=300, k=8, E=8),                       # E = k: every token hits every expert
    _small(T=257, h=8),                            # smallest bf16 row
    _small(T=200, h=520),                          # h not a multiple of 128
    _small(T=130, h=128, dtype="fp8"),             # one scale per row
    _small(T=333, h=1024, k=4, E=64, R=16, P=4, dtype="fp8"),
    _small(T=256, k=3, E=30, R=6, P=3, R_src=4),   # k not a power of two
    _small(T=96, k=32, E=64, R=8, P=2),            # largest top-k
    _small(T=512, k=8, E=1024, R=1024, P=16, R_src=512),  # largest E and R, 64 hosts
    _small(T=645, h=200, k=8, E=512, R=64, P=8, R_src=43),  # 45.9 KB dynamic + static > 48 KB: needs the opt-in
    _small(T=24, h=76800, k=4, E=16, R=8, P=2, dtype="fp8"),  # 600 scale groups, staged with their chunk
], ids=lambda w: f"T{w.T}_h{w.h}_k{w.k}_E{w.E}_R{w.R}_{w.dtype}")
def test_parity_edge_shapes(dev, oracle_mod, w):
    _full_check(oracle_mod, Case(w, dev, y_on_device=False))


def test_empty_batch(dev):
    import torch
    import combine_moe_layout_04_gb300 as moe
    w = _small(T=0)
    case = Case(w, dev, ids=np.zeros((0, w.k), np.int32), gates=np.zeros((0, w.k), np.float32),
                y_on_device=False)
    rc, bits = case.run()
    assert rc == 0 and bits == 0
    assert case.lay.expert_count.sum().item() == 0
    assert torch.all(case.lay.expert_offset == 0) and torch.all(case.lay.rank_offset == 0)
    st = case.stats_host()
    assert st["T"] == 0 and st["imbalance_ratio"] == 0.0
    assert moe.MOE_OK == 0


def test_all_tokens_to_one_expert_set(dev, oracle_mod):
    """Every token picks the same k experts: ratio E/k, empty experts and ranks."""
    w = _small(T=1000, k=4, E=32, R=8, P=4)
    ids = np.tile(np.array([[5, 9, 2, 30]], np.int32), (w.T, 1))
    case = Case(w, dev, ids=ids, y_on_device=False)
    _full_check(oracle_mod, case)
    assert case.stats_host()["imbalance_ratio"] == w.E / w.k


def test_custom_placement(dev, oracle_mod):
    """expert_to_rank as a random map with empty ranks; receive order follows (rank, e)."""
    w = _small(T=700, k=4, E=48, R=12, P=3, R_src=4)
    rng = np.random.default_rng(3)
    e2r = rng.integers(0, w.R - 2, size=w.E).astype(np.int32)   # ranks R-2, R-1 own nothing
    case = Case(w, dev, expert_to_rank=e2r, y_on_device=False)
    _full_check(oracle_mod, case, e2r=e2r)


def test_unbalanced_source_ranks(dev, oracle_mod):
    """The unbalanced-batch example: 16 ranks on 2 hosts, 384 vs 64 tokens."""
    per = [384] * 8 + [64] * 8
    src_off = np.concatenate([[0], np.cumsum(per)]).astype(np.int32)
    ids = np.concatenate([np.arange(n) % 16 for n in per]).astype(np.int32)[:, None]
    w = _small(T=int(src_off[-1]), k=1, E=16, R=16, P=8, R_src=16, h=64)
    case = Case(w, dev, ids=ids, src_offsets=src_off, y_on_device=False)
    _full_check(oracle_mod, case, src_off=src_off)
    st = case.stats_host()
    assert all(st["recv_remote"][r] == 192 and st["recv_local"][r] == 28 for r in range(8, 16))


def test_bad_ids_reported_without_fault(dev):
    import torch
    import combine_moe_layout_04_gb300 as moe
    w = _small(T=300, k=4, E=16)
    ids = mw.gen_ids(w)
    ids[7, 2] = 99          # out of range
    ids[250, 3] = ids[250, 0]  # repeated in a row
    case = Case(w, dev, ids=ids, y_on_device=False)
    rc, bits = case.run()
    assert rc == moe.MOE_ERR_BAD_IDS
    assert bits == moe.MOE_STATUS_ID_RANGE | moe.MOE_STATUS_ID_REPEAT
    pos = case.lay.pos.cpu().numpy().ravel()
    assert np.array_equal(np.sort(pos), np.arange(w.slots))   # still a permutation in bounds
    ids2 = mw.gen_ids(w)
    case.ids_d.copy_(torch.from_numpy(ids2))
    rc, bits = case.run()
    assert rc == moe.MOE_OK and bits == 0


def test_bad_placement_reported(dev):
    import combine_moe_layout_04_gb300 as moe
    w = _small(T=100)
    e2r = np.arange(w.E, dtype=np.int32) // 2
    e2r[3] = 77
    case = Case(w, dev, expert_to_rank=e2r, y_on_device=False)
    rc, bits = case.run()
    assert rc == moe.MOE_ERR_INVALID and bits & moe.MOE_STATUS_PLACEMENT


def test_deterministic_runs(dev):
    import torch
    w = mw.scaled(mw.WORKLOADS["decode-EP32-s1.1"], T=2048, R_src=16)
    case = Case(w, dev, y_on_device=False)
    case.run()
    first = [t.clone() for t in (case.lay.pos, case.lay.recv_src, case.recv, case.out, case.stats)]
    for _ in range(3):
        case.poison()
        case.run()
        now = (case.lay.pos, case.lay.recv_src, case.recv, case.out, case.stats)
        for a, b in zip(first, now):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_round_trip_identity_experts(dev):
    """Dispatch then combine with identity experts and unit weights gives k*x
    exactly (k = 8, a power of two), at the decode workload's full size."""
    import torch
    w = mw.WORKLOADS["decode-EP32-r8"]
    case = Case(w, dev, gates=np.ones((w.T, w.k), np.float32), y_on_device=True)
    case.run(combine=False)
    case.moe.moe_combine(case.prob, case.lay, case.recv, case.gates_d, case.out)
    want = bf16_to_dev(mw.f32_to_bf16_bits(mw.bf16_bits_to_f32(case.x) * np.float32(w.k)), dev)
    # equal as values: an input of -0.0 sums to +0.0 from the +0.0 start of the
    # fma chain, while k * (-0.0) is -0.0
    assert torch.equal(case.out.float(), want.float())


def test_layout_two_kernel_path_large_batch(dev, oracle_mod):
    """T = 200000 tokens (1563 blocks) is more than one cooperative grid can
    hold, so the layout runs as two kernels; results must not change."""
    w = mw.Workload("big", T=200000, h=8, k=2, E=16, R=4, P=2, R_src=4, routing="zipf", zipf_s=0.8)
    case = Case(w, dev, y_on_device=False)
    rc, bits = case.run(dispatch=False, combine=False)
    assert rc == 0 and bits == 0
    prob, ref = _check_layout(oracle_mod, case)
    _check_stats(oracle_mod, case, prob)


def test_stats_delivered_with_the_layout(dev):
    """moe_layout can write the statistics record itself (layout.stats); it
    equals what moe_stats_device copies out of the workspace."""
    import torch
    import combine_moe_layout_04_gb300 as moe
    w = mw.scaled(mw.WORKLOADS["decode-EP32-r8"], T=1024, R_src=8)
    case = Case(w, dev, y_on_device=False)
    lay = moe.Layout(case.prob, dev, with_stats=True)
    lay.stats.fill_(-1)
    moe.moe_layout(case.prob, case.ids_d, case.ws, lay)
    moe.moe_stats_device(case.prob, case.ws, case.stats)
    torch.cuda.synchronize()
    assert torch.equal(lay.stats, case.stats)
    assert moe.moe_move_faults() == 0


@pytest.mark.parametrize("name", ["prefill-fp8", "decode-EP32-r8", "decode-EP32-alt", "tiny"])
def test_host_stats_record_matches_oracle(dev, oracle_mod, name):
    """moe_stats, the call that synchronises and hands the record to the host
    ("Balancing and Beyond", sections 1 and 2: bytes leaving each rank and the
    imbalance ratio), read from the workspace and from layout.stats: every
    field equals the oracle's at the workload's full size."""
    import combine_moe_layout_04_gb300 as moe
    w = mw.WORKLOADS[name]
    step = w.steps - 1
    case = Case(w, dev, step=step, y_on_device=True)
    case.run(dispatch=False, combine=False, stats=False)
    prob, keep = oracle_problem(oracle_mod, w)
    ref = oracle_mod.stats(prob, case.ids)
    for lay, ws in ((case.lay, case.ws), (moe.Layout(case.prob, dev, with_stats=True), None)):
        if ws is None:
            moe.moe_layout(case.prob, case.ids_d, case.ws, lay)
        rc, rec = moe.moe_stats(case.prob, lay, ws)
        assert rc == moe.MOE_OK
        got = moe.decode_stats(case.prob, rec)
        assert got["status"] == 0 and got["num_hosts"] == w.H
        for field, val in ref.items():
            assert np.array_equal(np.asarray(got[field]), np.asarray(val)), f"stats {field} differs"


def test_host_stats_reports_bad_ids(dev):
    """The syncing moe_stats returns the status of the record it hands over."""
    import combine_moe_layout_04_gb300 as moe
    w = _small(T=300, k=4, E=16)
    ids = mw.gen_ids(w)
    ids[5, 1] = -2
    case = Case(w, dev, ids=ids, y_on_device=False)
    case.run(dispatch=False, combine=False, stats=False)
    rc, rec = moe.moe_stats(case.prob, case.lay, case.ws)
    assert rc == moe.MOE_ERR_BAD_IDS and rec[moe.MOE_ST_STATUS] == moe.MOE_STATUS_ID_RANGE


@pytest.mark.parametrize("name", ["prefill-fp8", "decode-EP32-r8"])
def test_stats_beside_the_movers(dev, oracle_mod, name):
    """Without layout.stats the layout kernel ends with its positions and
    moe_stats_device makes the record on a second stream while dispatch and
    combine run on the first: the record equals the oracle's, and the moved
    rows are those of the plain order of calls (full workload size, also
    replayed from a CUDA graph)."""
    import torch
    import combine_moe_layout_04_gb300 as moe
    w = mw.WORKLOADS[name]
    case = Case(w, dev, y_on_device=True)
    main, side = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    prob, keep = oracle_problem(oracle_mod, w)
    ref = oracle_mod.stats(prob, case.ids)

    def step(s):
        moe.moe_layout(case.prob, case.ids_d, case.ws, case.lay, s)
        side.wait_stream(s)
        moe.moe_stats_device(case.prob, case.ws, case.stats, side)
        moe.moe_dispatch(case.prob, case.lay, case.x_d, case.xs_d, case.recv, case.recv_s, s)
        moe.moe_combine(case.prob, case.lay, case.y_d, case.gates_d, case.out, s)
        s.wait_stream(side)

    def check():
        got = case.stats_host()
        assert got["status"] == 0
        for field, val in ref.items():
            assert np.array_equal(np.asarray(got[field]), np.asarray(val)), f"stats {field} differs"

    case.poison()
    case.stats.fill_(-1)
    main.wait_stream(torch.cuda.current_stream())  # after the poison, which runs on the current stream
    step(main)
    torch.cuda.synchronize()
    check()
    out0, recv0 = case.out.clone(), case.recv.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(main):
        g.capture_begin()
        step(main)
        g.capture_end()
    case.poison()
    case.stats.fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    check()
    assert torch.equal(case.out.view(torch.int16), out0.view(torch.int16))
    assert torch.equal(case.recv.view(torch.uint8), recv0.view(torch.uint8))
    assert moe.moe_move_faults() == 0
