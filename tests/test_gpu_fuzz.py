"""Seeded random problems through every call, against the oracle.

Each case draws T, h, k, E, R, P, the source split, the placement (contiguous
or random with empty ranks) and the dtype, then runs layout + statistics, flat
dispatch and combine, quantise-in-dispatch (fp8), the Mode 2 relay calls and
the expert-group calls, and compares every output with the oracle bit for bit.
"""
import numpy as np
import pytest

import moe_workloads as mw
from harness import Case, dev_to_bits, oracle_problem

pytestmark = pytest.mark.gpu

N_CASES = 160


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__ as ge
    ge.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    P = int(rng.choice([1, 2, 4, 8]))
    H = int(rng.choice([1, 2, 3, 4, 8]))
    R = P * H
    per = int(rng.choice([1, 2, 3, 4, 8]))
    E = R * per
    k = int(rng.integers(1, min(E, 12) + 1))
    dtype = "fp8" if rng.random() < 0.4 else "bf16"
    h = int(rng.choice([128, 256, 384, 1024])) if dtype == "fp8" else int(rng.choice([8, 64, 200, 520, 1024]))
    R_src = int(rng.integers(1, R + 1))
    T = int(rng.integers(0, 700)) // R_src * R_src
    routing = "zipf" if rng.random() < 0.5 else "uniform"
    w = mw.Workload(f"fuzz{seed}", T=T, h=h, k=k, E=E, R=R, P=P, R_src=R_src, dtype=dtype,
                    routing=routing, zipf_s=float(rng.uniform(0.2, 1.5)), seed=seed)
    e2r = None
    if rng.random() < 0.4:
        e2r = rng.integers(0, R, size=E).astype(np.int32)
        e2r[rng.integers(0, E)] = R - 1
    G = int(rng.choice([1, 2, 3, 4]))
    return w, e2r, G


@pytest.mark.parametrize("seed", range(N_CASES))
def test_fuzz_all_calls(dev, oracle_mod, seed):
    w, e2r, G = _draw(seed)
    _check_all_calls(dev, oracle_mod, w, e2r, G)


def _check_all_calls(dev, oracle_mod, w, e2r, G):
    import torch
    c = Case(w, dev, expert_to_rank=e2r, y_on_device=False)
    m = c.moe
    lay = m.Layout(c.prob, dev, with_stats=True)
    m.moe_layout(c.prob, c.ids_d, c.ws, lay)
    m.moe_dispatch(c.prob, lay, c.x_d, c.xs_d, c.recv, c.recv_s)
    m.moe_combine(c.prob, lay, c.y_d, c.gates_d, c.out)
    code, bits = m.moe_status(c.ws)
    assert code == 0 and bits == 0, (code, bits)
    prob, keep = oracle_problem(oracle_mod, w, None, e2r)
    ref = oracle_mod.layout(prob, c.ids)
    got = lay.to_host()
    for name, val in ref.items():
        assert np.array_equal(got[name], val), name
    st = m.decode_stats(c.prob, lay.stats.cpu().numpy())
    for name, val in oracle_mod.stats(prob, c.ids).items():
        assert np.array_equal(np.asarray(st[name]), np.asarray(val)), name
    if w.dtype == "fp8":
        rq, rs = oracle_mod.dispatch(prob, ref["pos"], c.xq, c.xs)
        assert np.array_equal(c.recv.cpu().numpy(), rq)
        assert np.array_equal(c.recv_s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    else:
        assert np.array_equal(dev_to_bits(c.recv), oracle_mod.dispatch(prob, ref["pos"], c.x))
    assert np.array_equal(dev_to_bits(c.out), oracle_mod.combine(prob, ref["pos"], c.y_host, c.gates))

    if w.dtype == "fp8" and w.T > 0:
        xb = mw.gen_x_bf16(w)
        xb_d = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
        m.moe_dispatch_quant(c.prob, lay, xb_d, c.recv, c.recv_s)
        codes, scales = oracle_mod.quantize_dispatch(prob, ref["pos"], xb)
        assert np.array_equal(c.recv.cpu().numpy(), codes)
        assert np.array_equal(c.recv_s.cpu().numpy().view(np.uint32), scales.view(np.uint32))

    # Mode 2 relay
    rel = m.Relay(c.prob, dev)
    cap = max(rel.capacity, 1)
    relay_rows = torch.empty((cap, w.h), dtype=c.recv.dtype, device=dev)
    relay_s = torch.empty((cap, w.h // 128), dtype=torch.float32, device=dev) if c.recv_s is not None else None
    partial = torch.empty((cap, w.h), dtype=torch.bfloat16, device=dev)
    m.moe_relay_layout(c.prob, lay, c.ws, rel)
    m.moe_dispatch_relay(c.prob, lay, rel, c.x_d, c.xs_d, relay_rows, relay_s, c.recv, c.recv_s)
    m.moe_combine_relay(c.prob, lay, rel, c.y_d, c.gates_d, partial, c.out)
    code, bits = m.moe_status(c.ws)
    assert code == 0 and bits == 0, (code, bits)
    rp = oracle_mod.relay_layout(prob, c.ids)
    assert np.array_equal(rel.relay_pos.cpu().numpy(), rp)
    n = int((rp >= 0).sum())
    if w.dtype == "fp8":
        r_rows, r_s, r_recv, r_rs = oracle_mod.relay_dispatch(prob, c.ids, ref["pos"], rp, c.xq, c.xs)
        assert np.array_equal(relay_rows[:n].cpu().numpy(), r_rows)
        assert np.array_equal(c.recv.cpu().numpy(), r_recv)
    else:
        r_rows, _, r_recv, _ = oracle_mod.relay_dispatch(prob, c.ids, ref["pos"], rp, c.x)
        assert np.array_equal(dev_to_bits(relay_rows[:n]), r_rows)
        assert np.array_equal(dev_to_bits(c.recv), r_recv)
    part, out = oracle_mod.relay_combine(prob, c.ids, ref["pos"], rp, c.y_host, c.gates)
    assert np.array_equal(dev_to_bits(partial[:n]), part)
    assert np.array_equal(dev_to_bits(c.out), out)

    # expert groups
    grp = torch.empty(w.E, dtype=torch.int32, device=dev)
    m.moe_expert_groups(c.prob, G, grp)
    grp_ref = oracle_mod.expert_groups(prob, G)
    assert np.array_equal(grp.cpu().numpy(), grp_ref)
    acc = torch.empty((max(w.T, 1), w.h), dtype=torch.float32, device=dev)
    for g in range(G):
        m.moe_dispatch_group(c.prob, lay, c.ids_d, grp, g, c.x_d, c.xs_d, c.recv, c.recv_s)
        m.moe_combine_group(c.prob, lay, c.ids_d, grp, g, G, c.y_d, c.gates_d, acc, c.out)
    _, out = oracle_mod.combine_groups(prob, c.ids, ref["pos"], grp_ref, G, c.y_host, c.gates)
    assert np.array_equal(dev_to_bits(c.out), out)
    assert m.moe_move_faults() == 0


LARGE = [
    # grids too large to be co-resident: the two-kernel layout path; relay tiles of 1024 tokens
    (mw.Workload("large-bf16", T=150000, h=16, k=8, E=64, R=16, P=4, R_src=16, routing="zipf", zipf_s=0.8,
                 seed=7), 2),
    (mw.Workload("large-fp8", T=100000, h=128, k=6, E=32, R=8, P=2, R_src=1, dtype="fp8", seed=8), 4),
]


@pytest.mark.parametrize("w,G", LARGE, ids=[w.name for w, _ in LARGE])
def test_large_batch_all_calls(dev, oracle_mod, w, G):
    """Every call at 100K-150K tokens (small rows keep the oracle quick)."""
    _check_all_calls(dev, oracle_mod, w, None, G)
