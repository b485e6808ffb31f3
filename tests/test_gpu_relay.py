"""Mode 2 relay on one buffer ("Balancing and Beyond", section 3.2): relay
rows, two-hop dispatch and two-hop combine on the GPU vs the oracle, through
the C-ABI.

Relay positions and moved bytes are bit-exact.  Both sides of the combine run
the same fp32 chains (ascending slots inside a host, then ascending hosts) with
the same two roundings to bf16, so the outputs are compared bit for bit; the
oracle's own pins bound them against the exact sum.
"""
import numpy as np
import pytest

import moe_workloads as mw
from harness import Case, bf16_to_dev, dev_to_bits, oracle_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__ as ge
    ge.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _host_of(w, ids, e2r=None):
    rank = (ids // (w.E // w.R)) if e2r is None else np.asarray(e2r)[ids]
    return rank // w.P


class RelayCase:
    """A Case plus relay arrays and buffers, run through the relay entry points."""

    def __init__(self, case: Case, capacity=None, alloc_rows=None):
        import torch
        moe, w, dev = case.moe, case.w, case.dev
        self.case = case
        self.rel = moe.Relay(case.prob, dev, capacity)
        cap = max(self.rel.capacity, 1) if alloc_rows is None else alloc_rows
        if alloc_rows is not None:
            self.rel.relay_src = torch.empty(alloc_rows, dtype=torch.int32, device=dev)
        if w.dtype == "fp8":
            self.relay_rows = torch.empty((cap, w.h), dtype=torch.uint8, device=dev)
            self.relay_s = torch.empty((cap, w.h // w.scale_group), dtype=torch.float32, device=dev)
        else:
            self.relay_rows = torch.empty((cap, w.h), dtype=torch.bfloat16, device=dev)
            self.relay_s = None
        self.partial = torch.empty((cap, w.h), dtype=torch.bfloat16, device=dev)

    def poison(self):
        import torch
        self.case.poison()
        for t in (self.rel.relay_pos, self.rel.relay_src, self.rel.slot_relay):
            t.fill_(-9)
        for t in (self.relay_rows, self.partial) + ((self.relay_s,) if self.relay_s is not None else ()):
            t.view(torch.uint8).fill_(0xEE)

    def run(self):
        c, m = self.case, self.case.moe
        m.moe_layout(c.prob, c.ids_d, c.ws, c.lay)
        m.moe_relay_layout(c.prob, c.lay, c.ws, self.rel)
        m.moe_dispatch_relay(c.prob, c.lay, self.rel, c.x_d, c.xs_d, self.relay_rows, self.relay_s,
                             c.recv, c.recv_s)
        m.moe_combine_relay(c.prob, c.lay, self.rel, c.y_d, c.gates_d, self.partial, c.out)
        return m.moe_status(c.ws)


def _check_relay_layout(oracle, rc: RelayCase, e2r=None):
    c, w = rc.case, rc.case.w
    prob, keep = oracle_problem(oracle, w, c.src_off, e2r)
    ref = oracle.layout(prob, c.ids)
    rp = oracle.relay_layout(prob, c.ids)
    got_rp = rc.rel.relay_pos.cpu().numpy()
    assert np.array_equal(got_rp, rp), "relay_pos differs"
    n = int((rp >= 0).sum())
    toks, hosts = np.nonzero(rp >= 0)
    src = rc.rel.relay_src.cpu().numpy()
    assert np.array_equal(src[rp[toks, hosts]], toks), "relay_src is not the inverse of relay_pos"
    host = _host_of(w, c.ids, e2r)
    want_sr = np.take_along_axis(rp, host, axis=1)
    assert np.array_equal(rc.rel.slot_relay.cpu().numpy(), want_sr), "slot_relay differs"
    return prob, ref, rp, n


def _check_moves(oracle, rc: RelayCase, prob, ref, rp, n):
    c, w = rc.case, rc.case.w
    if w.dtype == "fp8":
        relay, rs, recv, rcs = oracle.relay_dispatch(prob, c.ids, ref["pos"], rp, c.xq, c.xs)
        assert np.array_equal(rc.relay_rows[:n].cpu().numpy(), relay)
        assert np.array_equal(rc.relay_s[:n].cpu().numpy().view(np.uint32), rs.view(np.uint32))
        assert np.array_equal(c.recv.cpu().numpy(), recv)
        assert np.array_equal(c.recv_s.cpu().numpy().view(np.uint32), rcs.view(np.uint32))
    else:
        relay, _, recv, _ = oracle.relay_dispatch(prob, c.ids, ref["pos"], rp, c.x)
        assert np.array_equal(dev_to_bits(rc.relay_rows[:n]), relay)
        assert np.array_equal(dev_to_bits(c.recv), recv)
    y = c.y_host if c.y_host is not None else dev_to_bits(c.y_d)
    partial, out = oracle.relay_combine(prob, c.ids, ref["pos"], rp, y, c.gates)
    assert np.array_equal(dev_to_bits(rc.partial[:n]), partial), "partials differ"
    assert np.array_equal(dev_to_bits(c.out), out), "relay combine differs"


def _relay_check(oracle, case: Case, e2r=None):
    rc = RelayCase(case)
    rc.poison()
    code, bits = rc.run()
    assert code == 0 and bits == 0, (code, bits)
    prob, ref, rp, n = _check_relay_layout(oracle, rc, e2r)
    _check_moves(oracle, rc, prob, ref, rp, n)
    return rc


def _small(**kw):
    base = dict(name="relay", T=300, h=256, k=4, E=16, R=8, P=2, R_src=1)
    base.update(kw)
    return mw.Workload(**base)


RELAY_CASES = [
    mw.scaled(mw.WORKLOADS["tiny"]),
    mw.scaled(mw.WORKLOADS["decode-EP32-r8"], T=1000, R_src=8),       # 4 hosts, ragged tile
    mw.scaled(mw.WORKLOADS["decode-EP32-s1.1"], T=640, R_src=20),     # skewed routing
    mw.scaled(mw.WORKLOADS["prefill"], T=1000),                       # 2 hosts
    mw.scaled(mw.WORKLOADS["prefill-fp8"], T=900),                    # fp8 rows + scales
    _small(T=1),
    _small(T=257, h=8),                                               # smallest bf16 row
    _small(T=700, k=8, E=64, R=8, P=8),                               # one host: partial = flat combine
    _small(T=400, k=8, E=64, R=64, P=1),                              # one rank per host
    _small(T=333, h=1024, k=8, E=256, R=128, P=2, dtype="fp8"),       # 64 hosts (two host words per lane)
    _small(T=200, k=16, E=64, R=32, P=2),                             # k > 8: the LSU combine, 16 hosts
    _small(T=96, k=32, E=64, R=64, P=1),                              # largest top-k, 32+ hosts per token
    _small(T=128, k=32, E=1024, R=1024, P=16, R_src=64),             # the largest E, R, hosts and top-k together
    _small(T=5000, h=64, k=2, E=8, R=4, P=2),                         # several relay tiles, ragged tail
    _small(T=24, h=76800, dtype="fp8"),                               # 600 scale groups: too many to stage, plain copies
    _small(T=70000, h=64, k=2, E=8, R=4, P=2),                        # 512-token relay tiles
]


@pytest.mark.parametrize("w", RELAY_CASES,
                         ids=lambda w: f"{w.name}_T{w.T}_h{w.h}_k{w.k}_E{w.E}_R{w.R}_P{w.P}_{w.dtype}")
def test_relay_parity(dev, oracle_mod, w):
    _relay_check(oracle_mod, Case(w, dev, y_on_device=False))


def test_relay_one_host_equals_flat(dev, oracle_mod):
    """With every rank on one host the relay combine equals moe_combine bit
    for bit and the relay dispatch equals moe_dispatch."""
    import torch
    w = _small(T=640, h=512, k=6, E=48, R=8, P=8)
    case = Case(w, dev, y_on_device=False)
    rc = _relay_check(oracle_mod, case)
    out_relay, recv_relay = case.out.clone(), case.recv.clone()
    case.run(layout=False, stats=False)
    assert torch.equal(case.out.view(torch.int16), out_relay.view(torch.int16))
    assert torch.equal(case.recv.view(torch.int16), recv_relay.view(torch.int16))


def test_relay_custom_placement(dev, oracle_mod):
    """Random expert_to_rank with empty ranks (and so possibly empty hosts)."""
    w = _small(T=700, k=4, E=48, R=12, P=3, R_src=4)
    rng = np.random.default_rng(11)
    e2r = rng.integers(0, w.R - 3, size=w.E).astype(np.int32)   # host 3 (ranks 9..11) owns nothing
    _relay_check(oracle_mod, Case(w, dev, expert_to_rank=e2r, y_on_device=False), e2r=e2r)


def test_relay_empty_batch(dev):
    import combine_moe_layout_04_gb300 as moe
    w = _small(T=0)
    case = Case(w, dev, ids=np.zeros((0, w.k), np.int32), gates=np.zeros((0, w.k), np.float32),
                y_on_device=False)
    rc = RelayCase(case)
    code, bits = rc.run()
    assert code == moe.MOE_OK and bits == 0


def test_relay_capacity_too_small(dev, oracle_mod):
    """A relay capacity below what the layout needs: the status word reports
    it, the positions are still right, relay rows inside the capacity are
    right and nothing is written past it (the buffers are allocated larger
    and their tail must keep its poison)."""
    import torch
    import combine_moe_layout_04_gb300 as moe
    w = _small(T=500, k=4, E=16, R=8, P=2)
    case = Case(w, dev, y_on_device=False)
    rc = RelayCase(case, capacity=100, alloc_rows=400)
    rc.poison()
    code, bits = rc.run()
    assert code == moe.MOE_ERR_CAPACITY and (bits & moe.MOE_STATUS_RELAY_CAPACITY)
    prob, keep = oracle_problem(oracle_mod, w)
    rp = oracle_mod.relay_layout(prob, case.ids)
    assert int((rp >= 0).sum()) > 100
    assert np.array_equal(rc.rel.relay_pos.cpu().numpy(), rp)
    assert torch.all(rc.rel.relay_src[100:] == -9)
    assert torch.all(rc.relay_rows[100:].view(torch.uint8) == 0xEE)
    assert torch.all(rc.partial[100:].view(torch.uint8) == 0xEE)
    toks, hosts = np.nonzero((rp >= 0) & (rp < 100))
    assert np.array_equal(dev_to_bits(rc.relay_rows[:100])[rp[toks, hosts]], case.x[toks])


@pytest.mark.parametrize("name", ["decode-EP32-r8", "prefill-fp8"])
def test_relay_full_size(dev, oracle_mod, name):
    """Full workload sizes: relay positions in full; every relay and receive
    row compared on the device with the row the positions name; combine on
    sampled tokens, each against the oracle run on those tokens alone (a
    token's partials and sum depend on its own slots only)."""
    import torch
    w = mw.WORKLOADS[name]
    case = Case(w, dev, y_on_device=True)
    rc = RelayCase(case)
    rc.poison()
    code, bits = rc.run()
    assert code == 0 and bits == 0
    prob, ref, rp, n = _check_relay_layout(oracle_mod, rc)
    toks, hosts = np.nonzero(rp >= 0)
    order = np.argsort(rp[toks, hosts])
    relay_tok = torch.from_numpy(toks[order].astype(np.int64)).to(dev)
    assert torch.equal(rc.relay_rows[:n].view(torch.uint8), case.x_d.view(torch.uint8).index_select(0, relay_tok))
    src_tok = torch.from_numpy((ref["recv_src"] // w.k).astype(np.int64)).to(dev)
    assert torch.equal(case.recv.view(torch.uint8), case.x_d.view(torch.uint8).index_select(0, src_tok))
    if rc.relay_s is not None:
        assert torch.equal(rc.relay_s[:n].view(torch.int32), case.xs_d.view(torch.int32).index_select(0, relay_tok))
        assert torch.equal(case.recv_s.view(torch.int32), case.xs_d.view(torch.int32).index_select(0, src_tok))
    # sampled tokens through the oracle, one sub-problem
    sel = np.sort(np.random.default_rng(8).choice(w.T, size=256, replace=False))
    rows = torch.from_numpy(ref["pos"][sel].reshape(-1).astype(np.int64)).to(dev)
    y_sel = dev_to_bits(case.y_d.index_select(0, rows))       # slot order of the selected tokens
    sub, keep = oracle_mod.make_problem(len(sel), w.h, w.k, w.E, w.R, w.P, 1)
    ids_sub = case.ids[sel]
    lay_sub = oracle_mod.layout(sub, ids_sub)
    rp_sub = oracle_mod.relay_layout(sub, ids_sub)
    y_sub = np.empty_like(y_sel)
    y_sub[lay_sub["pos"].reshape(-1)] = y_sel
    part_sub, out_sub = oracle_mod.relay_combine(sub, ids_sub, lay_sub["pos"], rp_sub, y_sub, case.gates[sel])
    assert np.array_equal(dev_to_bits(case.out[torch.from_numpy(sel).to(dev)]), out_sub)
    got_part = dev_to_bits(rc.partial[torch.from_numpy(rp[sel][rp[sel] >= 0].astype(np.int64)).to(dev)])
    assert np.array_equal(got_part, part_sub[rp_sub[rp_sub >= 0]])


def test_relay_layout_twice_after_one_layout(dev, oracle_mod):
    """A second relay layout after the same moe_layout gives the same rows
    (many tiles: 70000 tokens in 512-token tiles)."""
    import torch
    w = _small(T=70000, h=64, k=4, E=16, R=8, P=2)
    case = Case(w, dev, y_on_device=False)
    rc = RelayCase(case)
    m = case.moe
    m.moe_layout(case.prob, case.ids_d, case.ws, case.lay)
    m.moe_relay_layout(case.prob, case.lay, case.ws, rc.rel)
    first = rc.rel.relay_pos.clone()
    rc.rel.relay_pos.fill_(-9)
    m.moe_relay_layout(case.prob, case.lay, case.ws, rc.rel)
    code, bits = m.moe_status(case.ws)
    assert code == 0 and bits == 0
    assert torch.equal(rc.rel.relay_pos, first)
    prob, keep = oracle_problem(oracle_mod, w)
    assert np.array_equal(first.cpu().numpy(), oracle_mod.relay_layout(prob, case.ids))
