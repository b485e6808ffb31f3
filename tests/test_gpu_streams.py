"""Independent problems on two streams at once.

A full-size prefill-fp8 layer and a decode layer, each with its own workspace
and buffers, run layout, dispatch, combine and the Mode 2 relay calls
concurrently: the cooperative layout kernel of one beside the row movers of
the other.  Both must write exactly what they write when run alone, with no
status or fault bit set.
"""
import pytest

import moe_workloads as mw
from harness import Case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__ as ge
    ge.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


class _Layer:
    def __init__(self, name, dev):
        import torch
        self.c = Case(mw.WORKLOADS[name], dev, y_on_device=True)
        m, p = self.c.moe, self.c.prob
        self.lay = m.Layout(p, dev, with_stats=True)
        self.rel = m.Relay(p, dev)
        cap = max(self.rel.capacity, 1)
        self.relay_rows = torch.empty((cap, self.c.w.h), dtype=self.c.recv.dtype, device=dev)
        self.relay_s = (torch.empty((cap, self.c.recv_s.shape[1]), dtype=torch.float32, device=dev)
                        if self.c.recv_s is not None else None)
        self.relay_recv = torch.empty_like(self.c.recv)
        self.relay_recv_s = torch.empty_like(self.c.recv_s) if self.c.recv_s is not None else None
        self.partial = torch.empty((cap, self.c.w.h), dtype=torch.bfloat16, device=dev)
        self.relay_out = torch.empty_like(self.c.out)

    def step(self, s):
        c, m = self.c, self.c.moe
        m.moe_layout(c.prob, c.ids_d, c.ws, self.lay, s)
        m.moe_dispatch(c.prob, self.lay, c.x_d, c.xs_d, c.recv, c.recv_s, s)
        m.moe_combine(c.prob, self.lay, c.y_d, c.gates_d, c.out, s)
        m.moe_relay_layout(c.prob, self.lay, c.ws, self.rel, s)
        m.moe_dispatch_relay(c.prob, self.lay, self.rel, c.x_d, c.xs_d, self.relay_rows, self.relay_s,
                             self.relay_recv, self.relay_recv_s, s)
        m.moe_combine_relay(c.prob, self.lay, self.rel, c.y_d, c.gates_d, self.partial, self.relay_out, s)

    def outputs(self):
        import torch
        ts = [self.c.recv, self.c.recv_s, self.c.out, self.lay.pos, self.lay.recv_src, self.lay.stats,
              self.rel.relay_pos, self.rel.slot_relay, self.relay_recv, self.relay_recv_s, self.relay_out]
        return [t.reshape(-1).view(torch.uint8).clone() for t in ts if t is not None]


def test_two_problems_on_two_streams(dev):
    import torch
    layers = [_Layer("prefill-fp8", dev), _Layer("decode-EP32-r8", dev)]
    cur = torch.cuda.current_stream(dev)
    alone = []
    for L in layers:
        L.step(cur)
        assert L.c.moe.moe_status(L.c.ws, cur) == (0, 0)
        alone.append(L.outputs())

    streams = [torch.cuda.Stream(dev) for _ in layers]
    for st in streams:
        st.wait_stream(cur)
    for _ in range(5):
        for L, st in zip(layers, streams):
            L.step(st)
    for st in streams:
        cur.wait_stream(st)
    for i, L in enumerate(layers):
        assert L.c.moe.moe_status(L.c.ws, cur) == (0, 0), i
        for j, (a, b) in enumerate(zip(alone[i], L.outputs())):
            assert torch.equal(a, b), (i, j)
    assert layers[0].c.moe.moe_move_faults(cur) == 0
