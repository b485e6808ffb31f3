"""The library's calls allocate nothing and never synchronise, so a caller can
capture a whole step (layout with its statistics, dispatch, combine; and the
relay and expert-group calls) in a CUDA graph and replay it.  The replayed
step must write exactly what the calls write when issued one by one."""
import numpy as np
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


def _snapshot(tensors):
    return [t.view(-1).view(__import__("torch").uint8).clone() for t in tensors]


@pytest.mark.parametrize("name,changes", [("prefill-fp8", dict(T=2048)), ("decode-EP32-r8", dict(T=1024, R_src=8))])
def test_step_graph_replay_equals_eager(dev, name, changes):
    import torch
    w = mw.scaled(mw.WORKLOADS[name], **changes)
    c = Case(w, dev, y_on_device=False)
    m = c.moe
    lay = m.Layout(c.prob, dev, with_stats=True)
    rel = m.Relay(c.prob, dev)
    cap = rel.capacity
    relay_rows = torch.empty((cap, w.h), dtype=c.recv.dtype, device=dev)
    relay_s = torch.empty((cap, w.h // 128), dtype=torch.float32, device=dev) if c.recv_s is not None else None
    partial = torch.empty((cap, w.h), dtype=torch.bfloat16, device=dev)
    grp = torch.empty(w.E, dtype=torch.int32, device=dev)
    m.moe_expert_groups(c.prob, 2, grp)
    acc = torch.empty((w.T, w.h), dtype=torch.float32, device=dev)
    out2 = torch.empty_like(c.out)
    out3 = torch.empty_like(c.out)

    def step(s):
        m.moe_layout(c.prob, c.ids_d, c.ws, lay, s)
        m.moe_dispatch(c.prob, lay, c.x_d, c.xs_d, c.recv, c.recv_s, s)
        m.moe_combine(c.prob, lay, c.y_d, c.gates_d, c.out, s)
        m.moe_relay_layout(c.prob, lay, c.ws, rel, s)
        m.moe_dispatch_relay(c.prob, lay, rel, c.x_d, c.xs_d, relay_rows, relay_s, c.recv, c.recv_s, s)
        m.moe_combine_relay(c.prob, lay, rel, c.y_d, c.gates_d, partial, out2, s)
        for g in range(2):
            m.moe_dispatch_group(c.prob, lay, c.ids_d, grp, g, c.x_d, c.xs_d, c.recv, c.recv_s, s)
            m.moe_combine_group(c.prob, lay, c.ids_d, grp, g, 2, c.y_d, c.gates_d, acc, out3, s)

    outputs = [c.out, out2, out3, lay.pos, lay.stats, rel.relay_pos, c.recv]
    cur = torch.cuda.current_stream(dev)
    step(cur)
    code, bits = m.moe_status(c.ws, cur)
    assert code == 0 and bits == 0
    eager = _snapshot(outputs)

    for t in outputs:
        t.view(-1).view(torch.uint8).fill_(0xA5)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(cur)
    with torch.cuda.stream(side):
        graph.capture_begin()
        step(side)
        graph.capture_end()
    cur.wait_stream(side)
    for _ in range(3):
        graph.replay()
    code, bits = m.moe_status(c.ws, cur)
    assert code == 0 and bits == 0
    for a, b in zip(eager, _snapshot(outputs)):
        assert torch.equal(a, b)
