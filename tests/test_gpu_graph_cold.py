"""A process whose very first library calls are made while a CUDA graph is
being captured: the launch-shape lookups the library makes on first use
(shared-memory opt-in, occupancy, SM count) must not break the capture, and
the replayed step must equal the same calls issued eagerly afterwards.  Runs
in a child process so that nothing is looked up before the capture."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import torch
import combine_moe_layout_04_gb300 as moe
import moe_workloads as mw
from harness import Case
dev = torch.device("cuda:0")
for name, changes in (("decode-EP32-r8", dict(T=1024, R_src=8)), ("prefill-fp8", dict(T=1536))):
    w = mw.scaled(mw.WORKLOADS[name], **changes)
    c = Case(w, dev, y_on_device=False)
    lay = moe.Layout(c.prob, dev, with_stats=True)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        s = torch.cuda.current_stream()
        moe.moe_layout(c.prob, c.ids_d, c.ws, lay, s)
        moe.moe_dispatch(c.prob, lay, c.x_d, c.xs_d, c.recv, c.recv_s, s)
        moe.moe_combine(c.prob, lay, c.y_d, c.gates_d, c.out, s)
    c.poison()
    g.replay()
    torch.cuda.synchronize()
    replayed = [t.clone() for t in (lay.pos, lay.stats, c.recv, c.out)]
    c.poison()
    moe.moe_layout(c.prob, c.ids_d, c.ws, lay)
    moe.moe_dispatch(c.prob, lay, c.x_d, c.xs_d, c.recv, c.recv_s)
    moe.moe_combine(c.prob, lay, c.y_d, c.gates_d, c.out)
    code, bits = moe.moe_status(c.ws)
    assert code == 0 and bits == 0, (code, bits)
    for a, b in zip(replayed, (lay.pos, lay.stats, c.recv, c.out)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), name
    del g
print("cold capture ok")
"""


def test_first_calls_inside_a_graph_capture():
    import __graft_entry__ as ge
    ge.build()
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "cold capture ok" in r.stdout
