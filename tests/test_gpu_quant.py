"""Quantise-in-dispatch on the GPU vs the oracle: e4m3 codes and fp32 scales
bit-exact, at moderate sizes in full and at the full prefill-fp8 size on
sampled tokens."""
import numpy as np
import pytest

import moe_workloads as mw
from harness import bf16_to_dev, oracle_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    import __graft_entry__ as ge
    ge.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _run(w, dev):
    import torch
    import combine_moe_layout_04_gb300 as moe
    prob = moe.Problem(w.T, w.h, w.k, w.E, w.R, w.P, w.R_src, moe.MOE_DTYPE_FP8_E4M3)
    lay = moe.Layout(prob, dev)
    ws = moe.alloc_workspace(prob, dev)
    ids = mw.gen_ids(w)
    x = mw.gen_x_bf16(w)
    recv = torch.full((w.slots, w.h), 0xAB, dtype=torch.uint8, device=dev)
    rs = torch.full((w.slots, w.h // 128), -1.0, dtype=torch.float32, device=dev)
    moe.moe_layout(prob, torch.from_numpy(ids).to(dev), ws, lay)
    moe.moe_dispatch_quant(prob, lay, bf16_to_dev(x, dev), recv, rs)
    rc, bits = moe.moe_status(ws)
    assert rc == moe.MOE_OK and bits == 0
    return ids, x, recv, rs


@pytest.mark.parametrize("w", [
    mw.Workload("q1", T=300, h=512, k=4, E=16, R=4, P=2, R_src=1, dtype="fp8"),
    mw.Workload("q2", T=129, h=128, k=1, E=8, R=4, P=2, R_src=1, dtype="fp8"),    # one scale group
    mw.Workload("q3", T=77, h=640, k=3, E=12, R=6, P=3, R_src=1, dtype="fp8"),    # partial 512-column chunk
    mw.Workload("q4", T=64, h=256, k=32, E=64, R=8, P=2, R_src=1, dtype="fp8"),   # largest top-k
    mw.scaled(mw.WORKLOADS["prefill-fp8-quant"], T=500),
], ids=lambda w: f"{w.name}_T{w.T}_h{w.h}_k{w.k}")
def test_quantize_dispatch_parity(dev, oracle_mod, w):
    ids, x, recv, rs = _run(w, dev)
    prob, keep = oracle_problem(oracle_mod, w)
    lay = oracle_mod.layout(prob, ids)
    codes, scales = oracle_mod.quantize_dispatch(prob, lay["pos"], x)
    assert np.array_equal(recv.cpu().numpy(), codes)
    assert np.array_equal(rs.cpu().numpy().view(np.uint32), scales.view(np.uint32))


def test_quantize_dispatch_full_size_sampled(dev, oracle_mod):
    """prefill-fp8-quant at full size: every receive row holds its token's codes
    (checked on the device), and 256 sampled tokens match the oracle."""
    import torch
    w = mw.WORKLOADS["prefill-fp8-quant"]
    ids, x, recv, rs = _run(w, dev)
    prob, keep = oracle_problem(oracle_mod, w)
    lay = oracle_mod.layout(prob, ids)
    pos = torch.from_numpy(lay["pos"].astype(np.int64)).to(dev)
    first = recv.index_select(0, pos[:, 0])
    for j in range(1, w.k):
        assert torch.equal(recv.index_select(0, pos[:, j]), first)
    toks = np.sort(np.random.default_rng(9).choice(w.T, 256, replace=False))
    sub, keep2 = oracle_mod.make_problem(len(toks), w.h, 1, 1, 1, 1, 1, 1, 128)
    codes, scales = oracle_mod.quantize_dispatch(sub, np.arange(len(toks), dtype=np.int32)[:, None], x[toks])
    rows = torch.from_numpy(lay["pos"][toks, 0].astype(np.int64)).to(dev)
    assert np.array_equal(recv.index_select(0, rows).cpu().numpy(), codes)
    assert np.array_equal(rs.index_select(0, rows).cpu().numpy().view(np.uint32), scales.view(np.uint32))
