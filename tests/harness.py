"""Test harness: seeded inputs on the device, the library path, oracle twins."""
from __future__ import annotations

import numpy as np

import moe_workloads as mw


def bf16_to_dev(bits: np.ndarray, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def dev_to_bits(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_problem(oracle, w: mw.Workload, src_offsets=None, expert_to_rank=None):
    eb = 1 if w.dtype == "fp8" else 2
    return oracle.make_problem(w.T, w.h, w.k, w.E, w.R, w.P, w.R_src, eb, w.scale_group,
                               expert_to_rank, src_offsets)


class Case:
    """Device inputs and outputs of one workload run through the C-ABI."""

    def __init__(self, w: mw.Workload, dev, step=0, ids=None, gates=None, y_on_device=None,
                 expert_to_rank=None, src_offsets=None):
        import torch
        import combine_moe_layout_04_gb300 as moe
        self.w, self.dev, self.moe = w, dev, moe
        self.ids = mw.gen_ids(w, step=step) if ids is None else np.ascontiguousarray(ids, np.int32)
        self.gates = mw.gen_gates(w, step=step) if gates is None else gates
        self.e2r = None if expert_to_rank is None else np.asarray(expert_to_rank, np.int32)
        self.src_off = None if src_offsets is None else np.asarray(src_offsets, np.int32)
        fp8 = w.dtype == "fp8"
        self.prob = moe.Problem(
            w.T, w.h, w.k, w.E, w.R, w.P, w.R_src,
            moe.MOE_DTYPE_FP8_E4M3 if fp8 else moe.MOE_DTYPE_BF16,
            None if self.e2r is None else torch.from_numpy(self.e2r).to(dev),
            None if self.src_off is None else torch.from_numpy(self.src_off).to(dev))
        self.lay = moe.Layout(self.prob, dev)
        self.ws = moe.alloc_workspace(self.prob, dev)
        self.stats = torch.empty(moe.moe_stats_words(self.prob), dtype=torch.int64, device=dev)
        self.ids_d = torch.from_numpy(self.ids).to(dev)
        self.gates_d = torch.from_numpy(np.ascontiguousarray(self.gates, np.float32)).to(dev)
        if fp8:
            self.xq, self.xs = mw.gen_x_fp8(w)
            self.x_d = torch.from_numpy(self.xq).to(dev)
            self.xs_d = torch.from_numpy(self.xs).to(dev)
            self.recv = torch.empty((w.slots, w.h), dtype=torch.uint8, device=dev)
            self.recv_s = torch.empty((w.slots, w.h // w.scale_group), dtype=torch.float32, device=dev)
        else:
            self.x = mw.gen_x_bf16(w)
            self.x_d = bf16_to_dev(self.x, dev)
            self.xs_d = None
            self.recv = torch.empty((w.slots, w.h), dtype=torch.bfloat16, device=dev)
            self.recv_s = None
        if y_on_device is None:
            y_on_device = w.slots * w.h > (1 << 26)
        if y_on_device:
            self.y_host = None
            self.y_d = mw.gen_y_device(w, dev)
        else:
            self.y_host = mw.gen_y_host(w)
            self.y_d = bf16_to_dev(self.y_host, dev)
        self.out = torch.empty((w.T, w.h), dtype=torch.bfloat16, device=dev)

    def poison(self):
        import torch
        self.recv.view(torch.uint8).fill_(0xFF)
        if self.recv_s is not None:
            self.recv_s.view(torch.uint8).fill_(0xFF)
        self.out.view(torch.uint8).fill_(0xFF)
        for n in ("expert_count", "expert_offset", "rank_count", "rank_offset", "host_count",
                  "host_offset", "pos", "recv_src"):
            getattr(self.lay, n).fill_(-7)
        self.lay.host_mask.fill_(0xAB)

    def run(self, layout=True, stats=True, dispatch=True, combine=True):
        m = self.moe
        if layout:
            m.moe_layout(self.prob, self.ids_d, self.ws, self.lay)
        if stats:
            m.moe_stats_device(self.prob, self.ws, self.stats)
        if dispatch:
            m.moe_dispatch(self.prob, self.lay, self.x_d, self.xs_d, self.recv, self.recv_s)
        if combine:
            m.moe_combine(self.prob, self.lay, self.y_d, self.gates_d, self.out)
        return m.moe_status(self.ws)

    def stats_host(self) -> dict:
        return self.moe.decode_stats(self.prob, self.stats.cpu().numpy())
