"""Benchmark: one MoE layer's layout + stats + dispatch + combine on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--tokens T] [--impl ours|reference]

A step is one pass of the whole hot path over one batch: moe_layout (which
also writes the statistics record; --stats beside makes it with
moe_stats_device on a second stream beside the row movers instead),
moe_dispatch and moe_combine, inputs resident in HBM.  The timed loop replays a CUDA graph of the step's calls
once per step; a second loop issues the calls one by one with events
between the kernels for the per-kernel breakdown.
The headline value is the effective HBM bandwidth of dispatch + combine: their
algorithmic bytes (read each token row once and write k copies; read k rows
and write one) divided by the whole step's time, layout and stats included.
The default workload is the largest one, "prefill-fp8" (T=16384, h=7168,
top-8 of 128 experts, fp8 e4m3 rows with fp32 scales, Zipf s=1.0 routing).

--impl reference times the single-threaded CPU oracle on a bounded sample of
the same workload (the slow plain definition, as it stands).
With N > 1 (torchrun), every rank runs an independent replica: the path has
no exchange step on one GPU, so the job total is N x the per-rank work.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dispatch+combine µs and effective HBM GB/s (fraction of GB300 peak) per layer"
FALLBACK_HBM_GBS = 6800.0
# kernels a step launches: layout (one cooperative kernel), dispatch, combine,
# and the statistics kernel when the record is made beside the movers
KERNELS_PER_STEP = {"inline": 3, "beside": 4}


def algorithmic_bytes(w, tokens=None):
    """Dispatch reads each row once and writes k copies (payload + fp8 scales);
    combine reads k bf16 rows and writes one."""
    T = w.T if tokens is None else tokens
    rho = w.h + 4 * (w.h // w.scale_group) if w.dtype == "fp8" else 2 * w.h
    # quantise-in-dispatch reads bf16 rows and writes k fp8 rows + scales
    dispatch = T * (2 * w.h + w.k * rho) if w.quantize else T * rho * (1 + w.k)
    combine = T * w.k * 2 * w.h + T * 2 * w.h
    return dispatch, combine


def read_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            stack = [d]
            while stack:
                cur = stack.pop()
                if isinstance(cur, dict):
                    for k, v in cur.items():
                        if k == "hbm_gbs" and isinstance(v, (int, float)):
                            return float(v), "measured"
                        stack.append(v)
        except (OSError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


# The sources a mover's DRAM traffic depends on: its kernels and the shared
# device helpers.  A traffic figure taken on other sources is not reported.
MOVER_SOURCES = ("moe_move_kernels.cu", "moe_internal.cuh")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "combine_moe_layout_04_gb300", "csrc")
    for n in MOVER_SOURCES:
        h.update(open(os.path.join(csrc, n), "rb").read())
    return h.hexdigest()[:16]


def read_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (profiles/dram_traffic.txt lines:
    <kernel> <workload> <bytes_per_launch> <source hash>)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    cur = kernel_source_hash()
    for line in open(path):
        f = line.split()
        if len(f) == 4 and f[0] == kernel and f[1] == workload and f[3] == cur:
            return int(float(f[2]))
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.rows = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [r for t, r in self.rows if t0 <= t <= t1]
        note = "sampled during the timed region"
        if not inside and self.rows:
            near = min(self.rows, key=lambda tr: min(abs(tr[0] - t0), abs(tr[0] - t1)))
            inside, note = [near[1]], "timed region shorter than the 200 ms sampling period: nearest sample"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        sm = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in inside for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside), "note": note}


def bind_near_gpu(dev):
    """Runs this process on the CPUs that the system lists as local to the GPU,
    so that the pinned host buffers of the end-to-end loop are allocated in the
    memory nearest it.  Returns the CPU list used, or None where it cannot be
    found."""
    import torch
    try:
        p = torch.cuda.get_device_properties(dev)
        path = f"/sys/bus/pci/devices/{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0/local_cpulist"
        text = open(path).read().strip()
        cpus = set()
        for part in text.split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        if cpus:
            os.sched_setaffinity(0, cpus)
            return text
    except (AttributeError, OSError, ValueError):
        pass
    return None


def dist_setup(backend="nccl"):
    """Rank of this replica from the torchrun environment.  Each rank works on
    its own GPU (LOCAL_RANK); the process group only carries the barrier and
    the max over ranks of the timings ("gloo" runs the same logic on CPU)."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value, world):
    """The largest value over the ranks (every rank gets it)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank, ms_max, world):
    """Whole-job throughput: every rank processed units_per_rank (bytes) in at
    most ms_max milliseconds."""
    return world * units_per_rank / (ms_max * 1e-3) / 1e9


# ----------------------------------------------------------------- oracle (CPU)

def oracle_pass(w, tokens, ids, gates, xin, y, times=None):
    """One pass of the oracle over the first `tokens` tokens of a workload;
    appends (layout + stats, dispatch, combine) seconds to `times` if given."""
    import oracle
    eb = 1 if w.dtype == "fp8" else 2
    prob, keep = oracle.make_problem(tokens, w.h, w.k, w.E, w.R, w.P, 1, eb, w.scale_group)
    t0 = time.perf_counter()
    lay = oracle.layout(prob, ids[:tokens])
    oracle.stats(prob, ids[:tokens])
    t1 = time.perf_counter()
    if w.quantize:
        oracle.quantize_dispatch(prob, lay["pos"], xin[:tokens])
    elif w.dtype == "fp8":
        oracle.dispatch(prob, lay["pos"], xin[0][:tokens], xin[1][:tokens])
    else:
        oracle.dispatch(prob, lay["pos"], xin[:tokens])
    t2 = time.perf_counter()
    oracle.combine(prob, lay["pos"], y, gates[:tokens])
    t3 = time.perf_counter()
    if times is not None:
        times.append((t1 - t0, t2 - t1, t3 - t2))


def host_cpu():
    """The host's CPU model (x86 model name, or Arm implementer and part) and
    its logical CPU count."""
    model = platform.machine()
    try:
        info = open("/proc/cpuinfo").read()
        names = [l.split(":", 1)[1].strip() for l in info.splitlines() if l.startswith("model name")]
        if names:
            model = names[0]
        else:
            impl = [l.split(":", 1)[1].strip() for l in info.splitlines() if l.startswith("CPU implementer")]
            part = [l.split(":", 1)[1].strip() for l in info.splitlines() if l.startswith("CPU part")]
            if impl and part:
                model = f"{platform.machine()} implementer {impl[0]} part {part[0]}"
    except OSError:
        pass
    return {"cpu_model": model, "nproc": os.cpu_count()}


def oracle_inputs(w, tokens):
    import moe_workloads as mw
    ids = mw.gen_ids(w)
    gates = mw.gen_gates(w)
    xin = mw.gen_x_fp8(w, rows=tokens) if (w.dtype == "fp8" and not w.quantize) else mw.gen_x_bf16(w, rows=tokens)
    y = mw.gen_y_host(w, rows=tokens * w.k)
    return ids, gates, xin, y


def cpu_baseline(w, seconds=10.0):
    """The oracle as it stands, single-threaded, on a token sample sized to run
    about `seconds`."""
    import oracle
    oracle.build()
    probe = 64
    ids, gates, xin, y = oracle_inputs(w, probe)
    t0 = time.perf_counter()
    oracle_pass(w, probe, ids, gates, xin, y)
    per_tok = (time.perf_counter() - t0) / probe
    tokens = int(max(probe, min(w.T, seconds / max(per_tok, 1e-9))))
    ids, gates, xin, y = oracle_inputs(w, tokens)
    # one warm-up pass, then the median of 5 (3 when a pass is long)
    reps = 5 if per_tok * tokens < 4.0 else 3
    oracle_pass(w, tokens, ids, gates, xin, y)
    times = []
    for _ in range(reps):
        oracle_pass(w, tokens, ids, gates, xin, y, times)
    import numpy as np
    med = np.median(np.array(times), axis=0)
    dt = float(med.sum())
    d, c = algorithmic_bytes(w, tokens)
    return {"value": round((d + c) / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {tokens} of {w.T} tokens of {w.name}: layout+stats+dispatch+combine, "
                      f"one warm-up pass and the median of {reps}, {dt:.2f} s a pass",
            "per_call_s": {"layout_stats": round(float(med[0]), 4), "dispatch": round(float(med[1]), 4),
                           "combine": round(float(med[2]), 4)},
            "host": dict(host_cpu(), threads_used=1)}


def run_reference(args, w):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    probe = 32
    ids, gates, xin, y = oracle_inputs(w, probe)
    t0 = time.perf_counter()
    oracle_pass(w, probe, ids, gates, xin, y)
    per_tok = (time.perf_counter() - t0) / probe
    budget = 90.0  # seconds for the whole warm-up + timed run
    tokens = int(max(8, min(w.T, budget / (args.steps + args.warmup) / max(per_tok, 1e-9))))
    ids, gates, xin, y = oracle_inputs(w, tokens)
    for _ in range(args.warmup):
        oracle_pass(w, tokens, ids, gates, xin, y)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_pass(w, tokens, ids, gates, xin, y)
    dt = (time.perf_counter() - t0) / args.steps
    d, c = algorithmic_bytes(w, tokens)
    value = (d + c) / dt / 1e9
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "impl": "reference",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: first {tokens} of {w.T} tokens of {w.name}"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(w):
    return {"workload": w.name, "T": w.T, "hidden": w.h, "topk": w.k, "experts": w.E, "ranks": w.R,
            "hosts": w.H, "src_ranks": w.R_src,
            "x": ("bf16, quantised to fp8 e4m3 + fp32 scale per 128 columns inside dispatch" if w.quantize
                  else "fp8 e4m3 + fp32 scale per 128 columns" if w.dtype == "fp8" else "bf16"),
            "y_out": "bf16", "routing": w.routing + (f" s={w.zipf_s}" if w.routing == "zipf" else ""),
            "l2": "inputs larger than L2: each step streams >1 GB (y, recv) through the 129 MB L2, "
                  "which evicts the previous step's x"}


# ----------------------------------------------------------------- GPU arm

def reference_rates(dev, nbytes, reps=5):
    """HBM rate of a plain library kernel on the same GPU in the same run, as a
    reference for the row movers: torch's copy (one read and one write per
    byte, the way the measured peak is taken) over `nbytes`, timed with CUDA
    events (median of `reps` after two warm-ups).  torch's fill and zero_ write
    at well under the copy rate on GB300 (3.9 TB/s), so they are no write-only
    reference."""
    import statistics as st
    import torch
    buf = torch.empty(2 * nbytes, dtype=torch.uint8, device=dev)
    a, b = buf[:nbytes], buf[nbytes:]
    a.fill_(7)
    times = []
    for i in range(reps + 2):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_(a)
        e1.record()
        torch.cuda.synchronize(dev)
        if i >= 2:
            times.append(e0.elapsed_time(e1) * 1e3)
    us = st.median(times)
    del buf
    return {"copy_read_write": {"us": round(us, 2), "gbs": round(2 * nbytes / (us * 1e-6) / 1e9, 1)},
            "bytes": nbytes}


def relay_bytes(w, n_relay):
    """Mode 2 relay on one buffer: dispatch reads each token row, writes and
    reads back its relay rows, writes k receive rows; combine reads k expert
    rows, writes and reads back the per-host partials, writes one row."""
    rho = w.h + 4 * (w.h // w.scale_group) if w.dtype == "fp8" else 2 * w.h
    dispatch = rho * (w.T + 2 * n_relay + w.T * w.k)
    combine = 2 * w.h * (w.T * w.k + 2 * n_relay + w.T)
    return dispatch, combine


def peo_bytes(w, ids, group, G):
    """Per-expert-group calls: group g's dispatch reads a token row once if the
    token has a slot in g and writes its slots of g; the combine chain reads
    the k expert rows once, writes the fp32 accumulator after the first group,
    reads and writes it in every middle group where the token has a slot, and
    reads it once more before writing the bf16 row."""
    import numpy as np
    rho = w.h + 4 * (w.h // w.scale_group) if w.dtype == "fp8" else 2 * w.h
    tg = group[ids]                                              # [T, k]
    has = np.stack([(tg == g).any(axis=1) for g in range(G)])    # [G, T]
    dispatch = rho * (int(has.sum()) + w.T * w.k)
    if G == 1:  # one group: a plain combine, no fp32 chain
        return dispatch, 2 * w.h * w.T * w.k + 2 * w.h * w.T
    mids = int(has[1:G - 1].sum()) if G > 2 else 0
    combine = 2 * w.h * w.T * w.k + 4 * w.h * w.T + 8 * w.h * mids + (4 * w.h + 2 * w.h) * w.T
    return dispatch, combine


def peo_measure(args, w, moe, prob, lay, ws, ids, ids_d, x_d, xs_d, recv, recv_s, y_d, gates_d, out,
                stream, world, dev, G):
    """Times the per-expert-group calls (G groups), run back to back on one
    stream and in the overlap schedule (dispatches on one stream, each group's
    combine on a second stream once its dispatch is done, so a combine runs
    beside the next group's dispatch).  The expert computation between a
    group's dispatch and combine is the identity (bf16) or the fixed y buffer
    (fp8); reported beside the flat step, not part of it."""
    import numpy as np
    import torch
    if w.quantize:
        return None
    grp = torch.empty(w.E, dtype=torch.int32, device=dev)
    moe.moe_expert_groups(prob, G, grp, stream)
    acc = torch.empty((w.T, w.h), dtype=torch.float32, device=dev)
    moe.moe_layout(prob, ids_d, ws, lay, stream)
    side = torch.cuda.Stream(dev)

    def serial():
        for g in range(G):
            moe.moe_dispatch_group(prob, lay, ids_d, grp, g, x_d, xs_d, recv, recv_s, stream)
            moe.moe_combine_group(prob, lay, ids_d, grp, g, G, y_d, gates_d, acc, out, stream)

    def overlapped():
        side.wait_stream(stream)
        for g in range(G):
            moe.moe_dispatch_group(prob, lay, ids_d, grp, g, x_d, xs_d, recv, recv_s, stream)
            ev = torch.cuda.Event()
            ev.record(stream)
            side.wait_event(ev)
            moe.moe_combine_group(prob, lay, ids_d, grp, g, G, y_d, gates_d, acc, out, side)
        stream.wait_stream(side)

    res = {"groups": G}
    n = min(args.steps, 200)
    # one serial pass with an event around every call: where the time goes
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * G + 1)]
    for _ in range(3):
        evs[0].record(stream)
        for g in range(G):
            moe.moe_dispatch_group(prob, lay, ids_d, grp, g, x_d, xs_d, recv, recv_s, stream)
            evs[2 * g + 1].record(stream)
            moe.moe_combine_group(prob, lay, ids_d, grp, g, G, y_d, gates_d, acc, out, stream)
            evs[2 * g + 2].record(stream)
        torch.cuda.synchronize(dev)
    res["dispatch_us_per_group"] = [round(evs[2 * g].elapsed_time(evs[2 * g + 1]) * 1e3, 1) for g in range(G)]
    res["combine_us_per_group"] = [round(evs[2 * g + 1].elapsed_time(evs[2 * g + 2]) * 1e3, 1) for g in range(G)]
    for name, fn in (("serial", serial), ("overlap", overlapped)):
        for _ in range(max(3, args.warmup)):
            fn()
        barrier(world)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        res[name + "_us"] = round(max_over_ranks(e0.elapsed_time(e1), world) * 1e3 / n, 2)
    rc, bits = moe.moe_status(ws, stream)
    if rc != moe.MOE_OK:
        raise RuntimeError(f"group device status {bits:#x}")
    grp_h = grp.cpu().numpy()
    d_bytes, c_bytes = peo_bytes(w, ids, grp_h, G)
    # routing skew makes the groups unequal: their shares of the slots
    res["slot_share"] = [round(float(v), 3) for v in np.bincount(grp_h[ids].ravel(), minlength=G) / ids.size]
    res["steps"] = n
    res["algorithmic_bytes"] = {"dispatch": d_bytes, "combine": c_bytes}
    res["overlap_gbs"] = round((d_bytes + c_bytes) / (res["overlap_us"] * 1e-6) / 1e9, 1)
    return res


def relay_measure(args, w, moe, prob, lay, ws, ids_d, x_d, xs_d, recv, recv_s, y_d, gates_d, out,
                  stream, world, dev):
    """Times the Mode 2 relay calls (relay layout, two-hop dispatch, two-hop
    combine) after a flat layout of the same batch; reported beside the flat
    step, not part of it.  Quantise-in-dispatch has no relay form."""
    import torch
    if w.quantize:
        return None
    rel = moe.Relay(prob, dev)
    moe.moe_layout(prob, ids_d, ws, lay, stream)
    n_relay = int(lay.host_offset[-1].item())
    row_dtype = x_d.dtype
    relay_rows = torch.empty((n_relay, w.h), dtype=row_dtype, device=dev)
    relay_s = (torch.empty((n_relay, w.h // w.scale_group), dtype=torch.float32, device=dev)
               if xs_d is not None else None)
    partial = torch.empty((n_relay, w.h), dtype=torch.bfloat16, device=dev)
    rel.capacity = n_relay

    def relay_step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        moe.moe_relay_layout(prob, lay, ws, rel, stream)
        if ev is not None:
            ev[1].record(stream)
        moe.moe_dispatch_relay(prob, lay, rel, x_d, xs_d, relay_rows, relay_s, recv, recv_s, stream)
        if ev is not None:
            ev[2].record(stream)
        moe.moe_combine_relay(prob, lay, rel, y_d, gates_d, partial, out, stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(max(3, args.warmup)):
        relay_step()
    rc, bits = moe.moe_status(ws, stream)
    if rc != moe.MOE_OK:
        raise RuntimeError(f"relay device status {bits:#x}")
    n = min(args.steps, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    barrier(world)
    torch.cuda.synchronize(dev)
    for i in range(n):
        relay_step(evs[i])
    torch.cuda.synchronize(dev)
    import numpy as np
    per = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in evs]) * 1e3  # µs
    lay_us, d_us, c_us = [max_over_ranks(v, world) for v in per.mean(axis=0).tolist()]
    d_bytes, c_bytes = relay_bytes(w, n_relay)
    return {"relay_rows": n_relay, "steps": n, "relay_layout_us": round(lay_us, 2),
            "dispatch_us": round(d_us, 2), "combine_us": round(c_us, 2),
            "algorithmic_bytes": {"dispatch": d_bytes, "combine": c_bytes},
            "dispatch_gbs": round(d_bytes / (d_us * 1e-6) / 1e9, 1),
            "combine_gbs": round(c_bytes / (c_us * 1e-6) / 1e9, 1),
            "gbs": round((d_bytes + c_bytes) / ((d_us + c_us) * 1e-6) / 1e9, 1)}


def run_ours(args, w):
    import numpy as np
    import torch

    import __graft_entry__ as ge
    world, rank, local = dist_setup()
    ge.build()
    import combine_moe_layout_04_gb300 as moe
    import moe_workloads as mw

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    host_cpus = bind_near_gpu(dev)
    fp8 = w.dtype == "fp8"
    ids = mw.gen_ids(w)
    gates = mw.gen_gates(w)
    # Launch shapes: the library's defaults unless MOE_* variables set some
    # (moe_tuning; MOE_DISPATCH_KIND=bulk, MOE_DISPATCH_WARPS=6, ...).
    tuning = moe.Tuning.from_env()
    prob = moe.Problem(w.T, w.h, w.k, w.E, w.R, w.P, w.R_src,
                       moe.MOE_DTYPE_FP8_E4M3 if fp8 else moe.MOE_DTYPE_BF16, tuning=tuning)
    # The layout leaves the statistics record to moe_stats_device, which runs
    # on a second stream beside dispatch and combine (the layout kernel then
    # ends when the positions the dispatch needs are written).
    beside = args.stats == "beside"
    lay = moe.Layout(prob, dev, with_stats=not beside)
    ws = moe.alloc_workspace(prob, dev)
    stats = lay.stats if not beside else torch.empty(moe.moe_stats_words(prob), dtype=torch.int64, device=dev)
    side = torch.cuda.Stream(dev)
    ids_d = torch.from_numpy(ids).to(dev)
    gates_d = torch.from_numpy(gates).to(dev)
    if fp8 and w.quantize:
        x_d = torch.from_numpy(mw.gen_x_bf16(w).view(np.int16)).to(dev).view(torch.bfloat16)
        xs_d = None
        recv = torch.empty((w.slots, w.h), dtype=torch.uint8, device=dev)
        recv_s = torch.empty((w.slots, w.h // w.scale_group), dtype=torch.float32, device=dev)
    elif fp8:
        xq, xs = mw.gen_x_fp8(w)
        x_d, xs_d = torch.from_numpy(xq).to(dev), torch.from_numpy(xs).to(dev)
        recv = torch.empty((w.slots, w.h), dtype=torch.uint8, device=dev)
        recv_s = torch.empty((w.slots, w.h // w.scale_group), dtype=torch.float32, device=dev)
    else:
        x_d = torch.from_numpy(mw.gen_x_bf16(w).view(np.int16)).to(dev).view(torch.bfloat16)
        xs_d, recv_s = None, None
        recv = torch.empty((w.slots, w.h), dtype=torch.bfloat16, device=dev)
    # Expert outputs: a separate bf16 buffer for fp8 dispatch; for bf16 the
    # experts are identities and combine reads the receive buffer.
    y_d = mw.gen_y_device(w, dev) if fp8 else recv
    out = torch.empty((w.T, w.h), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    # A workload whose routing is re-drawn every step (the skew sweep) cycles
    # through all its steps' ids and gates.
    n_route = max(1, w.steps)
    ids_bank = [ids_d] + [torch.from_numpy(mw.gen_ids(w, step=j)).to(dev) for j in range(1, n_route)]
    gates_bank = [gates_d] + [torch.from_numpy(mw.gen_gates(w, step=j)).to(dev) for j in range(1, n_route)]

    def step(ev=None, s=stream, j=0):
        # Events bracket each call on the main stream: before the layout,
        # before and after dispatch, after combine.  The statistics record is
        # made on the side stream, forked after the layout and joined at the
        # end of the step.
        if ev is not None:
            ev[0].record(s)
        moe.moe_layout(prob, ids_bank[j], ws, lay, s)
        if beside:
            side.wait_stream(s)
            moe.moe_stats_device(prob, ws, stats, side)
        if ev is not None:
            ev[1].record(s)
        if w.quantize:
            moe.moe_dispatch_quant(prob, lay, x_d, recv, recv_s, s)
        else:
            moe.moe_dispatch(prob, lay, x_d, xs_d, recv, recv_s, s)
        if ev is not None:
            ev[2].record(s)
        moe.moe_combine(prob, lay, y_d, gates_bank[j], out, s)
        if ev is not None:
            ev[3].record(s)
        if beside:
            s.wait_stream(side)

    for i in range(args.warmup):
        step(j=i % n_route)
    rc, bits = moe.moe_status(ws, stream)
    if rc != moe.MOE_OK:
        raise RuntimeError(f"device status {bits:#x}")

    # The step as a CUDA graph: the three calls (memset node, cooperative
    # layout kernel, dispatch, combine) captured once and replayed once per
    # step -- the same launches without the host's launch gaps.  The calls
    # allocate nothing and never synchronise, so they capture as they are.
    graphs = []
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        for j in range(n_route):  # one graph per routing of the cycle
            g = torch.cuda.CUDAGraph()
            g.capture_begin()
            step(s=cap, j=j)
            g.capture_end()
            graphs.append(g)
    stream.wait_stream(cap)
    for i in range(args.warmup):
        graphs[i % n_route].replay()
    rc, bits = moe.moe_status(ws, stream)
    if rc != moe.MOE_OK:
        raise RuntimeError(f"device status {bits:#x} after graph replays")
    out_graph = out.clone()  # the replayed step must give what the calls give
    j_graph = (args.warmup - 1) % n_route

    sampler = ClockSampler(local)
    time.sleep(0.5)
    barrier(world)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    h0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        graphs[i % n_route].replay()
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    h1 = time.time()
    time.sleep(0.3)
    sampler.stop()
    ms_step = max_over_ranks(start.elapsed_time(end), world) / args.steps

    # Per-call breakdown, warm: the same steps issued one call at a time, back
    # to back, with events before the layout, between the calls and after the
    # combine.  Each call starts with what the previous one left in L2 (for
    # bf16, the combine reads the receive rows the dispatch has just written).
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for i in range(args.steps):
        step(evs[i], j=i % n_route)
    p1.record(stream)
    torch.cuda.synchronize(dev)
    ms_step_eager = max_over_ranks(p0.elapsed_time(p1), world) / args.steps
    per = np.array([[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in evs]) * 1e3  # µs
    layout_us, dispatch_us, combine_us = [max_over_ranks(v, world) for v in per.mean(axis=0).tolist()]
    pct = {name: [round(float(v), 2) for v in np.percentile(per[:, i], [10, 50, 90])]
           for i, name in enumerate(("layout", "dispatch", "combine"))}
    layout_stats_us = ms_step_eager * 1e3 - dispatch_us - combine_us

    # Per-call breakdown, cold: before every call, outside its event pair, a
    # write of twice the L2 size evicts whatever the previous call left there.
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (129 << 20)
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    n_cold = min(args.steps, 200)
    cold_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(n_cold)]
    calls = (lambda s, j: moe.moe_layout(prob, ids_bank[j], ws, lay, s),
             lambda s, j: moe.moe_stats_device(prob, ws, stats, s),
             (lambda s, j: moe.moe_dispatch_quant(prob, lay, x_d, recv, recv_s, s)) if w.quantize else
             (lambda s, j: moe.moe_dispatch(prob, lay, x_d, xs_d, recv, recv_s, s)),
             lambda s, j: moe.moe_combine(prob, lay, y_d, gates_bank[j], out, s))
    names = ("layout", "stats", "dispatch", "combine")
    barrier(world)
    torch.cuda.synchronize(dev)
    for i in range(n_cold):
        for c, call in enumerate(calls):
            flush.fill_(i & 0xFF)
            cold_evs[i][2 * c].record(stream)
            call(stream, i % n_route)
            cold_evs[i][2 * c + 1].record(stream)
    torch.cuda.synchronize(dev)
    cold = np.array([[e[2 * c].elapsed_time(e[2 * c + 1]) for c in range(len(calls))] for e in cold_evs]) * 1e3
    cold_mean = [max_over_ranks(v, world) for v in cold.mean(axis=0).tolist()]
    del flush
    per_call = {
        "warm": {name: {"mean": round(layout_us if i == 0 else dispatch_us if i == 1 else combine_us, 2),
                        "p10_p50_p90": pct[name]} for i, name in enumerate(("layout", "dispatch", "combine"))},
        "cold": {name: {"mean": round(cold_mean[i], 2),
                        "p10_p50_p90": [round(float(v), 2) for v in np.percentile(cold[:, i], [10, 50, 90])]}
                 for i, name in enumerate(names)},
        "warm_steps": args.steps, "cold_steps": n_cold, "l2_flush_bytes": 2 * l2,
        "note": ("warm: calls back to back ("
                 + ("the layout writes the statistics record itself" if args.stats == "inline" else
                    "the statistics record on a side stream, not timed alone")
                 + "); cold: a write of 2x L2 before each call, outside its events; "
                 "cold stats: the record made apart from the layout (moe_stats_device)"),
    }
    step(j=j_graph)
    if not torch.equal(out.view(torch.int16), out_graph.view(torch.int16)):
        raise RuntimeError("the replayed step and the eager calls disagree")
    del out_graph

    ratios = []
    for j in range(n_route):
        moe.moe_layout(prob, ids_bank[j], ws, lay, stream)
        moe.moe_stats_device(prob, ws, stats, stream)
        ratios.append(moe.decode_stats(prob, stats.cpu().numpy())["imbalance_ratio"])

    refs = reference_rates(dev, recv.numel() * recv.element_size())

    relay = relay_measure(args, w, moe, prob, lay, ws, ids_d, x_d, xs_d, recv, recv_s, y_d, gates_d, out,
                          stream, world, dev)

    peo = [peo_measure(args, w, moe, prob, lay, ws, ids, ids_d, x_d, xs_d, recv, recv_s, y_d, gates_d, out,
                       stream, world, dev, G) for G in (2, 4)]

    d_bytes, c_bytes = algorithmic_bytes(w)
    peak, peak_src = read_peak()
    value = job_value(d_bytes + c_bytes, ms_step, world)
    dc_us = dispatch_us + combine_us
    dc_gbs = (d_bytes + c_bytes) / (dc_us * 1e-6) / 1e9
    comb_gbs = c_bytes / (combine_us * 1e-6) / 1e9
    traffic = read_traffic("combine_kernel", w.name)

    # End to end through the public API with host buffers: every step uploads
    # its inputs from pinned host memory, runs the calls and downloads the
    # combined output and the statistics record.  Steps are pipelined over two
    # sets of device buffers and three streams (uploads, calls, downloads), as
    # a serving loop would: the host link is full duplex, so step i's download
    # runs beside step i+1's upload, and step i's kernels beside it too.
    e2e_steps = min(args.steps, 30)
    h_ids = torch.from_numpy(ids).pin_memory()
    h_gates = torch.from_numpy(gates).pin_memory()
    h_x = x_d.cpu().pin_memory()
    h_xs = xs_d.cpu().pin_memory() if xs_d is not None else None
    h_y = y_d.cpu().pin_memory() if fp8 else None
    h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h_stats = [torch.empty(stats.shape, dtype=stats.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (h_ids, h_gates, h_x, h_xs, h_y) if t is not None)
    d2h = h_out[0].numel() * h_out[0].element_size() + h_stats[0].numel() * h_stats[0].element_size()

    def device_set():
        d = {"ids": torch.empty_like(ids_d), "gates": torch.empty_like(gates_d), "x": torch.empty_like(x_d),
             "xs": torch.empty_like(xs_d) if xs_d is not None else None,
             "recv": torch.empty_like(recv), "recv_s": torch.empty_like(recv_s) if recv_s is not None else None,
             "out": torch.empty_like(out), "lay": moe.Layout(prob, dev, with_stats=True),
             "ws": moe.alloc_workspace(prob, dev)}
        d["y"] = torch.empty_like(y_d) if fp8 else d["recv"]
        return d

    # the end-to-end loop downloads each step's record: its layouts compute it inline
    sets = [{"ids": ids_d, "gates": gates_d, "x": x_d, "xs": xs_d, "recv": recv, "recv_s": recv_s, "out": out,
             "lay": moe.Layout(prob, dev, with_stats=True), "ws": ws, "y": y_d}, device_set()]
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of set b uploaded
    ev_done = [torch.cuda.Event() for _ in range(2)]  # calls on set b finished
    ev_out = [torch.cuda.Event() for _ in range(2)]   # outputs of set b downloaded

    def e2e_step(i):
        b = i % 2
        d = sets[b]
        s_up.wait_event(ev_done[b])  # the previous calls on set b have read its inputs
        with torch.cuda.stream(s_up):
            d["ids"].copy_(h_ids, non_blocking=True)
            d["gates"].copy_(h_gates, non_blocking=True)
            d["x"].copy_(h_x, non_blocking=True)
            if h_xs is not None:
                d["xs"].copy_(h_xs, non_blocking=True)
            if h_y is not None:
                d["y"].copy_(h_y, non_blocking=True)
        ev_in[b].record(s_up)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])  # set b's previous outputs are on the host
        moe.moe_layout(prob, d["ids"], d["ws"], d["lay"], stream)
        if w.quantize:
            moe.moe_dispatch_quant(prob, d["lay"], d["x"], d["recv"], d["recv_s"], stream)
        else:
            moe.moe_dispatch(prob, d["lay"], d["x"], d["xs"], d["recv"], d["recv_s"], stream)
        moe.moe_combine(prob, d["lay"], d["y"], d["gates"], d["out"], stream)
        ev_done[b].record(stream)
        s_down.wait_event(ev_done[b])
        with torch.cuda.stream(s_down):
            h_out[b].copy_(d["out"], non_blocking=True)
            h_stats[b].copy_(d["lay"].stats, non_blocking=True)
        ev_out[b].record(s_down)

    def e2e_run(n):
        s_up.wait_stream(stream)
        s_down.wait_stream(stream)
        for i in range(n):
            e2e_step(i)
        stream.wait_stream(s_up)
        stream.wait_stream(s_down)

    e2e_run(2)
    barrier(world)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e2e_steps
    if not torch.equal(sets[1]["out"].view(torch.int16), out.view(torch.int16)):
        raise RuntimeError("the two device sets of the end-to-end loop disagree")
    h_stats = h_stats[(e2e_steps - 1) % 2]
    st = moe.decode_stats(prob, h_stats.numpy())

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(w),
        "dispatch_us": round(dispatch_us, 2), "combine_us": round(combine_us, 2),
        "p10_p50_p90_us": pct, "per_call_us": per_call,
        "tokens_per_s": round(world * w.T / (ms_step * 1e-3), 1),
        "tokens_per_s_dc": round(w.T / ((dispatch_us + combine_us) * 1e-6), 1),
        "layout_stats_us": round(layout_stats_us, 2), "dc_us": round(dc_us, 2),
        "ms_per_step_eager": round(ms_step_eager, 5),
        "timed_loop": "CUDA graph of the step (one per routing of a re-drawn cycle), replayed once per step",
        "dc_gbs": round(dc_gbs, 1), "dc_frac_of_peak": round(dc_gbs / peak, 4),
        "step_frac_of_peak": round(value / world / peak, 4),
        "algorithmic_bytes": {"dispatch": d_bytes, "combine": c_bytes},
        "imbalance_ratio": round(st["imbalance_ratio"], 4),
        "routing_steps": n_route,
        "imbalance_ratio_range": [round(min(ratios), 3), round(max(ratios), 3)],
        "roofline": {"bound": "hbm", "kernel": "combine_kernel", "achieved": round(comb_gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(comb_gbs / peak, 4),
                     "traffic": traffic, "peak_source": peak_src},
        "reference_kernels": dict(refs, note="torch's own copy kernel over the receive buffer's bytes (read + "
                                             "write), same GPU and run"),
        "dispatch_gbs": round(d_bytes / (dispatch_us * 1e-6) / 1e9, 1),
        "dispatch_frac_of_peak": round(d_bytes / (dispatch_us * 1e-6) / 1e9 / peak, 4),
        "e2e": {"value": round(world * (d_bytes + c_bytes) / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "h2d_link_gbs": round(h2d / (e2e_ms * 1e-3) / 1e9, 1),
                "schedule": "two device buffer sets; uploads, calls and downloads on three streams",
                "host_cpus": host_cpus},
        "gpu_launches": KERNELS_PER_STEP[args.stats] * args.steps,
        "tuning": {k: v for k, v in tuning.as_dict().items() if v} or "library defaults",
        "stats_record": ("moe_stats_device on a second stream beside dispatch and combine" if beside
                         else "written by the layout kernel"),
        "mode2_relay": dict(relay, frac_of_peak=round(relay["gbs"] / peak, 4)) if relay else None,
        "per_expert_groups": [p for p in peo if p],
        "clocks": sampler.summary(h0, h1),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="prefill-fp8")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stats", default="inline", choices=["beside", "inline"],
                    help="statistics record of the step: written by the layout kernel itself (inline), or made "
                         "by moe_stats_device on a second stream beside the row movers (beside).  On GB300 "
                         "inline took 494.4 against 495.1 us a prefill-fp8 step, beside 180.8 against "
                         "181.8 us a decode step: the fork and join cost about what the shorter layout saves")
    ap.add_argument("--tokens", type=int, default=None,
                    help="run the workload with this many tokens instead (a smaller case of the same kernels, "
                         "for profiling); the line names it <workload>@T<tokens>")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    import moe_workloads as mw
    w = mw.WORKLOADS[args.workload]
    if args.tokens is not None:
        if args.tokens <= 0 or args.tokens % w.R_src:
            ap.error(f"--tokens must be a positive multiple of the {w.R_src} source ranks of {w.name}")
        w = mw.scaled(w, T=args.tokens, name=f"{w.name}@T{args.tokens}")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
