"""CPU oracle for MoE token layout, statistics, dispatch and combine.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(the CUDA library in ``combine_moe_layout_04_gb300``) never does.

The arithmetic lives in ``moe_oracle.cpp`` (single-threaded C++17, plain
definitions).  This module only builds that file with g++ and marshals numpy
arrays through ctypes.  Each wrapper names the passage it follows:

* layout   -- stable receive order by (rank(e), e); counts, exclusive offsets,
              per-(token, host) mask ("Balancing and Beyond", section 3.2 relay
              and de-redundancy; section 3.4 receive buffer of batch x k rows).
* stats    -- imbalance ratio ("Balancing and Beyond", section 2 and the Terms
              list), Mode 0/1/2 copies and bytes (section 3.2, Panel 1),
              tokens x k x h x 2 B (section 1), per-rank receive counts
              ("Profiling when rank unbalance").
* dispatch -- recv[pos[t, j]] = x[t] ("Poor HybridEP performance ...",
              dispatch_with_permute).
* combine  -- gate-weighted sum of the k expert outputs in ascending slot order,
              fp32 fma, bf16 round-to-nearest-even (combine_with_unpermute).
* relay_layout / relay_dispatch / relay_combine -- Mode 2 on one buffer
              ("Balancing and Beyond", section 3.2): one relay row per (token,
              host), fan-out from it; per-host partial sums before the final
              sum.
* expert_groups / dispatch_group / combine_groups -- per-expert-group
              overlap ("Balancing and Beyond", section 3.3): the calls of one
              expert group; combine continues one fp32 chain across groups.
* swap_plan -- per-step intra-host expert swap ("Balancing and Beyond",
              section 3.1, Figure 2(b)): heaviest rank paired with lightest,
              one best exchange per pair, accepted if the pair's maximum falls
              by at least tau.
* quantize_dispatch -- bf16 -> fp8 e4m3 with an fp32 scale per 128 columns,
              done inside dispatch ("Balancing and Beyond", section 3.1, where
              the dispatch kernel converts to FP8 on its way and overlaps the
              token-count reduction with it); e4m3 from the OCP 8-bit float
              format.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_INVALID, ERR_BAD_IDS = 0, 1, 2

GLOBAL_FIELDS = (
    "T", "slots", "row_bytes", "max_expert_count", "argmax_expert",
    "min_expert_count", "max_rank_slots", "max_rank_tokens",
    "sum_mode0_copies", "sum_mode1_copies", "sum_mode2_copies",
    "max_src_mode1_copies", "max_src_mode2_copies",
    "max_recv_remote", "max_recv_relay",
    "sum_naive_bytes", "sum_mode0_bytes", "sum_mode1_bytes", "sum_mode2_bytes",
)
SRC_FIELDS = ("src_tokens", "src_copies", "src_mode0", "src_mode1", "src_mode2",
              "src_naive_bytes", "src_mode0_bytes", "src_mode1_bytes", "src_mode2_bytes")
DST_FIELDS = ("recv_slots", "recv_tokens", "recv_self", "recv_local",
              "recv_remote", "recv_relay")


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libmoe_oracle.so`` (g++, no fp contraction)."""
    with _lock:
        fresh = (os.path.exists(_LIB)
                 and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
        if force or not fresh:
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC",
                                   "-shared", "-o", tmp, _SRC])
            os.replace(tmp, _LIB)
    return _LIB


class Problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("h", ctypes.c_int32), ("k", ctypes.c_int32),
                ("E", ctypes.c_int32), ("R", ctypes.c_int32), ("P", ctypes.c_int32),
                ("R_src", ctypes.c_int32), ("elem_bytes", ctypes.c_int32),
                ("scale_group", ctypes.c_int32),
                ("expert_to_rank", ctypes.c_void_p), ("src_offsets", ctypes.c_void_p)]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        lib.oracle_layout.argtypes = [ctypes.POINTER(Problem)] + [p] * 10
        lib.oracle_layout.restype = ctypes.c_int
        lib.oracle_stats.argtypes = [ctypes.POINTER(Problem)] + [p] * 5
        lib.oracle_stats.restype = ctypes.c_int
        lib.oracle_dispatch.argtypes = [ctypes.POINTER(Problem)] + [p] * 5
        lib.oracle_dispatch.restype = None
        lib.oracle_combine.argtypes = [ctypes.POINTER(Problem)] + [p] * 4
        lib.oracle_combine.restype = None
        lib.oracle_relay_layout.argtypes = [ctypes.POINTER(Problem), p, p]
        lib.oracle_relay_layout.restype = ctypes.c_int
        lib.oracle_relay_dispatch.argtypes = [ctypes.POINTER(Problem)] + [p] * 9
        lib.oracle_relay_dispatch.restype = None
        lib.oracle_relay_combine.argtypes = [ctypes.POINTER(Problem)] + [p] * 7
        lib.oracle_relay_combine.restype = None
        lib.oracle_expert_groups.argtypes = [ctypes.POINTER(Problem), ctypes.c_int, p]
        lib.oracle_expert_groups.restype = ctypes.c_int
        lib.oracle_dispatch_group.argtypes = [ctypes.POINTER(Problem), p, p, p, ctypes.c_int, p, p, p, p]
        lib.oracle_dispatch_group.restype = None
        lib.oracle_combine_group.argtypes = [ctypes.POINTER(Problem), p, p, p, ctypes.c_int, ctypes.c_int,
                                             p, p, p, p]
        lib.oracle_combine_group.restype = None
        lib.oracle_swap_plan.argtypes = [ctypes.POINTER(Problem), p, ctypes.c_int32, p, p]
        lib.oracle_swap_plan.restype = ctypes.c_int
        lib.oracle_quantize_dispatch.argtypes = [ctypes.POINTER(Problem)] + [p] * 4
        lib.oracle_quantize_dispatch.restype = None
        lib.oracle_f32_to_e4m3_sat.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_e4m3_sat.restype = ctypes.c_uint8
        lib.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_f32.restype = ctypes.c_float
        lib.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    def __init__(self, code: int):
        super().__init__({ERR_INVALID: "invalid problem", ERR_BAD_IDS: "bad expert ids"}.get(code, str(code)))
        self.code = code


def make_problem(T, h, k, E, R, P, R_src, elem_bytes=2, scale_group=128,
                 expert_to_rank=None, src_offsets=None):
    """Returns (Problem, keepalive) for host-side calls."""
    keep = []
    e2r = None
    if expert_to_rank is not None:
        e2r = np.ascontiguousarray(expert_to_rank, dtype=np.int32)
        keep.append(e2r)
    so = None
    if src_offsets is not None:
        so = np.ascontiguousarray(src_offsets, dtype=np.int32)
        keep.append(so)
    prob = Problem(T, h, k, E, R, P, R_src, elem_bytes, scale_group,
                   None if e2r is None else e2r.ctypes.data, None if so is None else so.ctypes.data)
    return prob, keep


def layout(prob: Problem, ids: np.ndarray) -> dict:
    lib = _load()
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    H = prob.R // prob.P
    S = prob.T * prob.k
    out = dict(
        expert_count=np.zeros(prob.E, np.int32), expert_offset=np.zeros(prob.E + 1, np.int32),
        rank_count=np.zeros(prob.R, np.int32), rank_offset=np.zeros(prob.R + 1, np.int32),
        host_count=np.zeros(H, np.int32), host_offset=np.zeros(H + 1, np.int32),
        host_mask=np.zeros((prob.T, H), np.uint8), pos=np.zeros((prob.T, prob.k), np.int32),
        recv_src=np.zeros(S, np.int32))
    rc = lib.oracle_layout(ctypes.byref(prob), _ptr(ids), *[_ptr(out[n]) for n in (
        "expert_count", "expert_offset", "rank_count", "rank_offset", "host_count",
        "host_offset", "host_mask", "pos", "recv_src")])
    if rc != OK:
        raise OracleError(rc)
    return out


def stats(prob: Problem, ids: np.ndarray) -> dict:
    lib = _load()
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    glob = np.zeros(len(GLOBAL_FIELDS), np.int64)
    ratio = np.zeros(2, np.float64)
    src = np.zeros(len(SRC_FIELDS) * prob.R_src, np.int64)
    dst = np.zeros(len(DST_FIELDS) * prob.R, np.int64)
    rc = lib.oracle_stats(ctypes.byref(prob), _ptr(ids), _ptr(glob), _ptr(ratio), _ptr(src), _ptr(dst))
    if rc != OK:
        raise OracleError(rc)
    res = {n: int(glob[i]) for i, n in enumerate(GLOBAL_FIELDS)}
    res["imbalance_ratio"] = float(ratio[0])
    res["rank_imbalance"] = float(ratio[1])
    for i, n in enumerate(SRC_FIELDS):
        res[n] = src[i * prob.R_src:(i + 1) * prob.R_src].copy()
    for i, n in enumerate(DST_FIELDS):
        res[n] = dst[i * prob.R:(i + 1) * prob.R].copy()
    return res


def dispatch(prob: Problem, pos: np.ndarray, x: np.ndarray, x_scales=None):
    """x: [T, h] uint16 (bf16 bits) or uint8 (fp8 bits).  Returns recv (and recv_scales)."""
    lib = _load()
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    x = np.ascontiguousarray(x)
    S = prob.T * prob.k
    recv = np.zeros((S, prob.h), x.dtype)
    rs = None
    if x_scales is not None:
        x_scales = np.ascontiguousarray(x_scales, dtype=np.float32)
        rs = np.zeros((S, prob.h // prob.scale_group), np.float32)
    lib.oracle_dispatch(ctypes.byref(prob), _ptr(pos), _ptr(x), _ptr(x_scales), _ptr(recv), _ptr(rs))
    return (recv, rs) if x_scales is not None else recv


def combine(prob: Problem, pos: np.ndarray, y: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y: [rows, h] uint16 bf16 bits; w: [T, k] float32.  Returns out [T, h] uint16."""
    lib = _load()
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    y = np.ascontiguousarray(y, dtype=np.uint16)
    w = np.ascontiguousarray(w, dtype=np.float32)
    out = np.zeros((prob.T, prob.h), np.uint16)
    lib.oracle_combine(ctypes.byref(prob), _ptr(pos), _ptr(y), _ptr(w), _ptr(out))
    return out


def relay_layout(prob: Problem, ids: np.ndarray) -> np.ndarray:
    """Relay row of every (token, host) with the mask bit, -1 otherwise: [T, H]."""
    lib = _load()
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    H = prob.R // prob.P
    rp = np.zeros((prob.T, H), np.int32)
    rc = lib.oracle_relay_layout(ctypes.byref(prob), _ptr(ids), _ptr(rp))
    if rc != OK:
        raise OracleError(rc)
    return rp


def relay_dispatch(prob: Problem, ids, pos, relay_pos, x, x_scales=None):
    """Two-hop dispatch through the relay rows.  Returns (relay, relay_scales,
    recv, recv_scales) (scales None for bf16)."""
    lib = _load()
    ids = np.ascontiguousarray(ids, np.int32)
    pos = np.ascontiguousarray(pos, np.int32)
    rp = np.ascontiguousarray(relay_pos, np.int32)
    x = np.ascontiguousarray(x)
    n_relay = int((rp >= 0).sum())
    S = prob.T * prob.k
    relay = np.zeros((n_relay, prob.h), x.dtype)
    recv = np.zeros((S, prob.h), x.dtype)
    rs = rcv_s = None
    if x_scales is not None:
        x_scales = np.ascontiguousarray(x_scales, np.float32)
        G = prob.h // prob.scale_group
        rs = np.zeros((n_relay, G), np.float32)
        rcv_s = np.zeros((S, G), np.float32)
    lib.oracle_relay_dispatch(ctypes.byref(prob), _ptr(ids), _ptr(pos), _ptr(rp), _ptr(x), _ptr(x_scales),
                              _ptr(relay), _ptr(rs), _ptr(recv), _ptr(rcv_s))
    return relay, rs, recv, rcv_s


def relay_combine(prob: Problem, ids, pos, relay_pos, y, w):
    """Two-hop combine: bf16 per-host partials, then the ascending host sum.
    Returns (partial, out) as bf16 bits."""
    lib = _load()
    ids = np.ascontiguousarray(ids, np.int32)
    pos = np.ascontiguousarray(pos, np.int32)
    rp = np.ascontiguousarray(relay_pos, np.int32)
    y = np.ascontiguousarray(y, np.uint16)
    w = np.ascontiguousarray(w, np.float32)
    partial = np.zeros((int((rp >= 0).sum()), prob.h), np.uint16)
    out = np.zeros((prob.T, prob.h), np.uint16)
    lib.oracle_relay_combine(ctypes.byref(prob), _ptr(ids), _ptr(pos), _ptr(rp), _ptr(y), _ptr(w),
                             _ptr(partial), _ptr(out))
    return partial, out


def expert_groups(prob: Problem, G: int) -> np.ndarray:
    """Group of every expert: G contiguous runs of each rank's experts."""
    lib = _load()
    grp = np.zeros(prob.E, np.int32)
    rc = lib.oracle_expert_groups(ctypes.byref(prob), int(G), _ptr(grp))
    if rc != OK:
        raise OracleError(rc)
    return grp


def dispatch_group(prob: Problem, ids, pos, group, g, x, x_scales=None, recv=None, recv_scales=None):
    """Dispatch of group g's slots into recv (and recv_scales), in place when
    given; returns them."""
    lib = _load()
    ids = np.ascontiguousarray(ids, np.int32)
    pos = np.ascontiguousarray(pos, np.int32)
    group = np.ascontiguousarray(group, np.int32)
    x = np.ascontiguousarray(x)
    S = prob.T * prob.k
    if recv is None:
        recv = np.zeros((S, prob.h), x.dtype)
    if x_scales is not None:
        x_scales = np.ascontiguousarray(x_scales, np.float32)
        if recv_scales is None:
            recv_scales = np.zeros((S, prob.h // prob.scale_group), np.float32)
    lib.oracle_dispatch_group(ctypes.byref(prob), _ptr(ids), _ptr(pos), _ptr(group), int(g), _ptr(x),
                              _ptr(x_scales), _ptr(recv), _ptr(recv_scales))
    return recv, recv_scales


def combine_groups(prob: Problem, ids, pos, group, G, y, w):
    """All G group combines in order; returns (acc after each group but the
    last as a list of fp32 arrays, out as bf16 bits)."""
    lib = _load()
    ids = np.ascontiguousarray(ids, np.int32)
    pos = np.ascontiguousarray(pos, np.int32)
    group = np.ascontiguousarray(group, np.int32)
    y = np.ascontiguousarray(y, np.uint16)
    w = np.ascontiguousarray(w, np.float32)
    acc = np.zeros((prob.T, prob.h), np.float32)
    out = np.zeros((prob.T, prob.h), np.uint16)
    accs = []
    for g in range(G):
        lib.oracle_combine_group(ctypes.byref(prob), _ptr(ids), _ptr(pos), _ptr(group), g, int(G), _ptr(y),
                                 _ptr(w), _ptr(acc), _ptr(out))
        if g < G - 1:
            accs.append(acc.copy())
    return accs, out


def swap_plan(prob: Problem, expert_count: np.ndarray, tau: int):
    """Per-step intra-host expert swap.  Returns (new_expert_to_rank [E],
    swaps [H, P//2, 6] = rank a, rank b, x, y, old max, new max)."""
    lib = _load()
    cnt = np.ascontiguousarray(expert_count, dtype=np.int32)
    H = prob.R // prob.P
    new_e2r = np.zeros(prob.E, np.int32)
    swaps = np.zeros((H, prob.P // 2, 6), np.int32)
    rc = lib.oracle_swap_plan(ctypes.byref(prob), _ptr(cnt), int(tau), _ptr(new_e2r), _ptr(swaps))
    if rc != OK:
        raise OracleError(rc)
    return new_e2r, swaps


def quantize_dispatch(prob: Problem, pos: np.ndarray, x_bf16: np.ndarray):
    """Per-group amax/448 scales and e4m3 codes of bf16 x, dispatched to
    every receive row (quantise-in-dispatch).  Returns (codes, scales)."""
    lib = _load()
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    S = prob.T * prob.k
    codes = np.zeros((S, prob.h), np.uint8)
    scales = np.zeros((S, prob.h // prob.scale_group), np.float32)
    lib.oracle_quantize_dispatch(ctypes.byref(prob), _ptr(pos), _ptr(x), _ptr(codes), _ptr(scales))
    return codes, scales


def f32_to_e4m3(values) -> np.ndarray:
    lib = _load()
    v = np.asarray(values, np.float32).ravel()
    return np.array([lib.oracle_f32_to_e4m3_sat(float(f)) for f in v], np.uint8)


def e4m3_to_f32(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, np.uint8).ravel()
    return np.array([lib.oracle_e4m3_to_f32(int(u)) for u in c], np.float32)


def f32_to_bf16(values) -> np.ndarray:
    lib = _load()
    v = np.asarray(values, np.float32).ravel()
    return np.array([lib.oracle_f32_to_bf16_rne(float(f)) for f in v], np.uint16)


def bf16_to_f32(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, np.uint16).ravel()
    return np.array([lib.oracle_bf16_to_f32(int(u)) for u in b], np.float32)
