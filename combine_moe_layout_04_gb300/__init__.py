"""Python binding of libmoe_layout.so: MoE token layout, dispatch and combine on GB300.

Argument marshalling only.  Every step runs in the library's CUDA kernels
(``csrc/``); PyTorch provides device memory and streams.  The entry points
mirror the C-ABI declared in ``include/moe_layout.h``:

    moe_workspace_bytes, moe_layout, moe_stats_words, moe_stats (host record,
    synchronises), moe_stats_device, moe_dispatch, moe_combine, moe_status,
    moe_status_string, moe_layout_noalloc,
    moe_relay_layout, moe_dispatch_relay, moe_combine_relay (the Mode 2 relay),
    moe_expert_groups, moe_dispatch_group, moe_combine_group (per-expert groups)

``Problem`` and ``Layout`` are conveniences that build the C structs and
allocate the caller-owned device buffers.  If the shared library has not been
built, every call raises ``MoeLibraryMissing``; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_layout.so")

MOE_OK, MOE_ERR_INVALID, MOE_ERR_CUDA, MOE_ERR_BAD_IDS, MOE_ERR_ALIGN, MOE_ERR_CAPACITY, MOE_ERR_TIMEOUT = \
    0, 1, 2, 3, 4, 5, 6
MOE_NOALLOC_SCRATCH_BYTES = 2 << 20
MOE_DTYPE_BF16, MOE_DTYPE_FP8_E4M3 = 0, 1
MOE_STATUS_ID_RANGE, MOE_STATUS_ID_REPEAT, MOE_STATUS_PLACEMENT, MOE_STATUS_SRC_OFFSET = 1, 2, 4, 8
MOE_STATUS_TIMEOUT = 16
MOE_STATUS_RELAY_CAPACITY = 32
MOE_FP8_GROUP = 128
MOE_MAX_GROUPS = 64
MOE_MAX_HIDDEN = 1 << 20
MOE_STATS_HEADER_WORDS = 32
MOE_ST_STATUS = 0  # header word holding the device status bits
MOE_FAULT_WAIT_TIMEOUT = 1
MOE_MOVE_AUTO, MOE_MOVE_VECTOR, MOE_MOVE_BULK = 0, 1, 2
MOE_LAYOUT_AUTO, MOE_LAYOUT_SPLIT, MOE_LAYOUT_FUSED, MOE_LAYOUT_TWO_KERNELS = 0, 1, 2, 3

# Header word names in index order (include/moe_layout.h, MOE_ST_*).
STATS_HEADER = ("status", "T", "slots", "row_bytes", "max_expert_count", "argmax_expert",
                "min_expert_count", "max_rank_slots", "max_rank_tokens",
                "sum_mode0_copies", "sum_mode1_copies", "sum_mode2_copies",
                "max_src_mode1_copies", "max_src_mode2_copies", "max_recv_remote", "max_recv_relay",
                "sum_naive_bytes", "sum_mode0_bytes", "sum_mode1_bytes", "sum_mode2_bytes",
                "imbalance_ratio", "rank_imbalance", "num_hosts")
STATS_SRC = ("src_tokens", "src_copies", "src_mode0", "src_mode1", "src_mode2",
             "src_naive_bytes", "src_mode0_bytes", "src_mode1_bytes", "src_mode2_bytes")
STATS_DST = ("recv_slots", "recv_tokens", "recv_self", "recv_local", "recv_remote", "recv_relay")
EXPORTED = ("moe_workspace_bytes", "moe_layout", "moe_stats_words", "moe_stats", "moe_stats_device",
            "moe_dispatch",
            "moe_combine", "moe_status", "moe_status_string", "moe_layout_noalloc",
            "moe_move_faults", "moe_selftest_bounded_waits", "moe_dispatch_quant", "moe_swap_plan",
            "moe_relay_layout", "moe_dispatch_relay", "moe_combine_relay",
            "moe_expert_groups", "moe_dispatch_group", "moe_combine_group")


class MoeLibraryMissing(RuntimeError):
    pass


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {moe_status_string(code)} (code {code})")
        self.code = code


_TUNING_FIELDS = ("dispatch_kind", "dispatch_sms", "dispatch_ctas_per_sm", "dispatch_warps", "dispatch_stages",
                  "dispatch_chunk_bytes", "combine_kind", "combine_sms", "combine_ctas_per_sm", "layout_kind")


class _TuningC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in _TUNING_FIELDS] + [("reserved", ctypes.c_int32 * 6)]


class _ProblemC(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("hidden", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("num_ranks", ctypes.c_int32),
                ("ranks_per_host", ctypes.c_int32), ("num_src_ranks", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("expert_to_rank", ctypes.c_void_p),
                ("src_rank_offsets", ctypes.c_void_p), ("tuning", ctypes.POINTER(_TuningC))]


@dataclass
class Tuning:
    """Launch shapes of the layout and the row movers (moe_tuning in
    include/moe_layout.h); 0 keeps the library's default.  Shapes change
    speed only, never results."""
    dispatch_kind: int = MOE_MOVE_AUTO
    dispatch_sms: int = 0
    dispatch_ctas_per_sm: int = 0
    dispatch_warps: int = 0
    dispatch_stages: int = 0
    dispatch_chunk_bytes: int = 0
    combine_kind: int = MOE_MOVE_AUTO
    combine_sms: int = 0
    combine_ctas_per_sm: int = 0
    layout_kind: int = MOE_LAYOUT_AUTO

    def c(self) -> _TuningC:
        return _TuningC(*[int(getattr(self, n)) for n in _TUNING_FIELDS])

    def as_dict(self) -> dict:
        return {n: int(getattr(self, n)) for n in _TUNING_FIELDS}

    @classmethod
    def from_env(cls, environ=None) -> "Tuning":
        """MOE_DISPATCH_KIND, MOE_DISPATCH_SMS, ... (upper-case field names
        with a MOE_ prefix; mover kinds also as "auto", "vector" or "bulk",
        the layout kind as "auto", "split", "fused" or "two_kernels")."""
        env = os.environ if environ is None else environ
        move = {"auto": MOE_MOVE_AUTO, "vector": MOE_MOVE_VECTOR, "bulk": MOE_MOVE_BULK}
        layout = {"auto": MOE_LAYOUT_AUTO, "split": MOE_LAYOUT_SPLIT, "fused": MOE_LAYOUT_FUSED,
                  "two_kernels": MOE_LAYOUT_TWO_KERNELS}
        vals = {}
        for n in _TUNING_FIELDS:
            v = env.get("MOE_" + n.upper())
            if v is not None and v != "":
                kinds = layout if n == "layout_kind" else move
                vals[n] = kinds[v.lower()] if v.lower() in kinds else int(v)
        return cls(**vals)


_LAYOUT_FIELDS = ("expert_count", "expert_offset", "rank_count", "rank_offset", "host_count",
                  "host_offset", "host_mask", "pos", "recv_src")


class _LayoutC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _LAYOUT_FIELDS] + [("stats", ctypes.c_void_p)]


class _RelayC(ctypes.Structure):
    _fields_ = [("relay_pos", ctypes.c_void_p), ("relay_src", ctypes.c_void_p), ("slot_relay", ctypes.c_void_p),
                ("capacity", ctypes.c_int64)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Loads libmoe_layout.so (raises MoeLibraryMissing if it is not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise MoeLibraryMissing(f"{path} is not built; run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    vp, i = ctypes.c_void_p, ctypes.c_int
    P, L = ctypes.POINTER(_ProblemC), ctypes.POINTER(_LayoutC)
    lib.moe_workspace_bytes.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
    lib.moe_workspace_bytes.restype = i
    lib.moe_layout.argtypes = [P, vp, vp, L, vp]
    lib.moe_layout.restype = i
    lib.moe_stats_words.argtypes = [P]
    lib.moe_stats_words.restype = ctypes.c_size_t
    lib.moe_stats.argtypes = [P, L, vp, ctypes.POINTER(ctypes.c_int64), vp]
    lib.moe_stats.restype = i
    lib.moe_stats_device.argtypes = [P, vp, vp, vp]
    lib.moe_stats_device.restype = i
    lib.moe_dispatch.argtypes = [P, L, vp, vp, vp, vp, vp]
    lib.moe_dispatch.restype = i
    lib.moe_swap_plan.argtypes = [P, L, ctypes.c_int32, vp, vp, vp]
    lib.moe_swap_plan.restype = i
    lib.moe_dispatch_quant.argtypes = [P, L, vp, vp, vp, vp]
    lib.moe_dispatch_quant.restype = i
    lib.moe_combine.argtypes = [P, L, vp, vp, vp, vp]
    lib.moe_combine.restype = i
    Q = ctypes.POINTER(_RelayC)
    lib.moe_relay_layout.argtypes = [P, L, vp, Q, vp]
    lib.moe_relay_layout.restype = i
    lib.moe_dispatch_relay.argtypes = [P, L, Q, vp, vp, vp, vp, vp, vp, vp]
    lib.moe_dispatch_relay.restype = i
    lib.moe_combine_relay.argtypes = [P, L, Q, vp, vp, vp, vp, vp]
    lib.moe_combine_relay.restype = i
    i32 = ctypes.c_int32
    lib.moe_expert_groups.argtypes = [P, i32, vp, vp]
    lib.moe_expert_groups.restype = i
    lib.moe_dispatch_group.argtypes = [P, L, vp, vp, i32, vp, vp, vp, vp, vp]
    lib.moe_dispatch_group.restype = i
    lib.moe_combine_group.argtypes = [P, L, vp, vp, i32, i32, vp, vp, vp, vp, vp]
    lib.moe_combine_group.restype = i
    lib.moe_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    lib.moe_status.restype = i
    lib.moe_layout_noalloc.argtypes = [P, vp, L, vp]
    lib.moe_layout_noalloc.restype = i
    lib.moe_move_faults.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
    lib.moe_move_faults.restype = i
    lib.moe_selftest_bounded_waits.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
    lib.moe_selftest_bounded_waits.restype = i
    lib.moe_status_string.argtypes = [i]
    lib.moe_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class Problem:
    """One layer's routing problem (see include/moe_layout.h, moe_problem)."""
    num_tokens: int
    hidden: int
    topk: int
    num_experts: int
    num_ranks: int
    ranks_per_host: int
    num_src_ranks: int = 1
    dtype: int = MOE_DTYPE_BF16
    expert_to_rank: object = None      # device int32 tensor [E] or None
    src_rank_offsets: object = None    # device int32 tensor [R_src + 1] or None
    tuning: Optional[Tuning] = None    # launch shapes, or None for the defaults

    @property
    def num_hosts(self) -> int:
        return self.num_ranks // self.ranks_per_host

    @property
    def row_bytes(self) -> int:
        if self.dtype == MOE_DTYPE_FP8_E4M3:
            return self.hidden + 4 * (self.hidden // MOE_FP8_GROUP)
        return 2 * self.hidden

    def c(self) -> _ProblemC:
        # the struct keeps its tuning alive for as long as it is referenced
        pc = _ProblemC(self.num_tokens, self.hidden, self.topk, self.num_experts, self.num_ranks,
                       self.ranks_per_host, self.num_src_ranks, self.dtype,
                       _ptr(self.expert_to_rank), _ptr(self.src_rank_offsets), None)
        if self.tuning is not None:
            pc._tuning = self.tuning.c()
            pc.tuning = ctypes.pointer(pc._tuning)
        return pc


class Layout:
    """Caller-owned device arrays of a layout (moe_layout_t)."""

    def __init__(self, problem: Problem, device="cuda", with_stats: bool = False):
        import torch
        p = problem
        i32 = dict(dtype=torch.int32, device=device)
        self.expert_count = torch.empty(p.num_experts, **i32)
        self.expert_offset = torch.empty(p.num_experts + 1, **i32)
        self.rank_count = torch.empty(p.num_ranks, **i32)
        self.rank_offset = torch.empty(p.num_ranks + 1, **i32)
        self.host_count = torch.empty(p.num_hosts, **i32)
        self.host_offset = torch.empty(p.num_hosts + 1, **i32)
        self.host_mask = torch.empty((p.num_tokens, p.num_hosts), dtype=torch.uint8, device=device)
        self.pos = torch.empty((p.num_tokens, p.topk), **i32)
        self.recv_src = torch.empty(p.num_tokens * p.topk, **i32)
        # Optional: the statistics record, written by moe_layout itself.
        self.stats = (torch.empty(moe_stats_words(p), dtype=torch.int64, device=device)
                      if with_stats else None)

    def c(self) -> _LayoutC:
        stats = getattr(self, "stats", None)
        return _LayoutC(*[getattr(self, n).data_ptr() for n in _LAYOUT_FIELDS],
                        None if stats is None else stats.data_ptr())

    def to_host(self) -> dict:
        return {n: getattr(self, n).cpu().numpy() for n in _LAYOUT_FIELDS}


class Relay:
    """Caller-owned device arrays of the Mode 2 relay rows (moe_relay_t).  The
    default capacity, T * min(k, H), holds every layout of the problem."""

    def __init__(self, problem: Problem, device="cuda", capacity: Optional[int] = None):
        import torch
        p = problem
        i32 = dict(dtype=torch.int32, device=device)
        self.capacity = p.num_tokens * min(p.topk, p.num_hosts) if capacity is None else int(capacity)
        self.relay_pos = torch.empty((p.num_tokens, p.num_hosts), **i32)
        self.relay_src = torch.empty(max(self.capacity, 1), **i32)
        self.slot_relay = torch.empty((p.num_tokens, p.topk), **i32)

    def c(self) -> _RelayC:
        return _RelayC(self.relay_pos.data_ptr(), self.relay_src.data_ptr(), self.slot_relay.data_ptr(),
                       self.capacity)


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def moe_status_string(code: int) -> str:
    return load_library().moe_status_string(int(code)).decode()


def moe_workspace_bytes(problem: Problem) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().moe_workspace_bytes(ctypes.byref(problem.c()), ctypes.byref(n)),
           "moe_workspace_bytes")
    return n.value


def alloc_workspace(problem: Problem, device="cuda"):
    import torch
    return torch.empty(moe_workspace_bytes(problem), dtype=torch.uint8, device=device)


def moe_layout(problem: Problem, ids, workspace, layout: Layout, stream=None):
    _check(load_library().moe_layout(ctypes.byref(problem.c()), _ptr(ids), _ptr(workspace),
                                     ctypes.byref(layout.c()), _stream(stream)), "moe_layout")


def moe_layout_noalloc(problem: Problem, ids, layout: Layout, stream=None):
    """moe_layout without a workspace: the library's fixed device scratch is
    used instead (for callers that cannot allocate device memory).  Calls that
    may overlap on the GPU share that scratch and must be serialised."""
    _check(load_library().moe_layout_noalloc(ctypes.byref(problem.c()), _ptr(ids),
                                             ctypes.byref(layout.c()), _stream(stream)),
           "moe_layout_noalloc")


def moe_stats_words(problem: Problem) -> int:
    return int(load_library().moe_stats_words(ctypes.byref(problem.c())))


def moe_stats(problem: Problem, layout: Layout, workspace=None, stream=None):
    """The statistics record copied to host memory; synchronises the stream.
    Returns (code, record): code is what moe_status would return for the
    record's status word, record a numpy int64 array (decode_stats names its
    words).  With layout.stats set the record comes from there and the
    workspace may be None."""
    import numpy as np
    rec = np.zeros(moe_stats_words(problem), dtype=np.int64)
    rc = load_library().moe_stats(ctypes.byref(problem.c()), ctypes.byref(layout.c()), _ptr(workspace),
                                  rec.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _stream(stream))
    # A code that the record's status word explains came from the device; any
    # other is a host-side rejection or a failed copy, and the record is empty.
    from_record = rc in (MOE_OK, MOE_ERR_BAD_IDS, MOE_ERR_CAPACITY, MOE_ERR_TIMEOUT) or (
        rc == MOE_ERR_INVALID and int(rec[0]) & (MOE_STATUS_PLACEMENT | MOE_STATUS_SRC_OFFSET))
    if not from_record:
        raise MoeError(rc, "moe_stats")
    return rc, rec


def moe_stats_device(problem: Problem, workspace, stats, stream=None):
    """The statistics record copied to a device int64 tensor, asynchronously."""
    _check(load_library().moe_stats_device(ctypes.byref(problem.c()), _ptr(workspace), _ptr(stats),
                                           _stream(stream)), "moe_stats_device")


def moe_dispatch(problem: Problem, layout: Layout, x, x_scales, recv, recv_scales, stream=None):
    _check(load_library().moe_dispatch(ctypes.byref(problem.c()), ctypes.byref(layout.c()), _ptr(x),
                                       _ptr(x_scales), _ptr(recv), _ptr(recv_scales), _stream(stream)),
           "moe_dispatch")


def moe_swap_plan(problem: Problem, layout: Layout, tau: int, new_expert_to_rank, swaps=None, stream=None):
    """Per-step intra-host expert swap plan from the layout's expert counts."""
    _check(load_library().moe_swap_plan(ctypes.byref(problem.c()), ctypes.byref(layout.c()), int(tau),
                                        _ptr(new_expert_to_rank), _ptr(swaps), _stream(stream)),
           "moe_swap_plan")


def moe_dispatch_quant(problem: Problem, layout: Layout, x_bf16, recv, recv_scales, stream=None):
    """Dispatch that converts bf16 rows to e4m3 codes + fp32 scales per 128 columns."""
    _check(load_library().moe_dispatch_quant(ctypes.byref(problem.c()), ctypes.byref(layout.c()),
                                             _ptr(x_bf16), _ptr(recv), _ptr(recv_scales), _stream(stream)),
           "moe_dispatch_quant")


def moe_combine(problem: Problem, layout: Layout, y, weights, out, stream=None):
    _check(load_library().moe_combine(ctypes.byref(problem.c()), ctypes.byref(layout.c()), _ptr(y),
                                      _ptr(weights), _ptr(out), _stream(stream)), "moe_combine")


def moe_relay_layout(problem: Problem, layout: Layout, workspace, relay: Relay, stream=None):
    """Relay rows of a layout made with this workspace."""
    _check(load_library().moe_relay_layout(ctypes.byref(problem.c()), ctypes.byref(layout.c()), _ptr(workspace),
                                           ctypes.byref(relay.c()), _stream(stream)), "moe_relay_layout")


def moe_dispatch_relay(problem: Problem, layout: Layout, relay: Relay, x, x_scales, relay_rows, relay_scales,
                       recv, recv_scales, stream=None):
    """Two-hop dispatch: x to the relay rows, then the relay rows to recv."""
    _check(load_library().moe_dispatch_relay(ctypes.byref(problem.c()), ctypes.byref(layout.c()),
                                             ctypes.byref(relay.c()), _ptr(x), _ptr(x_scales), _ptr(relay_rows),
                                             _ptr(relay_scales), _ptr(recv), _ptr(recv_scales), _stream(stream)),
           "moe_dispatch_relay")


def moe_combine_relay(problem: Problem, layout: Layout, relay: Relay, y, weights, partial, out, stream=None):
    """Two-hop combine: per-host bf16 partials, then their sum in host order."""
    _check(load_library().moe_combine_relay(ctypes.byref(problem.c()), ctypes.byref(layout.c()),
                                            ctypes.byref(relay.c()), _ptr(y), _ptr(weights), _ptr(partial),
                                            _ptr(out), _stream(stream)), "moe_combine_relay")


def moe_expert_groups(problem: Problem, num_groups: int, expert_group, stream=None):
    """Group of every expert: G contiguous runs of each rank's experts."""
    _check(load_library().moe_expert_groups(ctypes.byref(problem.c()), int(num_groups), _ptr(expert_group),
                                            _stream(stream)), "moe_expert_groups")


def moe_dispatch_group(problem: Problem, layout: Layout, ids, expert_group, group: int, x, x_scales, recv,
                       recv_scales, stream=None):
    """Dispatch of the slots whose expert is in `group`."""
    _check(load_library().moe_dispatch_group(ctypes.byref(problem.c()), ctypes.byref(layout.c()), _ptr(ids),
                                             _ptr(expert_group), int(group), _ptr(x), _ptr(x_scales), _ptr(recv),
                                             _ptr(recv_scales), _stream(stream)), "moe_dispatch_group")


def moe_combine_group(problem: Problem, layout: Layout, ids, expert_group, group: int, num_groups: int, y, weights,
                      acc, out, stream=None):
    """Combine of one expert group; the groups continue one fp32 chain per
    token through `acc` and the last writes `out`."""
    _check(load_library().moe_combine_group(ctypes.byref(problem.c()), ctypes.byref(layout.c()), _ptr(ids),
                                            _ptr(expert_group), int(group), int(num_groups), _ptr(y),
                                            _ptr(weights), _ptr(acc), _ptr(out), _stream(stream)),
           "moe_combine_group")


def moe_status(workspace, stream=None):
    """Synchronises the stream; returns (code, status_bits)."""
    bits = ctypes.c_uint32(0)
    rc = load_library().moe_status(_ptr(workspace), ctypes.byref(bits), _stream(stream))
    return rc, bits.value


def moe_move_faults(stream=None) -> int:
    """Synchronises the stream; returns and clears the row movers' fault bits."""
    bits = ctypes.c_uint32(0)
    _check(load_library().moe_move_faults(ctypes.byref(bits), _stream(stream)), "moe_move_faults")
    return bits.value


def moe_selftest_bounded_waits(stream=None) -> int:
    """Runs the bounded-wait self-test; returns its bits (0xF = all good)."""
    bits = ctypes.c_uint32(0)
    _check(load_library().moe_selftest_bounded_waits(ctypes.byref(bits), _stream(stream)),
           "moe_selftest_bounded_waits")
    return bits.value


def decode_stats(problem: Problem, stats_host) -> dict:
    """Names the words of a statistics record copied to the host (numpy int64)."""
    import numpy as np
    s = np.asarray(stats_host, dtype=np.int64)
    out = {}
    for i, n in enumerate(STATS_HEADER):
        out[n] = int(s[i])
    for n in ("imbalance_ratio", "rank_imbalance"):
        out[n] = float(np.array([out[n]], np.int64).view(np.float64)[0])
    base = MOE_STATS_HEADER_WORDS
    rs, r = problem.num_src_ranks, problem.num_ranks
    for i, n in enumerate(STATS_SRC):
        out[n] = s[base + i * rs: base + (i + 1) * rs].copy()
    base += len(STATS_SRC) * rs
    for i, n in enumerate(STATS_DST):
        out[n] = s[base + i * r: base + (i + 1) * r].copy()
    return out
