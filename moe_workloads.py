"""Seeded synthetic inputs for MoE layout / dispatch / combine.

This module only draws inputs: routing ids, gate weights, hidden states and
expert outputs.  It holds none of the layout, statistics, dispatch or combine
arithmetic, so both the CUDA library's tests and the CPU oracle can take their
inputs from here.

Workload recipe (shapes from the pages' settings; no dataset is involved):

* hidden states x ~ N(0, 1), rounded to bf16; for fp8 workloads, quantised per
  128 columns with scale = amax / 448 and e4m3 codes of x / scale (the page
  "Poor HybridEP performance on dual-node 16x B300 GPUs" runs FP8 dispatch
  with scales; its payload bytes are about half of bf16).
* gate weights: softmax over the k chosen slots of N(0, 1) logits (fp32).
* routing: each token picks k distinct experts ("Balancing and Beyond",
  section 3.2).  Uniform routing takes the first k of a random permutation of
  the E experts.  Skewed routing gives expert e the popularity (rank of e)^-s
  in a seed-permuted order (a Zipf law) and draws k experts without
  replacement by the Gumbel-top-k trick; "Balancing and Beyond" section 2
  reports imbalance ratios of about 2.6 to 20 in production traces.
* expert outputs y ~ N(0, 1) bf16, one row per receive slot.

Every draw is a pure function of (seed, stream, step).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

# Draw streams, so that ids, gates and x never share random numbers.
_IDS, _GATES, _X, _Y, _PERM = 1, 2, 3, 4, 5

# Zipf exponents giving a target imbalance ratio at seed 0.  They were found by
# bisection with tests/golden/calibrate_zipf.py (which measures the ratio with
# the oracle) and are stored in tests/golden/zipf_calibration.json; a test
# re-checks that they still hit their targets.
ZIPF_S_DECODE_RATIO8 = 0.5216
# Sixteen per-step targets, geometric from 2.5 to 20 (E/k = 160/8 = 20 is the
# largest ratio possible: the hottest expert in every token).
ALT_RATIO_TARGETS = tuple(2.5 * (20.0 / 2.5) ** (i / 15.0) for i in range(16))
ZIPF_S_ALT_STEPS = (0.2424, 0.2774, 0.3127, 0.3633, 0.4167, 0.4390, 0.4814, 0.5394,
                    0.5719, 0.6442, 0.6922, 0.7599, 0.8424, 0.9290, 1.0655, 1.6718)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int                   # tokens
    h: int                   # hidden size
    k: int                   # top-k
    E: int                   # experts
    R: int                   # logical EP ranks
    P: int                   # ranks per host
    R_src: int               # source ranks (tokens split evenly among ranks 0..R_src-1)
    dtype: str = "bf16"      # "bf16" or "fp8"
    routing: str = "uniform" # "uniform" or "zipf"
    zipf_s: float = 0.0
    seed: int = 0
    steps: int = 1           # >1: routing re-drawn per step (per-step s table)
    scale_group: int = 128
    quantize: bool = False   # fp8 receive rows made from bf16 x inside dispatch

    @property
    def H(self) -> int:
        return self.R // self.P

    @property
    def slots(self) -> int:
        return self.T * self.k

    def s_for_step(self, step: int) -> float:
        if self.name.startswith("decode-EP32-alt"):
            return ZIPF_S_ALT_STEPS[step % len(ZIPF_S_ALT_STEPS)]
        return self.zipf_s


WORKLOADS = {
    # T=256, h=1024, 16 experts top-2 over 4 ranks x 4 experts, 2 hosts.
    "tiny": Workload("tiny", T=256, h=1024, k=2, E=16, R=4, P=2, R_src=4),
    # 32 ranks x 128 tokens, h=7168, 256 experts top-8, 4 hosts of 8 ranks,
    # Zipf skew calibrated to an imbalance ratio of about 8 ...
    "decode-EP32-r8": Workload("decode-EP32-r8", T=4096, h=7168, k=8, E=256, R=32, P=8,
                               R_src=32, routing="zipf", zipf_s=ZIPF_S_DECODE_RATIO8),
    # ... and with the literal exponent s = 1.1 (ratio about 28 under this sampler).
    "decode-EP32-s1.1": Workload("decode-EP32-s1.1", T=4096, h=7168, k=8, E=256, R=32, P=8,
                                 R_src=32, routing="zipf", zipf_s=1.1),
    # h=6144, 160 experts top-8 on 32 ranks (5 per rank), 4 hosts, skew
    # re-drawn each of 16 steps with ratios from 2.5 to 20.
    "decode-EP32-alt": Workload("decode-EP32-alt", T=4096, h=6144, k=8, E=160, R=32, P=8,
                                R_src=32, routing="zipf", steps=16),
    # 4096 tokens on one rank, h=7168, 128 experts top-8 over 16 ranks (8 local
    # experts), 2 hosts, uniform routing (the HybridEP issue's shape).
    "prefill": Workload("prefill", T=4096, h=7168, k=8, E=128, R=16, P=8, R_src=1),
    # As prefill but T=16384, fp8 e4m3 hidden states with fp32 scales per 128
    # columns, Zipf(s=1.0) skew.
    "prefill-fp8": Workload("prefill-fp8", T=16384, h=7168, k=8, E=128, R=16, P=8, R_src=1,
                            dtype="fp8", routing="zipf", zipf_s=1.0),
    # As prefill-fp8, but x arrives in bf16 and dispatch quantises it.
    "prefill-fp8-quant": Workload("prefill-fp8-quant", T=16384, h=7168, k=8, E=128, R=16, P=8, R_src=1,
                                  dtype="fp8", routing="zipf", zipf_s=1.0, quantize=True),
}


def _rng(w: Workload, stream: int, step: int = 0) -> np.random.Generator:
    return np.random.default_rng([w.seed, stream, step])


def gen_ids(w: Workload, step: int = 0, s: Optional[float] = None) -> np.ndarray:
    """Top-k expert ids [T, k] int32, k distinct experts per token."""
    rng = _rng(w, _IDS, step)
    if w.routing == "uniform":
        keys = rng.random((w.T, w.E))
        return np.argsort(keys, axis=1, kind="stable")[:, : w.k].astype(np.int32)
    s = w.s_for_step(step) if s is None else s
    perm = _rng(w, _PERM, step).permutation(w.E)
    popularity_rank = np.empty(w.E, np.float64)
    popularity_rank[perm] = np.arange(1, w.E + 1, dtype=np.float64)
    log_p = -s * np.log(popularity_rank)
    gumbel = -np.log(-np.log(rng.random((w.T, w.E)).clip(1e-300, 1.0 - 1e-16)))
    keys = log_p[None, :] + gumbel
    top = np.argpartition(-keys, w.k - 1, axis=1)[:, : w.k]
    order = np.argsort(-np.take_along_axis(keys, top, axis=1), axis=1, kind="stable")
    return np.take_along_axis(top, order, axis=1).astype(np.int32)


def gen_gates(w: Workload, step: int = 0) -> np.ndarray:
    """Gate weights [T, k] float32: softmax over the k slots of N(0,1) logits."""
    logits = _rng(w, _GATES, step).standard_normal((w.T, w.k))
    z = np.exp(logits - logits.max(axis=1, keepdims=True))
    return (z / z.sum(axis=1, keepdims=True)).astype(np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (library conversion) and return the bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def gen_x_bf16(w: Workload, rows: Optional[int] = None) -> np.ndarray:
    """Hidden states [T, h] as bf16 bit patterns (uint16)."""
    rows = w.T if rows is None else rows
    x = _rng(w, _X).standard_normal((rows, w.h), dtype=np.float32)
    return f32_to_bf16_bits(x)


def gen_x_fp8(w: Workload, rows: Optional[int] = None):
    """Hidden states as (e4m3 codes [T, h] uint8, fp32 scales [T, h/128])."""
    import torch
    rows = w.T if rows is None else rows
    g = w.scale_group
    x = _rng(w, _X).standard_normal((rows, w.h), dtype=np.float32).reshape(rows, w.h // g, g)
    amax = np.abs(x).max(axis=2)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = np.clip(x / scale[:, :, None], -448.0, 448.0).reshape(rows, w.h)
    codes = torch.from_numpy(np.ascontiguousarray(q)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, scale


def fp8_codes_to_f32(codes: np.ndarray) -> np.ndarray:
    import torch
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn).float().numpy()


def gen_y_host(w: Workload, rows: Optional[int] = None, seed_offset: int = 0) -> np.ndarray:
    """Expert outputs [rows, h] bf16 bits (host), rows defaults to T*k."""
    rows = w.slots if rows is None else rows
    y = _rng(w, _Y, seed_offset).standard_normal((rows, w.h), dtype=np.float32)
    return f32_to_bf16_bits(y)


def gen_y_device(w: Workload, device, rows: Optional[int] = None, seed_offset: int = 0):
    """Expert outputs [rows, h] bf16 drawn on a device (large workloads)."""
    import torch
    rows = w.slots if rows is None else rows
    g = torch.Generator(device=device)
    g.manual_seed(w.seed * 1000003 + _Y * 1009 + seed_offset)
    y = torch.empty((rows, w.h), dtype=torch.bfloat16, device=device)
    chunk = max(1, (1 << 27) // max(1, w.h))
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        y[r0:r1] = torch.randn((r1 - r0, w.h), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return y


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (for small parity cases)."""
    return dataclasses.replace(w, **changes)


def ratio_targets_geometric(lo: float, hi: float, n: int):
    return tuple(lo * (hi / lo) ** (i / (n - 1)) for i in range(n))


assert all(math.isclose(a, b) for a, b in zip(ALT_RATIO_TARGETS, ratio_targets_geometric(2.5, 20.0, 16)))
