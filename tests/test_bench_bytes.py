"""The bench's algorithmic byte counts, checked on CPU against the sizes the
workloads imply (no GPU)."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import moe_workloads as mw  # noqa: E402


def test_flat_bytes_of_the_largest_workload():
    """prefill-fp8: dispatch reads 16384 rows of 7168 + 224 B and writes 8
    copies; combine reads 8 bf16 rows per token and writes one."""
    d, c = bench.algorithmic_bytes(mw.WORKLOADS["prefill-fp8"])
    assert d == 16384 * 7392 * 9 == 1_089_994_752
    assert c == 16384 * 8 * 14336 + 16384 * 14336 == 2_113_929_216


def test_quantise_bytes_read_bf16_rows():
    d, _ = bench.algorithmic_bytes(mw.WORKLOADS["prefill-fp8-quant"])
    assert d == 16384 * (14336 + 8 * 7392)


def test_relay_bytes_add_one_write_and_one_read_per_relay_row():
    w = mw.WORKLOADS["decode-EP32-r8"]
    d0, c0 = bench.algorithmic_bytes(w)
    d, c = bench.relay_bytes(w, 1000)
    assert d - d0 == 2 * 1000 * 2 * w.h and c - c0 == 2 * 1000 * 2 * w.h
    assert bench.relay_bytes(w, 0) == (d0, c0)


def test_group_bytes():
    """One group is the flat pair; with more groups a token's row is read once
    per group it has a slot in, and the fp32 chain adds 4h (first) + 8h per
    middle group with a slot + 6h (last) per token."""
    w = mw.Workload("g", T=64, h=256, k=4, E=16, R=4, P=2, R_src=1)
    ids = mw.gen_ids(w)
    group1 = np.zeros(w.E, np.int32)
    assert bench.peo_bytes(w, ids, group1, 1) == bench.algorithmic_bytes(w)
    group2 = (np.arange(w.E) % (w.E // w.R)) * 2 // (w.E // w.R)
    d, c = bench.peo_bytes(w, ids, group2.astype(np.int32), 2)
    rho = 2 * w.h
    rows_read = sum(int((group2[ids] == g).any(axis=1).sum()) for g in range(2))
    assert d == rho * (rows_read + w.T * w.k)
    assert c == 2 * w.h * w.T * w.k + 10 * w.h * w.T


def test_tokens_option_runs_a_smaller_case():
    """--tokens runs the same workload with fewer tokens and names it so (the
    oracle arm, which needs no GPU); a count the source ranks do not divide
    is refused."""
    bench = os.path.join(ROOT, "bench.py")
    p = subprocess.run([sys.executable, bench, "--impl", "reference", "--workload", "prefill-fp8", "--tokens", "256",
                        "--steps", "2", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    d = json.loads(p.stdout.strip().splitlines()[-1])
    assert d["config"]["workload"] == "prefill-fp8@T256" and d["config"]["T"] == 256
    p = subprocess.run([sys.executable, bench, "--impl", "reference", "--workload", "decode-EP32-r8", "--tokens", "100"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode != 0 and "multiple of the 32 source ranks" in p.stderr
