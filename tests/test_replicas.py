"""The multi-GPU form of the bench is N independent replicas (the path has no
exchange step on one GPU).  Its host logic -- ranks from the torchrun
environment, the barrier, the max over ranks of the timings, the whole-job
value, one JSON line from rank 0 -- runs here on CPU over gloo, world size 2."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup("gloo")
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    ms = 1.0 + rank                       # rank 1 is the slower one
    ms_max = bench.max_over_ranks(ms, w)
    value = bench.job_value(2e9, ms_max, w)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"ms_max": ms_max, "value": value}, f)
    dist.destroy_process_group()


def test_rank_helpers_over_gloo(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        assert r["ms_max"] == 2.0                       # the slowest rank sets the time
        assert r["value"] == pytest.approx(world * 2e9 / 2e-3 / 1e9)   # N x per-rank bytes


def test_reference_arm_under_torchrun():
    """`bench.py --impl reference` launched like the GPU arm with 2 ranks:
    rank 0 alone runs the oracle and prints one line; rank 1 exits 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
           "--gpus", "2", "--steps", "2", "--warmup", "3"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle"
