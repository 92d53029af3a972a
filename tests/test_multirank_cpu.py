"""bench.py's multi-rank path on the CPU (gloo, two ranks, 127.0.0.1).

The verify call has no collective (replicas only); what runs on several ranks
is the bench's timing: the slowest rank's time per call is the job's, and the
reference arm runs on rank 0 alone while the other ranks exit without work.
"""
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


def _rank_main(rank, world, port, out_path):
    sys.path.insert(0, ROOT)
    import torch.distributed as tdist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + rank * 2.5, world)
        tdist.barrier()
        with open("%s.%d" % (out_path, rank), "w") as fh:
            fh.write(repr(got))
    finally:
        tdist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    out = str(tmp_path / "r")
    mp.spawn(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True)
    assert [float(open("%s.%d" % (out, r)).read()) for r in range(2)] == [12.5, 12.5]


def test_reference_arm_two_ranks_prints_once():
    pytest.importorskip("torch")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "chain9_p256", "--cpu-budget-s", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
