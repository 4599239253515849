"""The N > 1 host path of bench.py on CPU, as world-size-2 gloo process groups on
127.0.0.1: one process per rank, rendezvous from RANK / WORLD_SIZE / MASTER_*.

The layer runs as replicas (sequences are independent; there is no data-path
collective), so what N > 1 adds is host logic: the process group, the barriers around
the timed region, the max of the per-rank times, and rank 0 alone printing the line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_HELPER = r'''
import sys, types
sys.path.insert(0, sys.argv[1])
import bench
world, rank, local = bench.dist_setup(types.SimpleNamespace())
assert world == 2 and local == rank
bench.barrier(world)
t = bench.max_over_ranks(world, 1.5 + rank)      # per-rank times 1.5 and 2.5
assert t == 2.5, t
print("rank %d max %.1f" % (rank, t), flush=True)
bench.barrier(world)
'''


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(argv, timeout):
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="",
                   OMP_NUM_THREADS="2")
        procs.append(subprocess.Popen(argv, cwd=ROOT, env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=timeout)
            outs.append((p.returncode, out, err))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    return outs


def test_gloo_barrier_and_max_over_ranks():
    outs = _run_ranks([sys.executable, "-c", _HELPER, ROOT], timeout=120)
    for rank, (rc, out, err) in enumerate(outs):
        assert rc == 0, err[-2000:]
        assert "rank %d max 2.5" % rank in out


def test_reference_arm_prints_once_under_two_ranks():
    """--impl reference under two ranks: rank 0 times the oracle and prints one JSON line,
    rank 1 exits 0 without work."""
    outs = _run_ranks([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                       "--steps", "1", "--warmup", "0"], timeout=600)
    lines = []
    for rc, out, err in outs:
        assert rc == 0, err[-2000:]
        lines += [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    r = json.loads(lines[0])
    assert r["impl"] == "reference" and r["n_gpus"] == 2 and r["value"] > 0
    assert outs[1][1].strip() == ""
