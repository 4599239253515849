"""Replicas: `bench.py --gpus N` runs one replica of the layer per rank (sequences are
independent, there is no data-path collective). Two ranks here, as processes with a
gloo process group on 127.0.0.1 for the barriers (on the CPU), both on this GPU: neither
waits on the other's kernels, so they may run in any order or overlap. Each runs the whole
prefill (sdm_prefill_m0: projections, addressing, first touch, scan, fill) on the same
seeded batch, and both must give the bits of a run of that batch in this process: no
state of the library (the fork's side stream, cached tensor maps, the first-touch
table) leaks between callers."""
import os
import socket
import subprocess
import sys

import pytest
import torch

import sparse_memory_linear_key_b300 as sdm
import synth
from tests import sdm_testlib as tl

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# slot vectors of three row blocks (the last partial), several sequences, enough tokens
# for the many-token addressing
WL = synth.Workload("replica", B=3, T=300, d=1280, n=40, dk=64, W=16, dtype="bf16", seed=91)

_RANK = r'''
import os, sys
sys.path.insert(0, sys.argv[1])
import torch
import torch.distributed as dist
from tests.test_gpu_replicas import run_prefill
# gloo on the CPU for the barriers: the two ranks share this GPU, so no collective may
# run there (kernels of two processes waiting on each other)
dist.init_process_group("gloo")
rank = dist.get_rank()
torch.cuda.set_device(0)
dist.barrier()
y, banks, st = run_prefill()
dist.barrier()
torch.save({"y": y.cpu(), "banks": banks.cpu(), "status": st}, sys.argv[2] % rank)
dist.destroy_process_group()
print("rank %d done" % rank, flush=True)
'''


def run_prefill():
    cfg = tl.cfg_of(WL)
    p = tl.to_dev(synth.make_params(WL))
    tok = synth.make_tokens(WL)
    x, al, be = tok["x"].cuda(), tok["alpha"].cuda(), tok["beta"].cuda()
    banks = torch.empty(WL.B, WL.N, WL.d, dtype=WL.torch_dtype, device="cuda")
    y = torch.empty(WL.B, WL.T, WL.d, device="cuda")
    ws = sdm.alloc_workspace(sdm.prefill_m0_workspace_bytes(cfg, WL.B, WL.T))
    st = sdm.new_status()
    sdm.sdm_prefill_m0(cfg, p, p["M0"], x, al, be, banks, y, ws, st)
    torch.cuda.synchronize()
    return y, banks, sdm.read_status(st)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.fixture(scope="module", autouse=True)
def _build():
    from sparse_memory_linear_key_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_two_replicas_match_one_process(tmp_path):
    y_ref, banks_ref, st = run_prefill()
    assert st == 0
    port = _free_port()
    out = str(tmp_path / "rank%d.pt")
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK="0", WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK, ROOT, out], cwd=ROOT, env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    try:
        for p in procs:
            o, e = p.communicate(timeout=600)
            assert p.returncode == 0, (o, e[-3000:])
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    for rank in range(2):
        r = torch.load(out % rank)
        assert r["status"] == 0
        assert torch.equal(r["y"], y_ref.cpu()), rank
        assert torch.equal(r["banks"], banks_ref.cpu()), rank


def test_concurrent_calls_from_two_host_threads():
    """sdm_prefill_m0 forks its first-touch table and fill onto a side stream the library
    owns (one a device, shared by all callers) and joins it back. Two host threads calling
    it at once on their own streams, each with its own buffers, must each get the bits
    of a call made alone: the lock keeps one thread's fork-to-join sequence whole, and
    the events keep each call's work ordered on the device."""
    import threading
    y_ref, banks_ref, st = run_prefill()
    assert st == 0
    cfg = tl.cfg_of(WL)
    p = tl.to_dev(synth.make_params(WL))
    tok = synth.make_tokens(WL)
    x, al, be = tok["x"].cuda(), tok["alpha"].cuda(), tok["beta"].cuda()
    out = [None, None]
    err = []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                banks = torch.empty(WL.B, WL.N, WL.d, dtype=WL.torch_dtype, device="cuda")
                y = torch.empty(WL.B, WL.T, WL.d, device="cuda")
                ws = sdm.alloc_workspace(sdm.prefill_m0_workspace_bytes(cfg, WL.B, WL.T))
                stt = sdm.new_status()
                for _ in range(4):
                    sdm.sdm_prefill_m0(cfg, p, p["M0"], x, al, be, banks, y, ws, stt, stream=s)
            s.synchronize()
            out[i] = (y.cpu(), banks.cpu(), sdm.read_status(stt))
        except Exception as e:  # pragma: no cover - reported below
            err.append(repr(e))

    torch.cuda.synchronize()
    th = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not err, err
    for i in range(2):
        y, banks, st_i = out[i]
        assert st_i == 0
        assert torch.equal(y, y_ref.cpu()), i
        assert torch.equal(banks, banks_ref.cpu()), i
