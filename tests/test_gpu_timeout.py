"""Failure detection of the recurrence on the GPU, without a fault: every wait inside the
scan kernel is bounded; when one runs out the kernel records SDM_ETIMEOUT in the device
status word, raises an abort flag that every warp of every block watches, lets the copies
it started land, and returns -- the device stays usable.

The wait is made to run out by withholding one work item (sdm_scan_run_diag): the kernel
claims it and drops it, so its progress flag is never raised and the next token, which
writes the same slots, waits for it until a short bound (a few hundred microseconds)
ends the wait. Nothing here faults, traps or hangs the device: the dropped item touches
no memory, and each wait -- including the waits for copies in flight on the way out --
ends by itself."""
import numpy as np
import pytest
import torch

import oracle
import sparse_memory_linear_key_b300 as sdm
from tests import sdm_testlib as tl

pytestmark = pytest.mark.gpu

SHORT = 400_000          # SM clock cycles: ~0.2 ms at 2 GHz


@pytest.fixture(scope="module", autouse=True)
def _build():
    from sparse_memory_linear_key_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _case(T=8, W=8, N=64, d=64, seed=0, same_slots=True):
    rng = np.random.default_rng(seed)
    idx = np.zeros((T, 2, W), np.int32)
    for t in range(T):
        if same_slots:
            idx[t, 0] = np.arange(W)                  # every token writes slots 0..W-1
            idx[t, 1] = np.arange(W, 2 * W)
        else:
            idx[t, 0] = np.sort(rng.choice(N, W, replace=False))
            idx[t, 1] = np.sort(rng.choice(N, W, replace=False))
    wts = (rng.random((T, 2, W)) + 0.05).astype(np.float32)
    wts /= wts.sum(-1, keepdims=True)
    g = torch.Generator().manual_seed(seed)
    v = torch.randn(T, d, generator=g).to(torch.bfloat16)
    M0 = (torch.randn(N, d, generator=g) * 0.1).to(torch.bfloat16)
    al = torch.from_numpy(rng.uniform(0.5, 1.0, T).astype(np.float32))
    be = torch.from_numpy(rng.uniform(0.0, 1.0, T).astype(np.float32))
    return idx, wts, v, M0, al, be


@pytest.mark.parametrize("ring", [True, False])
def test_withheld_dependency_times_out_and_device_stays_usable(ring):
    T, W, N, d = 8, 8, 64, 64
    cfg = sdm.make_cfg(d, 8, 16, W, "bf16")
    idx, wts, v, M0, al, be = _case(T, W, N, d)
    dev = "cuda"
    idx_d, wts_d = torch.from_numpy(idx).to(dev), torch.from_numpy(wts).to(dev)
    v_d, al_d, be_d = v.to(dev), al.to(dev), be.to(dev)
    banks = torch.empty(1, N, d, dtype=torch.bfloat16, device=dev)
    sdm.sdm_init_bank(cfg, M0.to(dev), banks)
    y = torch.empty(T, d, device=dev)
    nbytes = sdm.scan_workspace_bytes(cfg, 1, T) if ring else sdm.scan_min_workspace_bytes(cfg, 1, T)
    ws = sdm.alloc_workspace(nbytes)
    st = sdm.new_status()
    sdm.sdm_scan_prepare(cfg, idx_d, 1, T, ws, st)
    # token 0 (item 0: one sequence, one row block) is withheld; token 1 writes the same
    # slots, so its references wait for token 0's progress flag, which nobody raises
    sdm.sdm_scan_run_diag(cfg, idx_d, wts_d, v_d, al_d, be_d, banks, y, 1, T, ws, SHORT, 0, st)
    torch.cuda.synchronize()
    assert sdm.read_status(st) == sdm.SDM_ETIMEOUT

    # the same call with nothing withheld (and the default bound) completes...
    st2 = sdm.new_status()
    sdm.sdm_init_bank(cfg, M0.to(dev), banks)
    sdm.sdm_scan_prepare(cfg, idx_d, 1, T, ws, st2)
    sdm.sdm_scan_run_diag(cfg, idx_d, wts_d, v_d, al_d, be_d, banks, y, 1, T, ws, 0, -1, st2)
    torch.cuda.synchronize()
    assert sdm.read_status(st2) == 0
    # ... and matches the oracle, so the context and the kernel are sound after the abort
    M = np.ascontiguousarray(oracle.storage(M0)[0].copy())
    yr = oracle.scan(M, oracle.storage(v)[0], al.numpy().astype(np.float64),
                     be.numpy().astype(np.float64), idx[:, 0], wts[:, 0].astype(np.float64),
                     idx[:, 1], wts[:, 1].astype(np.float64))
    assert tl.state_ok("bf16", y.cpu().numpy(), yr)[0]
    assert tl.state_ok("bf16", oracle.to_f64(banks[0].cpu()), oracle.to_f64(M))[0]


def test_normal_scan_after_a_timeout_passes_parity():
    """A plain sdm_scan of random slot sets on the same device, after an aborted run."""
    T, W, N, d = 8, 8, 64, 64
    cfg = sdm.make_cfg(d, 8, 16, W, "bf16")
    idx, wts, v, M0, al, be = _case(T, W, N, d)
    dev = "cuda"
    ws = sdm.alloc_workspace(sdm.scan_workspace_bytes(cfg, 1, T))
    st = sdm.new_status()
    banks = torch.empty(1, N, d, dtype=torch.bfloat16, device=dev)
    y = torch.empty(T, d, device=dev)
    idx_d = torch.from_numpy(idx).to(dev)
    sdm.sdm_scan_prepare(cfg, idx_d, 1, T, ws, st)
    sdm.sdm_scan_run_diag(cfg, idx_d, torch.from_numpy(wts).to(dev), v.to(dev), al.to(dev),
                          be.to(dev), banks, y, 1, T, ws, SHORT, 0, st)
    torch.cuda.synchronize()
    assert sdm.read_status(st) == sdm.SDM_ETIMEOUT
    idx2, wts2, v2, M02, al2, be2 = _case(T=300, W=16, N=256, d=96, seed=5, same_slots=False)
    cfg2 = sdm.make_cfg(96, 16, 16, 16, "bf16")
    banks2, y2, status = tl.run_scan_only(cfg2, M02, torch.from_numpy(idx2), torch.from_numpy(wts2),
                                          v2, al2, be2, 1, 300)
    assert status == 0
    M = np.ascontiguousarray(oracle.storage(M02)[0].copy())
    yr = oracle.scan(M, oracle.storage(v2)[0], al2.numpy().astype(np.float64),
                     be2.numpy().astype(np.float64), idx2[:, 0], wts2[:, 0].astype(np.float64),
                     idx2[:, 1], wts2[:, 1].astype(np.float64))
    assert tl.state_ok("bf16", y2.cpu().numpy(), yr)[0]
    assert tl.state_ok("bf16", oracle.to_f64(banks2[0].cpu()), oracle.to_f64(M))[0]
