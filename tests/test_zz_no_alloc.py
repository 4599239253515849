"""sdm_scan_noalloc: the scan for callers that cannot allocate device memory (a plugin
whose host application owns every device allocation, a latency-critical loop where
cudaMalloc would synchronise the device). It keeps its scratch in a library-owned
device array instead of a caller workspace, and must give what sdm_scan gives.

This file is collected last on purpose, so that a run stopping at the first failure
has already run every other test; it also passes when run alone."""
import ctypes

import numpy as np
import pytest
import torch

import sparse_memory_linear_key_b300 as sdm


def _case(seed, B, T, N, W, d):
    rng = np.random.default_rng(seed)
    n = int(round(N ** 0.5))
    cfg = sdm.make_cfg(d, n, 16, W, "bf16")
    ntok = B * T
    idx = np.zeros((ntok, 2, W), dtype=np.int32)
    for t in range(ntok):
        idx[t, 0] = np.sort(rng.choice(N, W, replace=False))
        idx[t, 1] = np.sort(rng.choice(N, W, replace=False))
    wts = (rng.random((ntok, 2, W)) + 0.05).astype(np.float32)
    wts /= wts.sum(-1, keepdims=True)
    g = torch.Generator().manual_seed(seed)
    v = torch.randn(ntok, d, generator=g).to(torch.bfloat16)
    M0 = (torch.randn(N, d, generator=g) * 0.1).to(torch.bfloat16)
    alpha = torch.from_numpy(rng.uniform(0.5, 1.0, ntok).astype(np.float32))
    beta = torch.from_numpy(rng.uniform(0.0, 1.0, ntok).astype(np.float32))
    dev = "cuda"
    return (cfg, torch.from_numpy(idx).to(dev), torch.from_numpy(wts).to(dev), v.to(dev),
            alpha.to(dev), beta.to(dev), M0.to(dev), B, T)


def _run(entry, case):
    cfg, idx, wts, v, alpha, beta, M0, B, T = case
    banks = torch.empty((B,) + tuple(M0.shape), dtype=M0.dtype, device="cuda")
    sdm.sdm_init_bank(cfg, M0, banks)
    y = torch.empty(B * T, cfg.d, device="cuda")
    st = sdm.new_status()
    if entry == "noalloc":
        sdm.sdm_scan_noalloc(cfg, idx, wts, v, alpha, beta, banks, y, B, T, st)
    else:
        ws = sdm.alloc_workspace(sdm.scan_workspace_bytes(cfg, B, T))
        sdm.sdm_scan(cfg, idx, wts, v, alpha, beta, banks, y, B, T, ws, st)
    torch.cuda.synchronize()
    return banks, y, int(st.item())


@pytest.mark.gpu
def test_noalloc_scan_matches_sdm_scan_twice():
    """Two calls in a row (a large one, then a smaller one that leaves the first call's
    contents in the tail of the shared array) each give exactly the bits of sdm_scan on
    the same inputs: both run the same kernels on the same scratch layout, so y and the
    banks must be equal, not merely close. The device's free memory is the same before
    and after the second call (the first one may load the library's device code, which
    brings the array with it; the reference calls run first, so that loading a kernel's
code is not counted either)."""
    from sparse_memory_linear_key_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cases = [_case(1, B=3, T=400, N=256, W=64, d=48), _case(2, B=2, T=97, N=64, W=8, d=32)]
    want = [_run("ws", c) for c in cases]    # (also loads every kernel the calls use)
    bufs = []
    for c in cases:
        cfg, idx, wts, v, alpha, beta, M0, B, T = c
        banks = torch.empty((B,) + tuple(M0.shape), dtype=M0.dtype, device="cuda")
        sdm.sdm_init_bank(cfg, M0, banks)
        bufs.append((banks, torch.empty(B * T, cfg.d, device="cuda"), sdm.new_status()))
    torch.cuda.synchronize()
    free = []
    for c, (banks, y, st) in zip(cases, bufs):       # two calls in a row
        cfg, idx, wts, v, alpha, beta, M0, B, T = c
        free.append(torch.cuda.mem_get_info()[0])
        sdm.sdm_scan_noalloc(cfg, idx, wts, v, alpha, beta, banks, y, B, T, st)
        torch.cuda.synchronize()
    free.append(torch.cuda.mem_get_info()[0])
    assert free[2] == free[1], free
    for (ba, ya, sa), (bb, yb, sb) in zip(bufs, want):
        assert int(sa.item()) == 0 and sb == 0
        assert torch.equal(ya, yb)
        assert torch.equal(ba, bb)


def test_noalloc_rejects_oversize_on_the_host():
    """More than SDM_SCAN_NOALLOC_MAX_BYTES of scratch (w = 64, d = 2048 bf16: more than
    27592 tokens) is refused with SDM_EWORKSPACE before any device work."""
    from sparse_memory_linear_key_b300 import build
    build.build()
    L = sdm.lib()
    cfg = sdm.make_cfg(2048, 480, 256, 64, "bf16")
    P = ctypes.c_void_p
    t_max = 27592
    assert sdm.scan_min_workspace_bytes(cfg, 1, t_max) <= sdm.SCAN_NOALLOC_MAX_BYTES
    assert sdm.scan_min_workspace_bytes(cfg, 1, t_max + 1) > sdm.SCAN_NOALLOC_MAX_BYTES
    rc = L.sdm_scan_noalloc(ctypes.byref(cfg), P(256), P(256), P(256), P(256), P(256), P(256),
                            P(256), 1, t_max + 1, P(256), None)
    assert rc == sdm.SDM_EWORKSPACE
    rc = L.sdm_scan_noalloc(ctypes.byref(cfg), P(256), P(256), P(256), P(256), P(256), P(256),
                            P(256), 4, 9000, P(256), None)
    assert rc == sdm.SDM_EWORKSPACE
    assert L.sdm_scan_noalloc(ctypes.byref(cfg), None, None, None, None, None, None, None, 0, 5,
                              None, None) == sdm.SDM_OK
