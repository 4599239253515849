"""Slot-access statistics against the oracle's set definitions (integer work: exact).
The pages' diagnostic ("Memory Access Patterns on a Needle-in-a-Haystack Task"):
per-slot write / read counts over a token range and the write-read bucket overlap."""
import numpy as np
import pytest
import torch

import oracle
import sparse_memory_linear_key_b300 as sdm
import synth
from tests import sdm_testlib as tl
from tests.test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from sparse_memory_linear_key_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _random_idx(B, T, W, N, seed, bad=False):
    rng = np.random.default_rng(seed)
    idx = np.stack([np.stack([np.sort(rng.choice(N // 2, W, replace=False)) for _ in range(2)])
                    for _ in range(B * T)]).astype(np.int32)
    if bad:   # a few ids out of range: not counted
        idx[3, 0, 0] = N + 5
        idx[7, 1, 2] = -1
    return idx


@pytest.mark.parametrize("B,T,W,N,seed", [(1, 64, 8, 1024, 1), (3, 257, 16, 1600, 2),
                                          (2, 100, 64, 230400, 3)])
def test_slot_counts_and_overlap_match_oracle(B, T, W, N, seed):
    n = int(round(N ** 0.5))
    cfg = sdm.make_cfg(64, n, 64, W, "bf16")
    idx = _random_idx(B, T, W, N, seed, bad=True)
    d_idx = torch.from_numpy(idx).cuda()
    counts = torch.empty(B, N, dtype=torch.int32, device="cuda")
    for kind, t0, t1 in ((0, 0, T), (1, T // 3, T), (0, 5, 5)):
        sdm.sdm_slot_counts(cfg, d_idx, B, T, kind, t0, t1, counts)
        want = oracle.slot_counts(idx, B, T, N, kind, t0, t1)
        assert np.array_equal(counts.cpu().numpy(), want), (kind, t0, t1)
    out = torch.empty(B, 3, dtype=torch.int32, device="cuda")
    ws = sdm.alloc_workspace(sdm.slot_overlap_workspace_bytes(cfg, B))
    for w0, w1, r0, r1 in ((0, T // 2, T // 2, T), (0, T, 0, T), (3, 3, 0, T), (T - 1, T, 0, 1)):
        sdm.sdm_slot_overlap(cfg, d_idx, B, T, w0, w1, r0, r1, out, ws)
        want = oracle.slot_overlap(idx, B, T, N, w0, w1, r0, r1)
        assert np.array_equal(out.cpu().numpy(), want), (w0, w1, r0, r1)


def test_slot_overlap_of_a_repeated_pattern():
    """The needle shape on real addressing: tokens whose read queries repeat earlier write
    queries read exactly the slots those tokens wrote (full overlap), tokens drawn
    independently share almost none."""
    wl = SMALL["w64-small"]
    cfg = tl.cfg_of(wl)
    L, wa, ra = 8, 20, 250

    def hook(q_w, q_r, v):
        q_w = q_w.view(wl.B, wl.T, -1)
        q_r = q_r.view(wl.B, wl.T, -1)
        q_r[:, ra:ra + L] = q_w[:, wa:wa + L]

    out = tl.run_staged(wl, synth.make_params(wl), synth.make_tokens(wl), query_hook=hook)
    assert out["status"] == 0
    o = torch.empty(wl.B, 3, dtype=torch.int32, device="cuda")
    ws = sdm.alloc_workspace(sdm.slot_overlap_workspace_bytes(cfg, wl.B))
    sdm.sdm_slot_overlap(cfg, out["idx"], wl.B, wl.T, wa, wa + L, ra, ra + L, o, ws)
    o = o.cpu().numpy()
    assert np.all(o[:, 2] == o[:, 0]) and np.all(o[:, 2] == o[:, 1])
    o2 = torch.empty(wl.B, 3, dtype=torch.int32, device="cuda")
    sdm.sdm_slot_overlap(cfg, out["idx"], wl.B, wl.T, wa, wa + L, 100, 100 + L, o2, ws)
    o2 = o2.cpu().numpy()
    assert np.all(o2[:, 2] < o2[:, 1] // 4)


def test_slot_stats_reject_bad_windows():
    cfg = sdm.make_cfg(64, 32, 64, 8, "bf16")
    idx = torch.zeros(4, 2, 8, dtype=torch.int32, device="cuda")
    counts = torch.empty(1, 1024, dtype=torch.int32, device="cuda")
    with pytest.raises(sdm.SdmError):
        sdm.sdm_slot_counts(cfg, idx, 1, 4, 0, 2, 5, counts)
    with pytest.raises(sdm.SdmError):
        sdm.sdm_slot_counts(cfg, idx, 1, 4, 2, 0, 4, counts)
