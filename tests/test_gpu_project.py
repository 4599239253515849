"""The projections (row a1: "Write & Read", the token embedding is projected to write keys
and, separately, to read queries) on the hand-written GEMM, against the oracle's fp64
products rounded once, at the widths of the pages' layers (d = 2048 and 3840, key width
256) and token counts that take every path of the kernel: 256-column tiles over the
whole K (many tokens), 64-column tiles split along K over CTA pairs (few tokens: d = 2048
with 1 to 127 tokens, d = 3840 and d = 1280 with 64 and 96), 64-column tiles over the
whole K (129 and 300 tokens; a one-block K at d = 64), full and ragged 128-token tiles,
x copies of fewer rows than a tile, a single token."""
import numpy as np
import pytest
import torch

import oracle
import sparse_memory_linear_key_b300 as sdm
from tests import sdm_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    from sparse_memory_linear_key_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _weights(d, dk, seed):
    g = torch.Generator().manual_seed(seed)
    return {"W_qw": (torch.randn(d, dk, generator=g) / d ** 0.5).to(torch.bfloat16),
            "W_qr": (torch.randn(d, dk, generator=g) / d ** 0.5).to(torch.bfloat16),
            "W_v": (torch.randn(d, d, generator=g) / d ** 0.5).to(torch.bfloat16),
            "K1": torch.zeros(32, dk // 2, dtype=torch.bfloat16),
            "K2": torch.zeros(32, dk // 2, dtype=torch.bfloat16)}


@pytest.mark.parametrize("d,ntok", [(2048, 1), (2048, 5), (2048, 64), (2048, 127), (2048, 129),
                                    (2048, 300), (2048, 1500), (3840, 64), (3840, 2000),
                                    (64, 700), (1280, 96)])
def test_projection_against_oracle(d, ntok):
    dk = 256 if d >= 256 else 64
    cfg = sdm.make_cfg(d, 32, dk, 8, "bf16")
    p = _weights(d, dk, seed=d + ntok)
    pd = {k: v.cuda() for k, v in p.items()}
    x = torch.randn(ntok, d, generator=torch.Generator().manual_seed(ntok)).to(torch.bfloat16)
    q_w = torch.empty(ntok, dk, dtype=torch.bfloat16, device="cuda")
    q_r = torch.empty_like(q_w)
    v = torch.empty(ntok, d, dtype=torch.bfloat16, device="cuda")
    sdm.sdm_project(cfg, pd, x.cuda(), q_w, q_r, v)
    # the same shape twice gives the same bits
    q_w2 = torch.empty_like(q_w)
    sdm.sdm_project(cfg, pd, x.cuda(), q_w2, torch.empty_like(q_r), torch.empty_like(v))
    torch.cuda.synchronize()
    assert torch.equal(q_w, q_w2)
    rows = np.arange(ntok) if ntok <= 300 else np.sort(
        np.random.default_rng(0).choice(ntok, 200, replace=False))
    xr = x[torch.as_tensor(rows)]
    for out, w in ((q_w, "W_qw"), (q_r, "W_qr"), (v, "W_v")):
        ref = oracle.to_f64(oracle.project(xr, p[w]))
        got = oracle.to_f64(out[torch.as_tensor(rows, device="cuda")].cpu())
        assert tl.projection_ok(got, ref, oracle.to_f64(xr), oracle.to_f64(p[w])), (w, d, ntok)
