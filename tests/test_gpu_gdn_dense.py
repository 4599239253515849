"""The dense-state comparator (the gated delta rule on a dense [d, 64] state that every
token updates) against the oracle's fp64 form. fp32 state on the GPU: max-abs 1e-4, the
fp32-state tolerance of the method itself."""
import numpy as np
import pytest
import torch

import oracle
import sparse_memory_linear_key_b300 as sdm

pytestmark = pytest.mark.gpu

ATOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _build():
    from sparse_memory_linear_key_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("B,T,d,io,with_s0", [(2, 300, 128, "bf16", False),
                                              (1, 257, 48, "f32", True),
                                              (3, 64, 2048, "bf16", True)])
def test_gdn_dense_matches_oracle(B, T, d, io, with_s0):
    W = 64
    g = torch.Generator().manual_seed(B * 1000 + T)
    cfg = sdm.make_cfg(d, 8, 16, W, io)
    dt = torch.bfloat16 if io == "bf16" else torch.float32
    # weights laid out as the addressing writes them: [B*T, 2, W], write then read
    wsel = torch.softmax(torch.randn(B * T, 2, W, generator=g) * 2, dim=-1).contiguous()
    v = torch.randn(B * T, d, generator=g).to(dt)
    alpha = torch.sigmoid(torch.randn(B * T, generator=g) + 3)
    beta = torch.sigmoid(torch.randn(B * T, generator=g))
    S0 = (torch.randn(B, d, W, generator=g) * 0.02) if with_s0 else None
    dw = wsel.cuda()
    y = torch.empty(B * T, d, device="cuda")
    S_out = torch.empty(B, d, W, device="cuda")
    sdm.sdm_gdn_dense_scan(cfg, dw, dw[:, 1], 2 * W, v.cuda(), alpha.cuda(), beta.cuda(), y, B, T,
                           S0=None if S0 is None else S0.cuda(), S_out=S_out)
    torch.cuda.synchronize()
    for b in range(B):
        sl = slice(b * T, (b + 1) * T)
        yr, Sr = oracle.gdn_dense(None if S0 is None else S0[b].numpy(), wsel[sl, 0].numpy(),
                                  wsel[sl, 1].numpy(), v[sl], alpha[sl].numpy(), beta[sl].numpy())
        assert np.abs(y[sl].cpu().numpy() - yr).max() <= ATOL, b
        assert np.abs(S_out[b].cpu().numpy() - Sr).max() <= ATOL, b


def test_gdn_dense_rejects_other_widths():
    cfg = sdm.make_cfg(64, 8, 16, 32, "bf16")
    x = torch.zeros(4, 64, device="cuda")
    with pytest.raises(sdm.SdmError):
        sdm.sdm_gdn_dense_scan(cfg, x, x, 64, x.to(torch.bfloat16), x[:, 0].contiguous(),
                               x[:, 0].contiguous(), x, 1, 4)
