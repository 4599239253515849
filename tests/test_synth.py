"""The seeded input generator: deterministic, right shapes and distributions."""
import math

import torch

import synth


def test_deterministic_and_shapes():
    wl = synth.WORKLOADS["tiny-f32"]
    a, b = synth.make_params(wl), synth.make_params(wl)
    for k in a:
        assert torch.equal(a[k], b[k])
    assert a["W_qw"].shape == (64, 64) and a["W_v"].shape == (64, 64)
    assert a["K1"].shape == (32, 32) and a["M0"].shape == (1024, 64)
    t = synth.make_tokens(wl)
    assert t["x"].shape == (1, 256, 64) and t["alpha"].shape == (1, 256)
    assert t["x"].dtype == torch.float32


def test_distributions():
    wl = synth.Workload("dist", B=2, T=2048, d=256, n=64, dk=64, W=8, dtype="bf16", seed=7)
    p = synth.make_params(wl)
    t = synth.make_tokens(wl)
    assert p["W_qw"].dtype == torch.bfloat16
    assert abs(p["W_v"].float().std().item() - 1 / math.sqrt(256)) < 2e-3
    assert abs(p["K1"].float().std().item() - 1 / math.sqrt(32)) < 1e-2
    assert abs(p["M0"].float().std().item() - 0.02) < 1e-3
    assert abs(t["x"].float().std().item() - 1.0) < 1e-2
    a, b = t["alpha"], t["beta"]
    assert (a > 0).all() and (a < 1).all() and (b > 0).all() and (b < 1).all()
    # alpha = sigmoid(N(3,1)): mean about 0.93; beta = sigmoid(N(0,1)): mean 0.5
    assert abs(a.mean().item() - 0.93) < 0.02 and abs(b.mean().item() - 0.5) < 0.02


def test_pool_and_pattern_injection():
    wl = synth.Workload("pool", B=2, T=100, d=32, n=16, dk=16, W=8, dtype="bf16", seed=9,
                        pool_frac=0.3, pool_size=4)
    pool = synth.make_pool(wl)
    frac = pool["mask"].float().mean().item()
    assert 0.2 < frac < 0.4
    qw = torch.zeros(2, 100, 16, dtype=torch.bfloat16)
    qr = torch.zeros_like(qw)
    v = torch.zeros(2, 100, 32, dtype=torch.bfloat16)
    synth.inject_queries(wl, qw, qr, v, pool=pool)
    m = pool["mask"]
    assert torch.equal(qw[m], pool["pool"][pool["pick_w"][m]])
    assert (qw[~m] == 0).all()
    wl2 = synth.Workload("pat", B=1, T=64, d=32, n=16, dk=16, W=8, dtype="bf16", seed=9,
                         pattern_len=4, pattern_write_at=10, pattern_read_at=50)
    pat = synth.make_pattern(wl2)
    qw = torch.zeros(1, 64, 16, dtype=torch.bfloat16)
    qr = torch.zeros_like(qw)
    v = torch.zeros(1, 64, 32, dtype=torch.bfloat16)
    synth.inject_queries(wl2, qw, qr, v, pattern=pat)
    assert torch.equal(qw[0, 10:14], pat["p"]) and torch.equal(qr[0, 50:54], pat["p"])
    assert torch.equal(v[0, 10:14], pat["v"])
