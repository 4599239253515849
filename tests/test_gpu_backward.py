"""Backward of the recurrence (the gated-delta write and the weighted read) against the
oracle's autograd of the per-token definition, teacher-forced with the CUDA path's own
addressing. Also exact: after the backward walk the banks are the initial banks again,
bit for bit (the tape restores every write)."""
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


def rel_err(got, want):
    return float(np.abs(np.asarray(got, np.float64) - want).max() / max(np.abs(want).max(), 1e-30))


def _walk_back_and_check(wl, cfg, M0, idx, wsel, v, al, be, tol, name):
    """Forward with a tape from banks = M0, the backward walk, then every gradient against
    the oracle's autograd, sequence by sequence."""
    B, T, d, N, W = wl.B, wl.T, wl.d, wl.N, wl.W
    dt = wl.torch_dtype
    banks = torch.empty(B, N, d, dtype=dt, device="cuda")
    sdm.sdm_init_bank(cfg, M0.cuda(), banks)
    banks0 = banks.clone()
    y = torch.empty(B * T, d, device="cuda")
    tape = torch.empty(B * T, W, d, dtype=dt, device="cuda")
    ws = sdm.alloc_workspace(sdm.scan_workspace_bytes(cfg, B, T))
    st = sdm.new_status()
    sdm.sdm_scan_prepare(cfg, idx, B, T, ws, st)
    sdm.sdm_scan_run_train(cfg, idx, wsel, v, al, be, banks, y, B, T, ws, tape, st)
    g = torch.Generator().manual_seed(7)
    dy = torch.randn(B * T, d, generator=g)
    dMf = torch.randn(B, N, d, generator=g) * 0.1
    dbank = dMf.cuda()
    dv = torch.empty(B * T, d, device="cuda")
    dal = torch.empty(B * T, device="cuda")
    dbe = torch.empty(B * T, device="cuda")
    dw = torch.empty(B * T, 2, W, device="cuda")
    wsb = sdm.alloc_workspace(sdm.scan_backward_workspace_bytes(cfg, B, T))
    sdm.sdm_scan_backward(cfg, idx, wsel, v, al, be, tape, banks, dy.cuda(), dbank, dv, dal, dbe,
                          dw, B, T, wsb)
    torch.cuda.synchronize()
    assert sdm.read_status(st) == 0
    assert torch.equal(banks, banks0)     # walked back to the initial state, exactly
    idx_h, w_h = idx.cpu().numpy(), wsel.cpu().numpy().astype(np.float64)
    type_ = oracle.BF16 if wl.dtype == "bf16" else oracle.F32
    for b in range(B):
        sl = slice(b * T, (b + 1) * T)
        ref = oracle.scan_backward(oracle.to_f64(M0), v[sl].cpu(), al[sl].cpu().numpy(),
                                   be[sl].cpu().numpy(), idx_h[sl, 0], w_h[sl, 0], idx_h[sl, 1],
                                   w_h[sl, 1], dy[sl].numpy(), dMf[b].numpy(), type_=type_)
        checks = [("dM_init", dbank[b].cpu().numpy(), ref["dM_init"]),
                  ("dv", dv[sl].cpu().numpy(), ref["dv"]),
                  ("dalpha", dal[sl].cpu().numpy(), ref["dalpha"]),
                  ("dbeta", dbe[sl].cpu().numpy(), ref["dbeta"]),
                  ("dk", dw[sl, 0].cpu().numpy(), ref["dk"]),
                  ("dr", dw[sl, 1].cpu().numpy(), ref["dr"])]
        for what, got, want in checks:
            e = rel_err(got, want)
            assert e <= tol, (name, b, what, e)


@pytest.mark.parametrize("name,tol", [("tiny-f32", 1e-4), ("ragged-f32", 1e-4),
                                      ("ragged-bf16", 2e-2), ("w64-small", 2e-2)])
def test_scan_backward_matches_autograd(name, tol):
    wl = SMALL[name]
    cfg = tl.cfg_of(wl)
    p = synth.make_params(wl)
    tok = synth.make_tokens(wl)
    out = tl.run_staged(wl, p, tok)       # the CUDA path's addressing and v
    _walk_back_and_check(wl, cfg, p["M0"], out["idx"], out["wsel"], out["v"],
                         out["alpha"].reshape(-1), out["beta"].reshape(-1), tol, name)


@pytest.mark.parametrize("dtype,W,d,tol", [("f32", 8, 80, 1e-4), ("bf16", 16, 144, 2e-2),
                                           ("bf16", 64, 64, 2e-2)])
def test_scan_backward_crowded_slots(dtype, W, d, tol):
    """Every slot drawn from a pool of 2W (offset into the bank), so consecutive tokens
    share most of their slots and most write slots are read by their own token too: the
    values the walk takes over from the token after it, and the reads folded into the
    write, are exercised on nearly every token. d = 80 and 144 leave a partial row block."""
    wl = synth.Workload("crowded", B=2, T=64, d=d, n=W, dk=16, W=W, dtype=dtype, seed=5)
    cfg = tl.cfg_of(wl)
    B, T, N = wl.B, wl.T, wl.N
    g = torch.Generator().manual_seed(11)
    pool, base = 2 * W, N - 2 * W - 3
    idx = torch.stack([torch.randperm(pool, generator=g)[:W] + base for _ in range(B * T * 2)])
    idx = idx.view(B * T, 2, W).to(torch.int32)
    w = torch.rand(B * T, 2, W, generator=g) + 0.05
    w = w / w.sum(-1, keepdim=True)
    v = torch.randn(B * T, d, generator=g).to(wl.torch_dtype)
    al = torch.rand(B * T, generator=g) * 0.5 + 0.5
    be = torch.rand(B * T, generator=g)
    M0 = synth.make_params(wl)["M0"]
    _walk_back_and_check(wl, cfg, M0, idx.cuda(), w.cuda(), v.cuda(), al.cuda(), be.cuda(), tol,
                         f"crowded-{dtype}-w{W}")


def test_scan_backward_from_m0_restores_m0():
    """The forward from M0 without a copy (first touch) also records its tape; walking
    back leaves every bank equal to M0."""
    wl = SMALL["n480-small-d"]
    cfg = tl.cfg_of(wl)
    p = synth.make_params(wl)
    tok = synth.make_tokens(wl)
    out = tl.run_staged(wl, p, tok)
    B, T, d, N, W = wl.B, wl.T, wl.d, wl.N, wl.W
    idx, wsel, v = out["idx"], out["wsel"], out["v"]
    al, be = out["alpha"].reshape(-1), out["beta"].reshape(-1)
    M0 = p["M0"].cuda()
    banks = torch.full((B, N, d), float("nan"), dtype=wl.torch_dtype, device="cuda")
    fw = torch.empty(B, N, dtype=torch.int32, device="cuda")
    ws = sdm.alloc_workspace(sdm.scan_workspace_bytes(cfg, B, T))
    st = sdm.new_status()
    tape = torch.empty(B * T, W, d, dtype=wl.torch_dtype, device="cuda")
    y = torch.empty(B * T, d, device="cuda")
    sdm.sdm_first_touch(cfg, idx, B, T, fw)
    sdm.sdm_scan_prepare(cfg, idx, B, T, ws, st)
    sdm.sdm_scan_run_train(cfg, idx, wsel, v, al, be, banks, y, B, T, ws, tape, st, M0=M0,
                           first_write=fw)
    sdm.sdm_fill_untouched(cfg, M0, fw, banks, B, T)
    assert torch.equal(y, out["y"])        # the same forward as the copy path
    dbank = torch.zeros(B, N, d, device="cuda")
    z = torch.empty(B * T, device="cuda")
    sdm.sdm_scan_backward(cfg, idx, wsel, v, al, be, tape, banks, torch.ones(B * T, d, device="cuda"),
                          dbank, torch.empty(B * T, d, device="cuda"), z, torch.empty_like(z),
                          torch.empty(B * T, 2, W, device="cuda"), B, T,
                          sdm.alloc_workspace(sdm.scan_backward_workspace_bytes(cfg, B, T)))
    torch.cuda.synchronize()
    assert sdm.read_status(st) == 0
    for b in range(B):
        assert torch.equal(banks[b], M0)


@pytest.mark.parametrize("name", ["tiny-f32", "w64-small", "n480-small-d", "n480-full-tiles"])
def test_address_backward_matches_autograd(name):
    """dq and dK from the selection-weight gradients, the kept slots fixed, against the
    oracle's autograd of the softmax of the kept combined scores (the oracle scores the
    CUDA path's own query bits)."""
    wl = SMALL[name]
    cfg = tl.cfg_of(wl)
    p = synth.make_params(wl)
    out = tl.run_staged(wl, p, synth.make_tokens(wl))
    ntok, W, n, dk = wl.B * wl.T, wl.W, wl.n, wl.dk
    g = torch.Generator().manual_seed(11)
    dw = torch.randn(ntok, 2, W, generator=g)
    dq_w = torch.empty(ntok, dk, device="cuda")
    dq_r = torch.empty_like(dq_w)
    dK1 = torch.empty(n, dk // 2, device="cuda")
    dK2 = torch.empty_like(dK1)
    ws = sdm.alloc_workspace(sdm.address_backward_workspace_bytes(cfg, ntok))
    pd = tl.to_dev(p)
    sdm.sdm_address_backward(cfg, pd["K1"], pd["K2"], out["q_w"], out["q_r"], out["idx"], out["wsel"],
                             dw.cuda(), dq_w, dq_r, dK1, dK2, ws)
    torch.cuda.synchronize()
    idx = out["idx"].cpu().numpy()
    wsel = out["wsel"].cpu().numpy()
    dK1r = np.zeros((n, dk // 2))
    dK2r = np.zeros((n, dk // 2))
    for kind, q, got in ((0, out["q_w"], dq_w), (1, out["q_r"], dq_r)):
        w, dq, k1, k2 = oracle.address_backward(q.cpu(), p["K1"], p["K2"], idx[:, kind],
                                                dw[:, kind].numpy())
        assert np.abs(w - wsel[:, kind]).max() <= 1e-5
        assert rel_err(got.cpu().numpy(), dq) <= 1e-4, (name, kind)
        dK1r += k1
        dK2r += k2
    assert rel_err(dK1.cpu().numpy(), dK1r) <= 1e-4, name
    assert rel_err(dK2.cpu().numpy(), dK2r) <= 1e-4, name


@pytest.mark.parametrize("name", ["tiny-f32", "w64-small"])
def test_project_backward_matches_oracle(name):
    wl = SMALL[name]
    cfg = tl.cfg_of(wl)
    p = synth.make_params(wl)
    x = synth.make_tokens(wl)["x"].reshape(-1, wl.d)
    ntok, d, dk = x.shape[0], wl.d, wl.dk
    g = torch.Generator().manual_seed(13)
    dqw, dqr, dvv = torch.randn(ntok, dk, generator=g), torch.randn(ntok, dk, generator=g), \
        torch.randn(ntok, d, generator=g)
    dx = torch.empty(ntok, d, device="cuda")
    dWqw = torch.empty(d, dk, device="cuda")
    dWqr = torch.empty_like(dWqw)
    dWv = torch.empty(d, d, device="cuda")
    ws = sdm.alloc_workspace(sdm.project_backward_workspace_bytes(cfg, ntok))
    sdm.sdm_project_backward(cfg, tl.to_dev(p), x.cuda(), dqw.cuda(), dqr.cuda(), dvv.cuda(), dx,
                             dWqw, dWqr, dWv, ws)
    torch.cuda.synchronize()
    ref = oracle.project_backward(x, p["W_qw"], p["W_qr"], p["W_v"], dqw.numpy(), dqr.numpy(),
                                  dvv.numpy())
    # fp32 layer: strict fp32 GEMMs. bf16 layer: TF32 tensor-core GEMMs, where x and the
    # weights are exact and each incoming gradient is rounded by at most u = 2^-11 of
    # itself, so an output's error is at most u * sum_k |a_k b_k|; with K <= 640 terms of
    # N(0,1)-like products that is u * 0.64 K against outputs of size ~4 sqrt(K) at the
    # largest, a relative 0.16 u sqrt(K) <= 2e-3 (the typical error is ~u / 4)
    tol = 1e-5 if wl.dtype == "f32" else 2e-3
    for got, want in zip((dx, dWqw, dWqr, dWv), ref):
        assert rel_err(got.cpu().numpy(), want) <= tol, name


def _offset_copy(t):
    """t's values in a buffer one element past a 16-byte boundary (a contiguous view)."""
    buf = torch.empty(t.numel() + 8, dtype=t.dtype, device="cuda")
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 16 != 0
    return v


@pytest.mark.parametrize("name", ["tiny-f32", "w64-small"])
def test_project_backward_unaligned_inputs_match_aligned(name):
    """The fp32 copies of x and the weights take their element-by-element path when a
    pointer is not 16-byte aligned; the gradients are the same bits either way (the copies
    are exact and the GEMMs read the same workspace)."""
    wl = SMALL[name]
    cfg = tl.cfg_of(wl)
    p = tl.to_dev(synth.make_params(wl))
    x = synth.make_tokens(wl)["x"].reshape(-1, wl.d).cuda()
    ntok, d, dk = x.shape[0], wl.d, wl.dk
    g = torch.Generator().manual_seed(17)
    dqw, dqr, dvv = (torch.randn(ntok, dk, generator=g).cuda(), torch.randn(ntok, dk, generator=g).cuda(),
                     torch.randn(ntok, d, generator=g).cuda())
    ws = sdm.alloc_workspace(sdm.project_backward_workspace_bytes(cfg, ntok))
    outs = []
    for shifted in (False, True):
        pp = dict(p)
        xx = x
        if shifted:
            for k in ("W_qw", "W_qr", "W_v"):
                pp[k] = _offset_copy(p[k])
            xx = _offset_copy(x)
        o = (torch.empty(ntok, d, device="cuda"), torch.empty(d, dk, device="cuda"),
             torch.empty(d, dk, device="cuda"), torch.empty(d, d, device="cuda"))
        sdm.sdm_project_backward(cfg, pp, xx, dqw, dqr, dvv, *o, ws)
        torch.cuda.synchronize()
        outs.append([t.cpu() for t in o])
    for a, b in zip(*outs):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("name,tol", [("tiny-f32", 1e-4), ("w64-small", 2e-2)])
def test_layer_backward_chain_matches_oracle(name, tol):
    """The whole layer's gradients: scan backward -> addressing backward -> projection
    backward on the GPU, against the same chain of oracle gradients (each oracle step
    fed the oracle's own upstream gradients)."""
    wl = SMALL[name]
    cfg = tl.cfg_of(wl)
    p = synth.make_params(wl)
    tok = synth.make_tokens(wl)
    out = tl.run_staged(wl, p, tok)
    B, T, d, N, W, dk, n = wl.B, wl.T, wl.d, wl.N, wl.W, wl.dk, wl.n
    ntok = B * T
    idx, wsel, v = out["idx"], out["wsel"], out["v"]
    al, be = out["alpha"].reshape(-1), out["beta"].reshape(-1)
    dt = wl.torch_dtype
    pd = tl.to_dev(p)
    banks = torch.empty(B, N, d, dtype=dt, device="cuda")
    sdm.sdm_init_bank(cfg, pd["M0"], banks)
    y = torch.empty(ntok, d, device="cuda")
    tape = torch.empty(ntok, W, d, dtype=dt, device="cuda")
    ws = sdm.alloc_workspace(sdm.scan_workspace_bytes(cfg, B, T))
    st = sdm.new_status()
    sdm.sdm_scan_prepare(cfg, idx, B, T, ws, st)
    sdm.sdm_scan_run_train(cfg, idx, wsel, v, al, be, banks, y, B, T, ws, tape, st)
    dy = torch.randn(ntok, d, generator=torch.Generator().manual_seed(17))
    dbank = torch.zeros(B, N, d, device="cuda")
    dv = torch.empty(ntok, d, device="cuda")
    dal = torch.empty(ntok, device="cuda")
    dbe = torch.empty(ntok, device="cuda")
    dws = torch.empty(ntok, 2, W, device="cuda")
    sdm.sdm_scan_backward(cfg, idx, wsel, v, al, be, tape, banks, dy.cuda(), dbank, dv, dal, dbe,
                          dws, B, T, sdm.alloc_workspace(sdm.scan_backward_workspace_bytes(cfg, B, T)))
    dq_w = torch.empty(ntok, dk, device="cuda")
    dq_r = torch.empty_like(dq_w)
    dK1 = torch.empty(n, dk // 2, device="cuda")
    dK2 = torch.empty_like(dK1)
    sdm.sdm_address_backward(cfg, pd["K1"], pd["K2"], out["q_w"], out["q_r"], idx, wsel, dws, dq_w,
                             dq_r, dK1, dK2,
                             sdm.alloc_workspace(sdm.address_backward_workspace_bytes(cfg, ntok)))
    dx = torch.empty(ntok, d, device="cuda")
    dW = [torch.empty(d, dk, device="cuda"), torch.empty(d, dk, device="cuda"),
          torch.empty(d, d, device="cuda")]
    x = tok["x"].reshape(ntok, d)
    sdm.sdm_project_backward(cfg, pd, x.cuda(), dq_w, dq_r, dv, dx, *dW,
                             sdm.alloc_workspace(sdm.project_backward_workspace_bytes(cfg, ntok)))
    torch.cuda.synchronize()
    assert sdm.read_status(st) == 0
    # the oracle chain
    idx_h, w_h = idx.cpu().numpy(), wsel.cpu().numpy().astype(np.float64)
    type_ = oracle.BF16 if wl.dtype == "bf16" else oracle.F32
    dvr = np.zeros((ntok, d))
    dwr = np.zeros((ntok, 2, W))
    for b in range(B):
        sl = slice(b * T, (b + 1) * T)
        ref = oracle.scan_backward(oracle.to_f64(p["M0"]), v[sl].cpu(), al[sl].cpu().numpy(),
                                   be[sl].cpu().numpy(), idx_h[sl, 0], w_h[sl, 0], idx_h[sl, 1],
                                   w_h[sl, 1], dy[sl].numpy(), None, type_=type_)
        dvr[sl], dwr[sl, 0], dwr[sl, 1] = ref["dv"], ref["dk"], ref["dr"]
    dqr_ = []
    dK1r = np.zeros((n, dk // 2))
    dK2r = np.zeros((n, dk // 2))
    for kind, q in ((0, out["q_w"]), (1, out["q_r"])):
        _, dq, k1, k2 = oracle.address_backward(q.cpu(), p["K1"], p["K2"], idx_h[:, kind],
                                                dwr[:, kind])
        dqr_.append(dq)
        dK1r += k1
        dK2r += k2
    dxr, *dWr = oracle.project_backward(x, p["W_qw"], p["W_qr"], p["W_v"], dqr_[0], dqr_[1], dvr)
    checks = [("dK1", dK1, dK1r), ("dK2", dK2, dK2r), ("dx", dx, dxr)] + \
        [("dW%d" % i, got, want) for i, (got, want) in enumerate(zip(dW, dWr))]
    for what, got, want in checks:
        e = rel_err(got.cpu().numpy(), want)
        assert e <= tol, (name, what, e)
