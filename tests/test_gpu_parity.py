"""GPU parity of the CUDA path (through the C-ABI) against the CPU oracle, element by
element, on seeded inputs small enough for the oracle to run in seconds but spanning
several blocks/machines and ragged tails. Full-size workloads: test_gpu_full.py."""
import numpy as np
import pytest
import torch

import oracle
import sparse_memory_linear_key_b300 as sdm
import synth
from tests import sdm_testlib as tl

pytestmark = pytest.mark.gpu

SMALL = {
    # the tiny fp32 workload itself (B1, T256, d64, n32, W8)
    "tiny-f32": synth.WORKLOADS["tiny-f32"],
    # ragged: T not a multiple of the token-parallel width or of the code block,
    # n not a power of two (padded sort), several machines per sequence
    "ragged-bf16": synth.Workload("ragged-bf16", B=3, T=333, d=96, n=40, dk=48, W=16,
                                  dtype="bf16", seed=77),
    "ragged-f32": synth.Workload("ragged-f32", B=2, T=201, d=48, n=24, dk=32, W=8,
                                 dtype="f32", seed=78),
    # W = n (the W = sqrt(N) edge), W = 32
    "w-eq-n": synth.Workload("w-eq-n", B=2, T=150, d=64, n=32, dk=64, W=32, dtype="bf16",
                             seed=79),
    # the pages' W = 64 with the real sub-key width, small bank
    "w64-small": synth.Workload("w64-small", B=2, T=300, d=128, n=96, dk=256, W=64,
                                dtype="bf16", seed=80),
    # the full 480 x 480 product-key grid and key width, small d
    "n480-small-d": synth.Workload("n480-small-d", B=1, T=257, d=32, n=480, dk=256, W=64,
                                   dtype="bf16", seed=81),
    # enough tokens for the scorer's tiles of 128 queries (fewer take replicated tiles
    # of 32), with a ragged last tile
    "n480-full-tiles": synth.Workload("n480-full-tiles", B=4, T=700, d=32, n=480, dk=256,
                                      W=64, dtype="bf16", seed=82),
    # slot vectors wider than one 1 KB row block of the scan, the last block partial:
    # bf16 d = 1280 is blocks of 512, 512 and 256 rows; fp32 d = 640 is 256, 256 and 128
    "multiblock-bf16": synth.Workload("multiblock-bf16", B=2, T=150, d=1280, n=24, dk=32,
                                      W=16, dtype="bf16", seed=83),
    "multiblock-f32": synth.Workload("multiblock-f32", B=2, T=130, d=640, n=16, dk=32, W=8,
                                     dtype="f32", seed=84),
}


def _inputs(wl):
    return synth.make_params(wl), synth.make_tokens(wl)


@pytest.fixture(scope="module", autouse=True)
def _build():
    from sparse_memory_linear_key_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_init_bank_bit_exact():
    for wl in (synth.WORKLOADS["tiny-f32"], SMALL["w64-small"]):
        p = synth.make_params(wl)
        cfg = tl.cfg_of(wl)
        banks = torch.empty(3, wl.N, wl.d, dtype=wl.torch_dtype, device="cuda")
        banks.fill_(7)
        sdm.sdm_init_bank(cfg, p["M0"].cuda(), banks)
        torch.cuda.synchronize()
        want = oracle.init_bank(p["M0"], 3)
        got, _ = oracle.storage(banks.cpu())
        assert np.array_equal(got, want)


@pytest.mark.parametrize("name", list(SMALL))
def test_projection_parity(name):
    wl = SMALL[name]
    p, tok = _inputs(wl)
    out = tl.run_staged(wl, p, tok)
    x = tok["x"].reshape(-1, wl.d)
    for key, w in (("q_w", "W_qw"), ("q_r", "W_qr"), ("v", "W_v")):
        ref = oracle.to_f64(oracle.project(x, p[w]))
        got = oracle.to_f64(out[key].cpu())
        if wl.dtype == "f32":
            np.testing.assert_allclose(got, ref, rtol=2e-5, atol=2e-5)
        else:
            assert tl.projection_ok(got, ref, oracle.to_f64(x), oracle.to_f64(p[w])), key


@pytest.mark.parametrize("name", list(SMALL))
def test_address_parity(name):
    """Slot sets exact (except near-ties) and weights within 1e-5, with the oracle
    scoring the CUDA path's own q bits."""
    wl = SMALL[name]
    p, tok = _inputs(wl)
    out = tl.run_staged(wl, p, tok)
    assert out["status"] == 0
    idx = out["idx"].cpu().numpy()
    wsel = out["wsel"].cpu().numpy()
    # ascending, distinct, in range
    assert np.all(np.diff(idx, axis=-1) > 0)
    assert idx.min() >= 0 and idx.max() < wl.N
    for kind, key in ((0, "q_w"), (1, "q_r")):
        S, k, _, gaps = oracle.address(out[key].cpu(), p["K1"], p["K2"], wl.W)
        n_bad, n_exc, unexc = tl.set_parity(idx[:, kind], S, gaps)
        tl.report_address(name, ("write", "read")[kind], wl.B * wl.T, len(unexc), n_exc)
        assert len(unexc) == 0, (name, kind, unexc[:5], n_bad, n_exc)
        err = tl.max_weight_err(idx[:, kind], wsel[:, kind], S, k, range(len(S)))
        assert err <= tl.WEIGHT_ATOL, (name, kind, err)
        np.testing.assert_allclose(wsel[:, kind].sum(-1), 1.0, atol=1e-5)


def test_address_tile_modes_agree():
    """The tensor-core scorer takes tiles of 128 queries for large batches and tiles of
    32 replicated queries for small ones. Each score is the same dot product either way
    and the selection is exact, so the addressing of a token must not depend on the
    batch it came in: bits of a 2,800-token call against calls on slices of it."""
    wl = SMALL["n480-full-tiles"]
    cfg = tl.cfg_of(wl)
    p = tl.to_dev(synth.make_params(wl, with_m0=False))
    g = torch.Generator().manual_seed(5)
    ntok = wl.B * wl.T
    q_w = torch.randn(ntok, wl.dk, generator=g).to(torch.bfloat16).cuda()
    q_r = torch.randn(ntok, wl.dk, generator=g).to(torch.bfloat16).cuda()
    st = sdm.new_status()

    def address(lo, hi):
        n = hi - lo
        idx = torch.empty(n, 2, wl.W, dtype=torch.int32, device="cuda")
        w = torch.empty(n, 2, wl.W, device="cuda")
        ws = sdm.alloc_workspace(sdm.address_workspace_bytes(cfg, n))
        sdm.sdm_address(cfg, p["K1"], p["K2"], q_w[lo:hi].contiguous(), q_r[lo:hi].contiguous(),
                        idx, w, ws, st)
        return idx.cpu(), w.cpu()

    idx_all, w_all = address(0, ntok)
    # 2800 tokens take tiles of 128 queries, 300 to 1000 tokens replicated tiles of 32
    for lo, hi in ((0, 300), (1000, 1557), (ntok - 999, ntok)):
        idx, w = address(lo, hi)
        assert torch.equal(idx, idx_all[lo:hi]), (lo, hi)
        assert torch.equal(w, w_all[lo:hi]), (lo, hi)
    assert sdm.read_status(st) == 0


@pytest.mark.parametrize("ntok", [200, 600, 2600])
def test_address_exact_ties(ntok):
    """Scores with exact ties everywhere: sub-keys and queries with entries in {-1, 0, 1},
    so every half score and every combined score is a small integer, the same in fp32 and
    fp64. The selection has no near-ties to excuse here, so the slot sets must equal the
    oracle's exactly: per half, equal scores go to the lower row, and among the combined
    scores, equal sums to the lower slot (the pages' top-k over the outer sum, read with
    that order). One query in eight is all zero (every score equal). 2,600 tokens take
    the tensor-core scorer's tiles of 128 queries, 600 tokens its replicated tiles of 32,
    200 tokens the few-token kernel."""
    n, dk, W = 480, 256, 64
    cfg = sdm.make_cfg(64, n, dk, W, "bf16")
    g = torch.Generator().manual_seed(17)

    def tern(*shape):
        return (torch.randint(0, 3, shape, generator=g) - 1).to(torch.bfloat16)

    K1, K2 = tern(n, dk // 2), tern(n, dk // 2)
    q_w, q_r = tern(ntok, dk), tern(ntok, dk)
    q_w[::8] = 0
    q_r[3::8] = 0
    idx = torch.empty(ntok, 2, W, dtype=torch.int32, device="cuda")
    w = torch.empty(ntok, 2, W, device="cuda")
    ws = sdm.alloc_workspace(sdm.address_workspace_bytes(cfg, ntok))
    st = sdm.new_status()
    sdm.sdm_address(cfg, K1.cuda(), K2.cuda(), q_w.cuda(), q_r.cuda(), idx, w, ws, st)
    torch.cuda.synchronize()
    assert sdm.read_status(st) == 0
    got = idx.cpu().numpy()
    for kind, q in ((0, q_w), (1, q_r)):
        S, _, _, _ = oracle.address(q, K1, K2, W)
        bad = np.nonzero(np.any(np.sort(got[:, kind], axis=1) != np.sort(S, axis=1), axis=1))[0]
        assert len(bad) == 0, (kind, bad[:5])


@pytest.mark.parametrize("ntok", [1, 7, 64, 256])
@pytest.mark.parametrize("shape", ["n480-w64", "w-eq-n", "ragged-f32-w8", "n96-w16"])
def test_address_few_tokens(ntok, shape):
    """Batches of at most 256 tokens (a decode step) take one block per query on the SIMT
    cores: slot sets exact against the oracle except counted near-ties, weights within
    1e-5, ascending and distinct."""
    d, n, dk, W, dt = {"n480-w64": (64, 480, 256, 64, "bf16"), "w-eq-n": (64, 32, 64, 32, "bf16"),
                       "ragged-f32-w8": (48, 24, 32, 8, "f32"),
                       "n96-w16": (64, 96, 128, 16, "bf16")}[shape]
    cfg = sdm.make_cfg(d, n, dk, W, dt)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    g = torch.Generator().manual_seed(ntok + n)
    K1 = (torch.randn(n, dk // 2, generator=g) / (dk // 2) ** 0.5).to(tdt)
    K2 = (torch.randn(n, dk // 2, generator=g) / (dk // 2) ** 0.5).to(tdt)
    q_w = torch.randn(ntok, dk, generator=g).to(tdt)
    q_r = torch.randn(ntok, dk, generator=g).to(tdt)
    if ntok >= 7:
        q_r[3] = q_w[3]                           # a read query equal to a write query
    idx = torch.empty(ntok, 2, W, dtype=torch.int32, device="cuda")
    w = torch.empty(ntok, 2, W, device="cuda")
    st = sdm.new_status()
    ws = sdm.alloc_workspace(sdm.address_workspace_bytes(cfg, ntok))
    sdm.sdm_address(cfg, K1.cuda(), K2.cuda(), q_w.cuda(), q_r.cuda(), idx, w, ws, st)
    torch.cuda.synchronize()
    assert sdm.read_status(st) == 0
    gi, gw = idx.cpu().numpy(), w.cpu().numpy()
    assert np.all(np.diff(gi, axis=-1) > 0) and gi.min() >= 0 and gi.max() < n * n
    for kind, q in ((0, q_w), (1, q_r)):
        S, k, _, gaps = oracle.address(q, K1, K2, W)
        n_bad, n_exc, unexc = tl.set_parity(gi[:, kind], S, gaps)
        tl.report_address("few-tokens %s x%d" % (shape, ntok), ("write", "read")[kind], ntok,
                          len(unexc), n_exc)
        assert len(unexc) == 0, (shape, ntok, kind, n_bad, n_exc)
        assert tl.max_weight_err(gi[:, kind], gw[:, kind], S, k, range(ntok)) <= tl.WEIGHT_ATOL
    if ntok >= 7:
        assert np.array_equal(gi[3, 0], gi[3, 1]) and np.array_equal(gw[3, 0], gw[3, 1])


@pytest.mark.parametrize("name", list(SMALL))
def test_scan_parity(name):
    """The recurrence on every row of every sequence, teacher-forced with the CUDA
    path's addressing, against the oracle: y and the final bank."""
    wl = SMALL[name]
    p, tok = _inputs(wl)
    out = tl.run_staged(wl, p, tok)
    assert out["status"] == 0
    rows = np.arange(wl.d)
    y = out["y"].cpu().numpy().reshape(wl.B, wl.T, wl.d)
    for b in range(wl.B):
        yr, M = tl.oracle_scan_rows(wl, p["M0"], out, b, rows)
        ok, m = tl.state_ok(wl.dtype, y[b], yr)
        assert ok, (name, b, "y", m)
        ok, m = tl.state_ok(wl.dtype, tl.bank_rows_cpu(out["banks"], b, rows), oracle.to_f64(M))
        assert ok, (name, b, "bank", m)


def test_prefill_entry_point_matches_staged():
    """sdm_prefill (one call) gives the same bits as the staged calls."""
    wl = SMALL["ragged-bf16"]
    p, tok = _inputs(wl)
    out = tl.run_staged(wl, p, tok)
    cfg = tl.cfg_of(wl)
    pd = tl.to_dev(p)
    banks = torch.empty(wl.B, wl.N, wl.d, dtype=wl.torch_dtype, device="cuda")
    sdm.sdm_init_bank(cfg, pd["M0"], banks)
    y = torch.empty(wl.B, wl.T, wl.d, device="cuda")
    idx = torch.empty(wl.B * wl.T, 2, wl.W, dtype=torch.int32, device="cuda")
    wsel = torch.empty(wl.B * wl.T, 2, wl.W, device="cuda")
    ws = sdm.alloc_workspace(sdm.workspace_bytes(cfg, wl.B, wl.T))
    st = sdm.new_status()
    sdm.sdm_prefill(cfg, pd, tok["x"].cuda(), tok["alpha"].cuda(), tok["beta"].cuda(), banks, y,
                    ws, st, idx_out=idx, w_out=wsel)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(idx, out["idx"]) and torch.equal(wsel, out["wsel"])
    assert torch.equal(y.reshape(-1, wl.d), out["y"])
    assert torch.equal(banks, out["banks"])


def test_tiny_f32_free_running():
    """The whole layer with the oracle's own projections and addressing (no teacher
    forcing) on the tiny fp32 workload."""
    wl = synth.WORKLOADS["tiny-f32"]
    p, tok = _inputs(wl)
    out = tl.run_staged(wl, p, tok)
    ref = oracle.prefill_sequence(tok["x"][0], p, tok["alpha"][0], tok["beta"][0], wl.W)
    idx = out["idx"].cpu().numpy()
    for kind, S, g in ((0, ref["S"], ref["gap_w"]), (1, ref["R"], ref["gap_r"])):
        n_bad, n_exc, unexc = tl.set_parity(idx[:, kind], S, g)
        tl.report_address(wl.name, ("write", "read")[kind], wl.B * wl.T, n_bad - n_exc, n_exc,
                          mode="free-running (oracle's own q)")
        assert n_bad == 0, (kind, n_bad, n_exc)
    y = out["y"].cpu().numpy()
    assert np.abs(y - ref["y"]).max() <= tl.F32_ATOL
    M = oracle.to_f64(out["banks"][0].cpu())
    assert np.abs(M - ref["M"]).max() <= tl.F32_ATOL


# ------------------------------------------------- the scan under heavy collisions

def _random_sets(rng, T, N, W):
    return np.stack([np.sort(rng.choice(N, W, replace=False)) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("B,T,N,W,d,dtype,seed", [
    (1, 500, 64, 8, 16, "bf16", 1),       # 8 of 64 slots per token: collisions at every dt
    (1, 700, 16, 8, 16, "f32", 2),        # half the bank written by every token
    (2, 300, 256, 64, 32, "bf16", 3),     # W = 64 of 256
    (1, 64, 64, 64, 16, "bf16", 4),       # every token writes and reads ALL slots
    (3, 97, 1024, 16, 48, "f32", 5),
])
def test_scan_collisions(B, T, N, W, d, dtype, seed):
    """Random ascending slot sets from a tiny bank (so consecutive tokens share many
    slots, and read sets hit the same token's write set): the collision forwarding
    of the token-parallel scan must reproduce the sequential oracle."""
    rng = np.random.default_rng(seed)
    n = int(round(N ** 0.5))
    cfg = sdm.make_cfg(d, n, 16, W, dtype)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    ntok = B * T
    idx = np.zeros((ntok, 2, W), dtype=np.int32)
    idx[:, 0] = _random_sets(rng, ntok, N, W)
    idx[:, 1] = _random_sets(rng, ntok, N, W)
    # some tokens read exactly what they write
    same = rng.random(ntok) < 0.2
    idx[same, 1] = idx[same, 0]
    wts = rng.random((ntok, 2, W)).astype(np.float32) + 0.05
    wts /= wts.sum(-1, keepdims=True)
    v = torch.randn(ntok, d, generator=torch.Generator().manual_seed(seed)).to(dt)
    M0 = (torch.randn(N, d, generator=torch.Generator().manual_seed(seed + 1)) * 0.1).to(dt)
    alpha = torch.from_numpy(rng.uniform(0.5, 1.0, ntok).astype(np.float32))
    beta = torch.from_numpy(rng.uniform(0.0, 1.0, ntok).astype(np.float32))
    banks, y, status = tl.run_scan_only(cfg, M0, torch.from_numpy(idx), torch.from_numpy(wts),
                                        v, alpha, beta, B, T)
    assert status == 0
    yg = y.cpu().numpy().reshape(B, T, d)
    for b in range(B):
        M = np.ascontiguousarray(oracle.storage(M0)[0].copy())
        sl = slice(b * T, (b + 1) * T)
        yr = oracle.scan(M, oracle.storage(v[sl])[0], alpha[sl].numpy().astype(np.float64),
                         beta[sl].numpy().astype(np.float64), idx[sl, 0],
                         wts[sl, 0].astype(np.float64), idx[sl, 1], wts[sl, 1].astype(np.float64))
        ok, m = tl.state_ok(dtype, yg[b], yr)
        assert ok, ("y", b, m)
        ok, m = tl.state_ok(dtype, oracle.to_f64(banks[b].cpu()), oracle.to_f64(M))
        assert ok, ("bank", b, m)


@pytest.mark.parametrize("B", [1, 200, 400, 800, 2000])
def test_scan_token_parallel_widths(B):
    """The launch picks 16, 8, 4, 2 or 1 tokens in flight per machine depending on
    how many machines there are; every width must agree with the oracle."""
    rng = np.random.default_rng(B)
    T, N, W, d = 40, 64, 8, 16
    cfg = sdm.make_cfg(d, 8, 16, W, "bf16")
    ntok = B * T
    idx = np.zeros((ntok, 2, W), dtype=np.int32)
    idx[:, 0] = _random_sets(rng, ntok, N, W)
    idx[:, 1] = _random_sets(rng, ntok, N, W)
    wts = (rng.random((ntok, 2, W)) + 0.05).astype(np.float32)
    wts /= wts.sum(-1, keepdims=True)
    v = torch.randn(ntok, d, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    M0 = (torch.randn(N, d, generator=torch.Generator().manual_seed(10)) * 0.1).to(torch.bfloat16)
    alpha = torch.from_numpy(rng.uniform(0.5, 1.0, ntok).astype(np.float32))
    beta = torch.from_numpy(rng.uniform(0.0, 1.0, ntok).astype(np.float32))
    banks, y, status = tl.run_scan_only(cfg, M0, torch.from_numpy(idx), torch.from_numpy(wts),
                                        v, alpha, beta, B, T)
    assert status == 0
    yg = y.cpu().numpy().reshape(B, T, d)
    bk = banks.cpu()
    for b in sorted(set([0, B // 2, B - 1])):
        M = np.ascontiguousarray(oracle.storage(M0)[0].copy())
        sl = slice(b * T, (b + 1) * T)
        yr = oracle.scan(M, oracle.storage(v[sl])[0], alpha[sl].numpy().astype(np.float64),
                         beta[sl].numpy().astype(np.float64), idx[sl, 0],
                         wts[sl, 0].astype(np.float64), idx[sl, 1], wts[sl, 1].astype(np.float64))
        assert tl.state_ok("bf16", yg[b], yr)[0]
        assert tl.state_ok("bf16", oracle.to_f64(bk[b]), oracle.to_f64(M))[0]


def test_single_token_and_single_sequence():
    """T = 1 (the decode shape) and B = 1 through sdm_decode_step and sdm_prefill."""
    wl = synth.Workload("t1", B=5, T=1, d=64, n=32, dk=64, W=16, dtype="bf16", seed=90)
    p, tok = _inputs(wl)
    out = tl.run_staged(wl, p, tok)
    cfg = tl.cfg_of(wl)
    pd = tl.to_dev(p)
    banks = torch.empty(wl.B, wl.N, wl.d, dtype=torch.bfloat16, device="cuda")
    sdm.sdm_init_bank(cfg, pd["M0"], banks)
    y = torch.empty(wl.B, wl.d, device="cuda")
    ws = sdm.alloc_workspace(sdm.workspace_bytes(cfg, wl.B, 1))
    st = sdm.new_status()
    sdm.sdm_decode_step(cfg, pd, tok["x"][:, 0].cuda().contiguous(),
                        tok["alpha"][:, 0].cuda().contiguous(),
                        tok["beta"][:, 0].cuda().contiguous(), banks, y, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(y, out["y"]) and torch.equal(banks, out["banks"])
    for b in range(wl.B):
        yr, M = tl.oracle_scan_rows(wl, p["M0"], out, b, np.arange(wl.d))
        assert tl.state_ok("bf16", y[b].cpu().numpy()[None], yr)[0]


@pytest.mark.parametrize("B,N,W,d,seed", [
    (64, 4096, 64, 2048, 11),     # the decode shape: 64 sequences x 4 row blocks
    (37, 1024, 64, 1280, 12),     # row blocks of 512, 512 and 256 rows; many own reads
    (9, 256, 32, 640, 13),
    (200, 64, 16, 96, 14),        # more items than two CTAs an SM hold at once
])
def test_one_token_kernel_matches_persistent_scan(B, N, W, d, seed):
    """With one token a sequence the scan runs every (sequence, row block) item in one wave
    (scan_step.cu) with the persistent kernel's arithmetic. Against the persistent kernel
    itself (the diagnostic entry point with an explicit wait bound takes it) on the same
    inputs: the same bits, y and banks; against the oracle: every row of the first and
    last sequences. A fifth of the tokens read exactly the slots they write, the others
    share some (the new values must reach the read)."""
    rng = np.random.default_rng(seed)
    n = int(round(N ** 0.5))
    cfg = sdm.make_cfg(d, n, 16, W, "bf16")
    idx = np.zeros((B, 2, W), dtype=np.int32)
    idx[:, 0] = _random_sets(rng, B, N, W)
    idx[:, 1] = _random_sets(rng, B, N, W)
    for b in range(B):
        if rng.random() < 0.2:
            idx[b, 1] = idx[b, 0]
        else:                                   # share about a quarter of the write set
            keep = rng.choice(W, W // 4, replace=False)
            rest = np.setdiff1d(np.arange(N), idx[b, 0])
            extra = rng.choice(rest, W - W // 4, replace=False)
            idx[b, 1] = np.sort(np.concatenate([idx[b, 0, keep], extra]))
    wts = (rng.random((B, 2, W)) + 0.05).astype(np.float32)
    wts /= wts.sum(-1, keepdims=True)
    v = torch.randn(B, d, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    M0 = (torch.randn(N, d, generator=torch.Generator().manual_seed(seed + 1)) * 0.1).to(torch.bfloat16)
    alpha = torch.from_numpy(rng.uniform(0.5, 1.0, B).astype(np.float32))
    beta = torch.from_numpy(rng.uniform(0.0, 1.0, B).astype(np.float32))
    dev = [t.cuda().contiguous() for t in (torch.from_numpy(idx), torch.from_numpy(wts), v, alpha, beta)]
    st = sdm.new_status()
    ws = sdm.alloc_workspace(sdm.scan_workspace_bytes(cfg, B, 1))
    outs = []
    for persistent in (False, True):
        banks = torch.empty((B,) + tuple(M0.shape), dtype=M0.dtype, device="cuda")
        sdm.sdm_init_bank(cfg, M0.cuda(), banks)
        y = torch.full((B, d), float("nan"), device="cuda")
        sdm.sdm_scan_prepare(cfg, dev[0], B, 1, ws, st)
        if persistent:
            sdm.sdm_scan_run_diag(cfg, *dev, banks, y, B, 1, ws, 2 * 10 ** 9, -1, st)
        else:
            sdm.sdm_scan_run(cfg, *dev, banks, y, B, 1, ws, st)
        torch.cuda.synchronize()
        assert sdm.read_status(st) == 0
        outs.append((y, banks))
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])
    y, banks = outs[0]
    for b in (0, B - 1):
        M = np.ascontiguousarray(oracle.storage(M0)[0].copy())
        yr = oracle.scan(M, oracle.storage(v[b:b + 1])[0], alpha[b:b + 1].numpy().astype(np.float64),
                         beta[b:b + 1].numpy().astype(np.float64), idx[b:b + 1, 0],
                         wts[b:b + 1, 0].astype(np.float64), idx[b:b + 1, 1],
                         wts[b:b + 1, 1].astype(np.float64))
        ok, m = tl.state_ok("bf16", y[b].cpu().numpy()[None], yr)
        assert ok, ("y", b, m)
        touched = np.union1d(idx[b, 0], idx[b, 1])
        ok, m = tl.state_ok("bf16", oracle.to_f64(banks[b].cpu())[touched], oracle.to_f64(M)[touched])
        assert ok, ("bank", b, m)


def test_zero_tokens_is_a_no_op():
    wl = SMALL["ragged-bf16"]
    cfg = tl.cfg_of(wl)
    banks = torch.zeros(1, wl.N, wl.d, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(1, wl.d, device="cuda")
    st = sdm.new_status()
    ws = sdm.alloc_workspace(256)
    idx = torch.zeros(1, 2, wl.W, dtype=torch.int32, device="cuda")
    sdm.sdm_scan(cfg, idx, torch.zeros(1, 2, wl.W, device="cuda"),
                 torch.zeros(1, wl.d, dtype=torch.bfloat16, device="cuda"),
                 torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda"), banks, y, 1, 0, ws,
                 st)
    torch.cuda.synchronize()
    assert st.item() == 0 and int(banks.abs().sum().item()) == 0


def test_out_of_range_slot_is_reported_not_faulted():
    """A slot id outside [0, N) reaching the scan is skipped and reported as
    SDM_ERANGE in the device status word."""
    B, T, N, W, d = 1, 10, 64, 8, 16
    cfg = sdm.make_cfg(d, 8, 16, W, "bf16")
    rng = np.random.default_rng(0)
    idx = np.zeros((T, 2, W), dtype=np.int32)
    idx[:, 0] = _random_sets(rng, T, N, W)
    idx[:, 1] = _random_sets(rng, T, N, W)
    idx[3, 1, -1] = N + 5          # ascending order kept: the last one is the largest
    wts = np.full((T, 2, W), 1.0 / W, dtype=np.float32)
    M0 = torch.zeros(N, d, dtype=torch.bfloat16)
    banks, y, status = tl.run_scan_only(cfg, M0, torch.from_numpy(idx), torch.from_numpy(wts),
                                        torch.ones(T, d, dtype=torch.bfloat16),
                                        torch.full((T,), 0.9), torch.full((T,), 0.5), B, T)
    assert status == sdm.SDM_ERANGE


def test_decode_steps_captured_in_a_graph_match_eager():
    """sdm_decode_step allocates nothing (all scratch is in the caller's workspace), so a
    sequence of decode steps can be captured in a CUDA graph after a first call; the
    replay gives the same bits as the eager calls."""
    wl = synth.Workload("g", B=8, T=6, d=64, n=32, dk=64, W=16, dtype="bf16", seed=77)
    p, tok = _inputs(wl)
    cfg = tl.cfg_of(wl)
    pd = tl.to_dev(p)
    x = tok["x"].cuda()
    al = tok["alpha"].cuda()
    be = tok["beta"].cuda()
    ws = sdm.alloc_workspace(sdm.workspace_bytes(cfg, wl.B, 1))
    st = sdm.new_status()

    def run(banks, y):
        for t in range(wl.T):
            sdm.sdm_decode_step(cfg, pd, x[:, t].contiguous(), al[:, t].contiguous(),
                                be[:, t].contiguous(), banks, y[t], ws, st)

    banks_e = torch.empty(wl.B, wl.N, wl.d, dtype=torch.bfloat16, device="cuda")
    sdm.sdm_init_bank(cfg, pd["M0"], banks_e)
    y_e = torch.empty(wl.T, wl.B, wl.d, device="cuda")
    run(banks_e, y_e)                       # eager (also the first call)
    banks_g = torch.empty_like(banks_e)
    sdm.sdm_init_bank(cfg, pd["M0"], banks_g)
    y_g = torch.zeros_like(y_e)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(banks_g, y_g)
    sdm.sdm_init_bank(cfg, pd["M0"], banks_g)   # capture did not run the work
    g.replay()
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(y_g, y_e) and torch.equal(banks_g, banks_e)


@pytest.mark.parametrize("B,T", [(3, 60), (2, 400)])
def test_prefill_m0_captured_in_a_graph_matches_eager(B, T):
    """sdm_prefill_m0 forks a side stream (the first-touch table and the fill beside the
    collision codes; for a few tokens also the v projection beside q) and joins it back,
    so a captured call becomes a graph with parallel branches. After a first call (which
    creates the side stream), the captured call replayed gives the eager call's bits.
    180 tokens take the few-token path, 800 the many-token one."""
    wl = synth.Workload("gp", B=B, T=T, d=128, n=40, dk=64, W=16, dtype="bf16", seed=93)
    p, tok = _inputs(wl)
    cfg = tl.cfg_of(wl)
    pd = tl.to_dev(p)
    x, al, be = tok["x"].cuda(), tok["alpha"].cuda(), tok["beta"].cuda()
    ws = sdm.alloc_workspace(sdm.prefill_m0_workspace_bytes(cfg, B, T))
    st = sdm.new_status()

    def run(banks, y):
        sdm.sdm_prefill_m0(cfg, pd, pd["M0"], x, al, be, banks, y, ws, st)

    banks_e = torch.empty(B, wl.N, wl.d, dtype=torch.bfloat16, device="cuda")
    y_e = torch.empty(B, T, wl.d, device="cuda")
    run(banks_e, y_e)
    torch.cuda.synchronize()
    banks_g = torch.zeros_like(banks_e)
    y_g = torch.zeros_like(y_e)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(banks_g, y_g)
    g.replay()
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(y_g, y_e) and torch.equal(banks_g, banks_e)
