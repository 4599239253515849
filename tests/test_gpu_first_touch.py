"""Bank initialisation fused into the recurrence (first touch): the banks start as M0
without a copy, the scan loads M0 for slots no earlier token of the sequence wrote, and
only never-written slots get M0's row afterwards. The arithmetic and the values it reads
are those of sdm_init_bank + the plain path, so every result must be bit-identical.
The first-touch table itself is integer work, checked exactly against its definition."""
import numpy as np
import pytest
import torch

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


def _garbage_like(t):
    g = torch.Generator(device="cuda").manual_seed(9)
    return torch.randn(t.shape, generator=g, device="cuda").to(t.dtype) * 1e3


# more sequences than a warp has lanes: the fill takes the first-writer table 32
# sequences at a time
MANY_SEQ = synth.Workload("many-seq", B=40, T=24, d=192, n=24, dk=32, W=8, dtype="bf16",
                          seed=85)


@pytest.mark.parametrize("name", ["tiny-f32", "ragged-bf16", "w64-small", "n480-full-tiles",
                                  "multiblock-bf16", "multiblock-f32", "many-seq"])
def test_prefill_m0_matches_init_then_prefill(name):
    wl = MANY_SEQ if name == "many-seq" else SMALL[name]
    cfg = tl.cfg_of(wl)
    p = tl.to_dev(synth.make_params(wl))
    tok = synth.make_tokens(wl)
    x, al, be = tok["x"].cuda(), tok["alpha"].cuda(), tok["beta"].cuda()
    st = sdm.new_status()
    B, T = wl.B, wl.T
    # reference: copy M0, then the plain one-call prefill
    banks_a = torch.empty(B, wl.N, wl.d, dtype=wl.torch_dtype, device="cuda")
    sdm.sdm_init_bank(cfg, p["M0"], banks_a)
    y_a = torch.empty(B, T, wl.d, device="cuda")
    idx_a = torch.empty(B * T, 2, wl.W, dtype=torch.int32, device="cuda")
    ws = sdm.alloc_workspace(sdm.workspace_bytes(cfg, B, T))
    sdm.sdm_prefill(cfg, p, x, al, be, banks_a, y_a, ws, st, idx_out=idx_a)
    # fused: banks full of garbage on entry
    banks_b = _garbage_like(banks_a)
    y_b = torch.empty_like(y_a)
    idx_b = torch.empty_like(idx_a)
    ws_m0 = sdm.alloc_workspace(sdm.prefill_m0_workspace_bytes(cfg, B, T))
    sdm.sdm_prefill_m0(cfg, p, p["M0"], x, al, be, banks_b, y_b, ws_m0, st, idx_out=idx_b)
    torch.cuda.synchronize()
    assert sdm.read_status(st) == 0
    assert torch.equal(idx_a, idx_b)
    assert torch.equal(y_a, y_b), name
    assert torch.equal(banks_a, banks_b), name


def test_first_touch_table_is_the_first_writer():
    wl = SMALL["ragged-bf16"]
    cfg = tl.cfg_of(wl)
    B, T, W, N = wl.B, wl.T, wl.W, wl.N
    g = np.random.default_rng(3)
    # slot sets drawn from a small range so that slots repeat often; some tokens repeat
    # their predecessor's set exactly
    idx = np.zeros((B * T, 2, W), np.int32)
    for i in range(B * T):
        if i % T and g.random() < 0.2:
            idx[i] = idx[i - 1]
        else:
            idx[i, 0] = np.sort(g.choice(N // 4, W, replace=False))
            idx[i, 1] = np.sort(g.choice(N // 4, W, replace=False))
    fw = torch.empty(B, N, dtype=torch.int32, device="cuda")
    assert sdm.first_touch_bytes(cfg, B) == B * N * 4
    sdm.sdm_first_touch(cfg, torch.from_numpy(idx).cuda(), B, T, fw)
    got = fw.cpu().numpy()
    want = np.full((B, N), np.iinfo(np.int32).max, np.int64)
    for b in range(B):
        for t in range(T - 1, -1, -1):
            want[b, idx[b * T + t, 0]] = t
    never = want == np.iinfo(np.int32).max
    assert np.array_equal(got[~never], want[~never])
    assert np.all(got[never] >= T)


@pytest.mark.parametrize("name", ["ragged-f32", "n480-small-d", "multiblock-bf16"])
def test_staged_first_touch_matches_copy(name):
    """first_touch + scan_run_m0 + fill_untouched against init_bank + scan_run, on the
    minimum workspace (no forwarding ring) and on the full one."""
    wl = SMALL[name]
    cfg = tl.cfg_of(wl)
    p, tok = tl.to_dev(synth.make_params(wl)), synth.make_tokens(wl)
    out = tl.run_staged(wl, synth.make_params(wl), tok)
    B, T = wl.B, wl.T
    idx, wsel, v = out["idx"], out["wsel"], out["v"]
    al, be = tok["alpha"].cuda(), tok["beta"].cuda()
    st = sdm.new_status()
    for ring in (True, False):
        nbytes = sdm.scan_workspace_bytes(cfg, B, T) if ring else sdm.scan_min_workspace_bytes(cfg, B, T)
        ws = sdm.alloc_workspace(nbytes)
        banks_a = torch.empty(B, wl.N, wl.d, dtype=wl.torch_dtype, device="cuda")
        sdm.sdm_init_bank(cfg, p["M0"], banks_a)
        y_a = torch.empty(B * T, wl.d, device="cuda")
        sdm.sdm_scan_prepare(cfg, idx, B, T, ws, st)
        sdm.sdm_scan_run(cfg, idx, wsel, v, al, be, banks_a, y_a, B, T, ws, st)
        banks_b = _garbage_like(banks_a)
        y_b = torch.empty_like(y_a)
        fw = torch.empty(B, wl.N, dtype=torch.int32, device="cuda")
        sdm.sdm_first_touch(cfg, idx, B, T, fw)
        sdm.sdm_scan_prepare(cfg, idx, B, T, ws, st)
        sdm.sdm_scan_run_m0(cfg, idx, wsel, v, al, be, p["M0"], fw, banks_b, y_b, B, T, ws, st)
        sdm.sdm_fill_untouched(cfg, p["M0"], fw, banks_b, B, T)
        torch.cuda.synchronize()
        assert sdm.read_status(st) == 0
        assert torch.equal(y_a, y_b), (name, ring)
        assert torch.equal(banks_a, banks_b), (name, ring)


def test_prefill_m0_with_no_tokens_is_the_copy():
    wl = SMALL["w64-small"]
    cfg = tl.cfg_of(wl)
    p = tl.to_dev(synth.make_params(wl))
    banks = torch.zeros(wl.B, wl.N, wl.d, dtype=wl.torch_dtype, device="cuda")
    x = torch.empty(wl.B, 0, wl.d, dtype=wl.torch_dtype, device="cuda")
    e = torch.empty(wl.B, 0, device="cuda")
    y = torch.empty(wl.B, 0, wl.d, device="cuda")
    ws = sdm.alloc_workspace(max(256, sdm.prefill_m0_workspace_bytes(cfg, wl.B, 0)))
    st = sdm.new_status()
    sdm.sdm_prefill_m0(cfg, p, p["M0"], x, e, e, banks, y, ws, st)
    torch.cuda.synchronize()
    for b in range(wl.B):
        assert torch.equal(banks[b], p["M0"])


@pytest.mark.parametrize("name", ["multiblock-bf16", "multiblock-f32", "w64-small"])
@pytest.mark.parametrize("staged", [False, True])
def test_first_touch_against_oracle(name, staged):
    """The fused path alone against the oracle, every row of every sequence: banks full
    of garbage on entry, the scan reading M0 for slots not yet written in the sequence
    (per row block: these workloads have two or three 1 KB blocks, the last partial),
    never-written slots filled from M0 afterwards. The oracle starts each sequence from
    M0 itself and is teacher-forced with the CUDA path's addressing and v bits."""
    import oracle
    wl = SMALL[name]
    cfg = tl.cfg_of(wl)
    p_cpu = synth.make_params(wl)
    p = tl.to_dev(p_cpu)
    tok = synth.make_tokens(wl)
    B, T, ntok = wl.B, wl.T, wl.B * wl.T
    x, al, be = tok["x"].cuda(), tok["alpha"].cuda(), tok["beta"].cuda()
    dt = wl.torch_dtype
    q_w = torch.empty(ntok, wl.dk, dtype=dt, device="cuda")
    q_r = torch.empty_like(q_w)
    v = torch.empty(ntok, wl.d, dtype=dt, device="cuda")
    sdm.sdm_project(cfg, p, x.reshape(ntok, wl.d), q_w, q_r, v)
    idx = torch.empty(ntok, 2, wl.W, dtype=torch.int32, device="cuda")
    wsel = torch.empty(ntok, 2, wl.W, device="cuda")
    st = sdm.new_status()
    banks = _garbage_like(torch.empty(B, wl.N, wl.d, dtype=dt, device="cuda"))
    y = torch.empty(ntok, wl.d, device="cuda")
    if staged:
        ws_a = sdm.alloc_workspace(sdm.address_workspace_bytes(cfg, ntok))
        sdm.sdm_address(cfg, p["K1"], p["K2"], q_w, q_r, idx, wsel, ws_a, st)
        fw = torch.empty(B, wl.N, dtype=torch.int32, device="cuda")
        ws = sdm.alloc_workspace(sdm.scan_workspace_bytes(cfg, B, T))
        sdm.sdm_first_touch(cfg, idx, B, T, fw)
        sdm.sdm_scan_prepare(cfg, idx, B, T, ws, st)
        sdm.sdm_scan_run_m0(cfg, idx, wsel, v, al, be, p["M0"], fw, banks, y, B, T, ws, st)
        sdm.sdm_fill_untouched(cfg, p["M0"], fw, banks, B, T)
    else:
        ws = sdm.alloc_workspace(sdm.prefill_m0_workspace_bytes(cfg, B, T))
        sdm.sdm_prefill_m0(cfg, p, p["M0"], x, al, be, banks, y.view(B, T, wl.d), ws, st,
                           idx_out=idx, w_out=wsel)
    torch.cuda.synchronize()
    assert sdm.read_status(st) == 0
    out = {"idx": idx, "wsel": wsel, "v": v, "alpha": al, "beta": be}
    rows = np.arange(wl.d)
    yg = y.cpu().numpy().reshape(B, T, wl.d)
    for b in range(B):
        yr, M = tl.oracle_scan_rows(wl, p_cpu["M0"], out, b, rows)
        ok, m = tl.state_ok(wl.dtype, yg[b], yr)
        assert ok, (name, staged, b, "y", m)
        ok, m = tl.state_ok(wl.dtype, tl.bank_rows_cpu(banks, b, rows), oracle.to_f64(M))
        assert ok, (name, staged, b, "bank", m)
