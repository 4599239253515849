#!/usr/bin/env python3
"""Benchmark of one Sparse Delta Memory (SDM) layer forward pass on B300.

Workload (N=1): prefill of 4 sequences x 4096 tokens, d = 2048, N = 480^2 slots,
W = 64, key width 256, bf16 banks (the 1.4B-scale layer of the pages). One step is
one pass of the whole hot path over that batch: the projections, product-key
addressing, the collision codes, and the recurrent scan with the bank initialisation
from M0 fused into it (first touch: the scan reads M0 for slots its sequence has not
written yet, and never-written slots get M0's row afterwards; bit-identical to a copy
of M0 into every bank first). Inputs are synthetic and seeded (synth/).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--no-decode]

Prints one JSON line (rank 0). `value` is tokens/s over the whole job with inputs
resident in HBM; `e2e` is the same metric through the public one-call API with the
inputs copied from pinned host memory and y copied back inside the timed region;
`roofline` is the scan kernel's algorithmic HBM bytes over its event-timed duration
against the measured copy bandwidth; `cpu_baseline` is the CPU oracle on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

WORKLOAD = "prefill-d2048-b4"
DECODE_WORKLOAD = "decode-d2048-b64"
METRIC = "SDM layer tokens/s (prefill, decode) on 1 B300; scan HBM GB/s vs 8 TB/s"
ORACLE_SAMPLE_TOKENS = 6144


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="sdm", choices=["sdm", "reference"])
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=None,
                    help="tokens per sequence instead of the workload's (for profiling a "
                         "small case of the same kernels)")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--only-decode", action="store_true",
                    help="run the decode arm alone (for profiling it)")
    ap.add_argument("--decode-steps", type=int, default=None,
                    help="decode steps instead of the workload's 512 (for profiling)")
    ap.add_argument("--batch", type=int, default=None,
                    help="sequences instead of the workload's (for profiling a small case)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the lines of the other prefill workloads (d = 3840 pool, 131k)")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, x: float) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# DRAM bytes (read + write) of one scan_kernel launch on this workload, from one ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum, 1 pass, full size). They hold
# for the kernel sources they were taken on; any change to those makes them stale.
SCAN_TRAFFIC = {"B": 4, "T": 4096, "bytes": 8439371776 + 4434630912,
                "sources_sha256": {"scan.cu": "12e47d24b7e3e77e", "sdm_common.cuh": "1f984e99590cd1ea",
                                   "scan_math.cuh": "d17a68a734fe9bd2"}}


def scan_traffic(B, T):
    import hashlib
    if (B, T) != (SCAN_TRAFFIC["B"], SCAN_TRAFFIC["T"]):
        return None
    csrc = os.path.join(ROOT, "sparse_memory_linear_key_b300", "csrc")
    for name, want in SCAN_TRAFFIC["sources_sha256"].items():
        with open(os.path.join(csrc, name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest()[:16] != want:
                return None
    return SCAN_TRAFFIC["bytes"]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6400.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- the GPU arm

# Events of one staged step: 0 start, 1 projected, 2 addressed, 3 codes done, 4 side
# stream joined, 5 scanned (caller's stream); 6 side start, 7 first touch done, 8 fill done
# (side stream). Stage -> (from, to).
STAGE_EVENTS = {"project": (0, 1), "address": (1, 2), "codes": (2, 3), "first_touch": (6, 7),
                "fill": (7, 8), "scan": (4, 5)}


def make_staged_step(sdm, cfg, p, x_proj, q_w, q_r, v_proj, alpha, beta, idx, wsel, v, banks, y,
                     B, T, ws_a, ws_s, first_write, st, stream, q_out=None):
    """One prefill step from M0 through the public staged calls, ordered as
    sdm_prefill_m0 orders them: projections, addressing, then the first-touch table and the
    fill of never-written slots on a side stream beside the collision codes, then the
    scan once both are done. q_out: where the projections go when the addressing reads
    other queries (workloads with injected queries), else q_w / q_r themselves."""
    side = torch.cuda.Stream()
    fork, join = torch.cuda.Event(), torch.cuda.Event()
    pw, pr = (q_out if q_out is not None else (q_w, q_r))

    def step(e=None):
        rec = (lambda j, s_: e[j].record(s_)) if e is not None else (lambda j, s_: None)
        rec(0, stream)
        sdm.sdm_project(cfg, p, x_proj, pw, pr, v_proj)
        rec(1, stream)
        sdm.sdm_address(cfg, p["K1"], p["K2"], q_w, q_r, idx, wsel, ws_a, st)
        rec(2, stream)
        fork.record(stream)
        side.wait_event(fork)
        rec(6, side)
        sdm.sdm_first_touch(cfg, idx, B, T, first_write, stream=side)
        rec(7, side)
        sdm.sdm_fill_untouched(cfg, p["M0"], first_write, banks, B, T, stream=side)
        rec(8, side)
        join.record(side)
        sdm.sdm_scan_prepare(cfg, idx, B, T, ws_s, st)
        rec(3, stream)
        stream.wait_event(join)
        rec(4, stream)
        sdm.sdm_scan_run_m0(cfg, idx, wsel, v, alpha, beta, p["M0"], first_write, banks, y, B, T,
                            ws_s, st)
        rec(5, stream)

    return step


def stage_times(ev):
    ms = {n: statistics.mean(e[a].elapsed_time(e[b]) for e in ev)
          for n, (a, b) in STAGE_EVENTS.items()}
    # how long the scan waited for the side stream after the codes were done
    ms["join_wait"] = statistics.mean(e[3].elapsed_time(e[4]) for e in ev)
    return ms


def gpu_arm(args, world, rank):
    import sparse_memory_linear_key_b300 as sdm
    from sparse_memory_linear_key_b300 import build
    build.build()
    sdm.lib()

    wl = synth.WORKLOADS[WORKLOAD]
    if args.tokens:
        wl = wl.with_(T=args.tokens)
    if args.batch:
        wl = wl.with_(B=args.batch)
    dev = "cuda"
    cfg = sdm.make_cfg(wl.d, wl.n, wl.dk, wl.W, wl.dtype)
    p_cpu = synth.make_params(wl)
    tok_cpu = synth.make_tokens(wl)
    p = {k: v.to(dev) for k, v in p_cpu.items()}
    x = tok_cpu["x"].to(dev)
    alpha = tok_cpu["alpha"].to(dev)
    beta = tok_cpu["beta"].to(dev)
    B, T, d = wl.B, wl.T, wl.d
    ntok = B * T
    banks = torch.empty(B, wl.N, d, dtype=torch.bfloat16, device=dev)
    q_w = torch.empty(ntok, wl.dk, dtype=torch.bfloat16, device=dev)
    q_r = torch.empty_like(q_w)
    v = torch.empty(ntok, d, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(ntok, 2, wl.W, dtype=torch.int32, device=dev)
    wsel = torch.empty(ntok, 2, wl.W, dtype=torch.float32, device=dev)
    y = torch.empty(ntok, d, dtype=torch.float32, device=dev)
    ws_a = sdm.alloc_workspace(sdm.address_workspace_bytes(cfg, ntok))
    ws_s = sdm.alloc_workspace(sdm.scan_workspace_bytes(cfg, B, T))
    first_write = torch.empty(B, wl.N, dtype=torch.int32, device=dev)
    st = sdm.new_status()
    stream = torch.cuda.current_stream()

    # Bank initialisation is fused: the scan reads M0 for slots not yet written in the
    # sequence (first-touch table), and the slots a sequence never writes get M0's row
    # -- bit-identical to copying M0 into every bank first. The table and the fill run on
    # a side stream beside the collision codes (as sdm_prefill_m0 runs them).
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(9)] for _ in range(args.steps)]
    step = make_staged_step(sdm, cfg, p, x, q_w, q_r, v, alpha, beta, idx, wsel, v, banks, y, B, T,
                            ws_a, ws_s, first_write, st, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if sdm.read_status(st) != 0:
        raise RuntimeError("device status %d" % sdm.read_status(st))

    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        t0.record(stream)
        for i in range(args.steps):
            step(ev[i])
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    status = sdm.read_status(st)
    if status != 0:
        raise RuntimeError("device status %d during the timed steps" % status)
    # for the slot-set check of the CPU-baseline leg: 128 sampled tokens' q bits and sets
    import numpy as np
    toks = np.sort(np.random.default_rng(7).choice(ntok, 128, replace=False))
    samples = [(WORKLOAD, address_sample(q_w, q_r, idx, toks, x=x.reshape(ntok, d)))]
    elapsed_ms = t0.elapsed_time(t1)
    elapsed_ms = max_over_ranks(world, elapsed_ms)
    stage_ms = stage_times(ev)
    ms_per_step = elapsed_ms / args.steps
    # the codes alone (outside the timed region): in the step they share the GPU with the
    # fill, whose HBM traffic stretches them, but the scan waits for the fill anyway.
    # Five calls captured in a CUDA graph, so that no host launch gap is timed.
    gc = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gc):
        for _ in range(5):
            sdm.sdm_scan_prepare(cfg, idx, B, T, ws_s, st)
    gc.replay()
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    gc.replay()
    c1.record(stream)
    torch.cuda.synchronize()
    stage_ms["codes_alone"] = c0.elapsed_time(c1) / 5
    del gc
    value = ntok * world * args.steps / (elapsed_ms / 1e3)

    # roofline of the scan kernel: algorithmic bytes per launch / launch duration
    s_bytes = 2
    per_tok = (3 * wl.W * d * s_bytes          # write-set read + write, read-set read
               + d * s_bytes + d * 4            # v in, y out
               + 2 * wl.W * (4 + 4 + 2) + 8)    # slot ids, weights, codes, alpha, beta
    scan_bytes = per_tok * ntok
    scan_s = stage_ms["scan"] / 1e3
    peak, peak_kind = measured_peaks()
    achieved = scan_bytes / scan_s / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": scan_traffic(B, T),
                "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.4 TB/s",
                "kernel": "scan_kernel<bf16,64>", "bytes_per_token": per_tok,
                "vs_8tbs": round(achieved / 8000.0, 4),
                "literal_2Wd_count_frac_8tbs": round(
                    (2 * wl.W * d * s_bytes + 2 * wl.W * 8) * ntok / scan_s / 1e9 / 8000.0, 4)}

    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; x~N(0,1), weights N(0,1/sqrt(fan_in)), M0~N(0,0.02))",
        "config": {"workload": WORKLOAD, "B": B, "T": T, "d": d, "N": wl.N, "W": wl.W,
                   "dk": wl.dk, "state": "bf16", "parallelism": "replicas" if world > 1 else "1gpu",
                   "l2": "inputs larger than L2: each step moves > 15 GB of bank and M0 rows",
                   "step": "projections + addressing + codes + bank init fused as first touch "
                           "(M0 read by the scan for slots not yet written, never-written slots "
                           "filled from M0; the first-touch table and the fill on a side stream "
                           "beside the codes) + scan"},
        "stages_ms": {k: round(v_, 4) for k, v_ in stage_ms.items()},
        "scan_tokens_per_s": round(ntok / scan_s, 1),
        # the same step without bank initialisation (as on banks already holding a
        # state): the step less the time the scan waited for the side stream (first-touch
        # table and fill) after the codes, from the event times; the scan reads the same
        # bytes from M0 as from a copied bank
        "prefill_without_bank_init": {
            "value": round(ntok * world / ((ms_per_step - stage_ms["join_wait"]) / 1e3), 1),
            "unit": "tokens/s",
            "ms_per_step": round(ms_per_step - stage_ms["join_wait"], 4)},
        "roofline": roofline,
        "clocks": clocks.summary(),
        # the library's own kernels in the timed region: projections, scorer, candidate
        # selection, codes, first touch, scan, fill (plus three cudaMemsetAsync a step)
        "gpu_launches": 7 * args.steps,
        "library_launches": {},
    }

    # ---- the dense-state comparator on the same tokens: the gated delta rule on a
    # dense [d, 64] state per sequence, with this step's write / read weights, v and gates
    y_g = torch.empty(ntok, d, dtype=torch.float32, device=dev)

    def gdn():
        sdm.sdm_gdn_dense_scan(cfg, wsel, wsel[:, 1], 2 * wl.W, v, alpha, beta, y_g, B, T)

    for _ in range(3):
        gdn()
    torch.cuda.synchronize()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    n_g = max(3, args.steps // 5)
    g0.record(stream)
    for _ in range(n_g):
        gdn()
    g1.record(stream)
    torch.cuda.synchronize()
    g_ms = g0.elapsed_time(g1) / n_g
    res["dense_comparator"] = {
        "what": "gated delta rule on a dense [d, 64] fp32 state per sequence (the state size "
                "of SDM's 64 active slots), same tokens, weights, v and gates, iso-FLOP",
        "ms": round(g_ms, 4), "tokens_per_s": round(ntok / (g_ms / 1e3), 1),
        "vs_sdm_scan": round(g_ms / stage_ms["scan"], 4),
        "state_bytes_per_sequence": d * 64 * 4,
        "sdm_state_bytes_per_sequence": wl.N * d * 2,
        # HBM bytes a token moves: v in, y out, both weight vectors, gates (the state
        # stays on chip) against the SDM scan's 800,008
        "hbm_bytes_per_token": d * 2 + d * 4 + 2 * 64 * 4 + 8,
        "kernel": "gdn_dense_kernel: sequential in t per row, state in registers",
        "gpu_launches_per_call": 1}
    del y_g

    # ---- training: the forward that records the tape, and the backward of the
    # recurrence (dv, dalpha, dbeta, weight gradients, initial-bank gradient) on the same
    # tokens. Timed once each after a warm-up pair; the banks walk back to M0 and are
    # re-filled from M0 by the next forward.
    if not args.no_backward:
        tape = torch.empty(ntok, wl.W, d, dtype=torch.bfloat16, device=dev)
        dy = torch.randn(ntok, d, device=dev)
        dbank = torch.zeros(B, wl.N, d, device=dev)
        dv = torch.empty(ntok, d, device=dev)
        dal = torch.empty(ntok, device=dev)
        dbe = torch.empty(ntok, device=dev)
        dws = torch.empty(ntok, 2, wl.W, device=dev)
        wsb = sdm.alloc_workspace(sdm.scan_backward_workspace_bytes(cfg, B, T))

        def train_pair(e=None):
            sdm.sdm_first_touch(cfg, idx, B, T, first_write)
            sdm.sdm_scan_prepare(cfg, idx, B, T, ws_s, st)
            if e is not None:
                e[0].record(stream)
            sdm.sdm_scan_run_train(cfg, idx, wsel, v, alpha, beta, banks, y, B, T, ws_s, tape, st,
                                   M0=p["M0"], first_write=first_write)
            if e is not None:
                e[1].record(stream)
            sdm.sdm_fill_untouched(cfg, p["M0"], first_write, banks, B, T)
            dbank.zero_()
            if e is not None:
                e[2].record(stream)
            sdm.sdm_scan_backward(cfg, idx, wsel, v, alpha, beta, tape, banks, dy, dbank, dv, dal,
                                  dbe, dws, B, T, wsb)
            if e is not None:
                e[3].record(stream)

        train_pair()
        torch.cuda.synchronize()
        te = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        train_pair(te)
        torch.cuda.synchronize()
        if sdm.read_status(st) != 0:
            raise RuntimeError("device status during the training pair")
        fwd_ms, bwd_ms = te[0].elapsed_time(te[1]), te[2].elapsed_time(te[3])
        # the rest of the layer's gradients: addressing (dq, dK) and projections (dx, dW)
        dq_w = torch.empty(ntok, wl.dk, device=dev)
        dq_r = torch.empty_like(dq_w)
        dK1 = torch.empty(wl.n, wl.dk // 2, device=dev)
        dK2 = torch.empty_like(dK1)
        dx = torch.empty(ntok, d, device=dev)
        dW = [torch.empty(d, wl.dk, device=dev), torch.empty(d, wl.dk, device=dev),
              torch.empty(d, d, device=dev)]
        wsa_b = sdm.alloc_workspace(sdm.address_backward_workspace_bytes(cfg, ntok))
        wsp_b = sdm.alloc_workspace(sdm.project_backward_workspace_bytes(cfg, ntok))
        xb = x.reshape(ntok, d)

        def front_bwd(e=None):
            if e is not None:
                e[0].record(stream)
            sdm.sdm_address_backward(cfg, p["K1"], p["K2"], q_w, q_r, idx, wsel, dws, dq_w, dq_r,
                                     dK1, dK2, wsa_b)
            if e is not None:
                e[1].record(stream)
            sdm.sdm_project_backward(cfg, p, xb, dq_w, dq_r, dv, dx, *dW, wsp_b)
            if e is not None:
                e[2].record(stream)

        front_bwd()
        fe = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        front_bwd(fe)
        torch.cuda.synchronize()
        addr_bwd_ms, proj_bwd_ms = fe[0].elapsed_time(fe[1]), fe[1].elapsed_time(fe[2])
        del dq_w, dq_r, dK1, dK2, dx, dW, wsa_b, wsp_b
        # the backward walk's algorithmic bytes per token: at each read slot the bank row
        # (bf16) and the gradient row read and written (fp32); at each write slot the
        # gradient row read and written, the tape row read and the bank row restored;
        # dy and dv (fp32) and v (bf16)
        bwd_tok = wl.W * d * (2 + 4 + 4) + wl.W * d * (4 + 4 + 2 + 2) + d * (4 + 4 + 2)
        peak_b, _ = measured_peaks()
        bwd_gbs = bwd_tok * ntok / (bwd_ms / 1e3) / 1e9
        res["training"] = {
            "what": "scan forward recording the tape (pre-write slot values), then the backward "
                    "of the recurrence, the addressing and the projections; bf16 tape and banks, "
                    "fp32 gradients",
            "forward_with_tape_ms": round(fwd_ms, 3), "backward_ms": round(bwd_ms, 3),
            "backward_tokens_per_s": round(ntok / (bwd_ms / 1e3), 1),
            "address_backward_ms": round(addr_bwd_ms, 3),
            "project_backward_ms": round(proj_bwd_ms, 3),
            "layer_backward_tokens_per_s": round(
                ntok / ((bwd_ms + addr_bwd_ms + proj_bwd_ms) / 1e3), 1),
            "tape_bytes": tape.numel() * 2,
            "backward_roofline": {"bound": "hbm", "bytes_per_token": bwd_tok,
                                  "achieved": round(bwd_gbs, 1), "peak": peak_b, "unit": "GB/s",
                                  "frac": round(bwd_gbs / peak_b, 4),
                                  "timed": "the whole sdm_scan_backward call (descriptor pre-pass, "
                                           "walk, partial-sum reduction)"},
            "kernel": "scan_bwd_kernel: one block per (sequence, 64 rows), reverse token order, "
                      "each token's gathers issued one token ahead"}
        del tape, dy, dbank, dv, dal, dbe, dws, wsb
        torch.cuda.empty_cache()

    # ---- e2e: the one-call public API with host buffers. Every step copies its inputs
    # in from pinned host memory, runs sdm_prefill_m0 and copies y back out; the copies
    # run on their own streams (the copy engines), double-buffered, so that step i+1's
    # inputs come in and step i-1's y goes out while step i computes.
    x_h = tok_cpu["x"].pin_memory()
    a_h = tok_cpu["alpha"].pin_memory()
    b_h = tok_cpu["beta"].pin_memory()
    y_h = torch.empty(B, T, d, dtype=torch.float32).pin_memory()
    ws_p = sdm.alloc_workspace(sdm.prefill_m0_workspace_bytes(cfg, B, T))
    x_d = [torch.empty_like(x) for _ in range(2)]
    a_d = [torch.empty_like(alpha) for _ in range(2)]
    b_d = [torch.empty_like(beta) for _ in range(2)]
    y_d = [torch.empty(B, T, d, dtype=torch.float32, device=dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]      # step's inputs on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]    # step computed (inputs free, y ready)
    ev_out = [torch.cuda.Event() for _ in range(2)]     # step's y copied out (y buffer free)
    used = [False, False]

    def e2e_step(i):
        j = i & 1
        with torch.cuda.stream(s_in):
            if used[j]:
                s_in.wait_event(ev_done[j])                  # step i-2 has read these inputs
            x_d[j].copy_(x_h, non_blocking=True)
            a_d[j].copy_(a_h, non_blocking=True)
            b_d[j].copy_(b_h, non_blocking=True)
            ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        if used[j]:
            stream.wait_event(ev_out[j])                     # step i-2's y has been copied out
        sdm.sdm_prefill_m0(cfg, p, p["M0"], x_d[j], a_d[j], b_d[j], banks, y_d[j], ws_p, st)
        ev_done[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[j])
            y_h.copy_(y_d[j], non_blocking=True)
            ev_out[j].record(s_out)
        used[j] = True

    for i in range(max(2, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    # the pipeline's fill (first copy in) and drain (last copy out) are timed too
    # (a serving loop's steady state: the one-off first copy in and last copy out are
    # spread over twice the timed steps)
    n_e2e = max(20, 2 * args.steps)
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(n_e2e):
        e2e_step(i)
    stream.wait_stream(s_out)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1))
    if sdm.read_status(st) != 0:
        raise RuntimeError("device status during e2e")
    h2d = x_h.numel() * x_h.element_size() + a_h.numel() * 4 + b_h.numel() * 4
    d2h = y_h.numel() * 4
    res["e2e"] = {"value": round(ntok * world * n_e2e / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
                  "ms_per_step": round(e2e_ms / n_e2e, 4),
                  "api": "sdm_prefill_m0 per step; copies on two side streams, double-buffered, "
                         "overlapping the neighbouring steps' compute"}
    del ws_p, x_d, y_d

    if not args.no_decode:
        res["decode"] = decode_arm(sdm, args, world)
        samples.append(res["decode"].pop("_sample"))

    del banks, q_w, q_r, v, idx, wsel, y, ws_a, ws_s
    torch.cuda.empty_cache()
    # the pages' other prefill shapes: the 8B-width layer with repeated pool queries, and
    # one 131,072-token sequence with the inserted key/value pattern
    if not args.no_workloads and args.tokens is None and args.batch is None:
        res["workloads"] = {}
        for name in ("prefill-d3840-pool", "long-131k"):
            line = prefill_line(sdm, name, steps=max(3, min(10, args.steps // 5)), warmup=2)
            samples.append(line.pop("_sample"))
            res["workloads"][name] = line
            res["gpu_launches"] += line["gpu_launches_per_step"] * line["steps"]
    return res, p_cpu, tok_cpu, samples


def decode_arm(sdm, args, world):
    """64 sequences, 1024 prior writes by a prefill, then `decode_steps` timed
    sdm_decode_step calls (one token per sequence per call)."""
    wl = synth.WORKLOADS[DECODE_WORKLOAD]
    dev = "cuda"
    cfg = sdm.make_cfg(wl.d, wl.n, wl.dk, wl.W, wl.dtype)
    p = {k: v.to(dev) for k, v in synth.make_params(wl).items()}
    tok = synth.make_tokens(wl)
    dec = synth.make_decode_tokens(wl)
    B = wl.B
    banks = torch.empty(B, wl.N, wl.d, dtype=torch.bfloat16, device=dev)
    sdm.sdm_init_bank(cfg, p["M0"], banks)
    st = sdm.new_status()
    ws = sdm.alloc_workspace(sdm.workspace_bytes(cfg, B, wl.T))
    y0 = torch.empty(B, wl.T, wl.d, device=dev)
    sdm.sdm_prefill(cfg, p, tok["x"].to(dev), tok["alpha"].to(dev), tok["beta"].to(dev), banks,
                    y0, ws, st)
    del ws, y0
    wsd = sdm.alloc_workspace(sdm.workspace_bytes(cfg, B, 1))
    xd = dec["x"].to(dev)
    ad = dec["alpha"].to(dev)
    bd = dec["beta"].to(dev)
    S = args.decode_steps if args.decode_steps else wl.decode_steps
    y = torch.empty(S, B, wl.d, device=dev)

    def steps():
        for s_ in range(S):
            sdm.sdm_decode_step(cfg, p, xd[s_], ad[s_], bd[s_], banks, y[s_], wsd, st)

    # eager: one host call per step
    stream = torch.cuda.current_stream()
    steps()
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    steps()
    e1.record(stream)
    torch.cuda.synchronize()
    eager_ms = max_over_ranks(world, e0.elapsed_time(e1))
    # the same S calls captured once in a CUDA graph and replayed
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        steps()
    g.replay()
    torch.cuda.synchronize()
    barrier(world)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    g.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(world, g0.elapsed_time(g1))
    if sdm.read_status(st) != 0:
        raise RuntimeError("device status during decode")
    per_step_bytes = 3 * wl.W * wl.d * 2 * B
    out = {"workload": DECODE_WORKLOAD, "value": round(B * S * world / (ms / 1e3), 1),
           "unit": "tokens/s", "steps": S, "us_per_step": round(ms * 1e3 / S, 2),
           "state_hbm_gbs": round(per_step_bytes * S / (ms / 1e3) / 1e9, 1),
           "eager_us_per_step": round(eager_ms * 1e3 / S, 2),
           "note": "%d sdm_decode_step calls (projections, addressing, scan) "
                   "captured in one CUDA graph; eager = one host call per step" % S}
    peak, _ = measured_peaks()
    out["state_roofline_frac"] = round(out["state_hbm_gbs"] / peak, 4)
    # one more step, after the timed ones, returning the slot sets it used; the same
    # projection kernel on the same x gives the q bits it scored (slot-set check)
    idx1 = torch.empty(B, 2, wl.W, dtype=torch.int32, device=dev)
    y1 = torch.empty(B, wl.d, device=dev)
    sdm.sdm_decode_step(cfg, p, xd[0], ad[0], bd[0], banks, y1, wsd, st, idx_out=idx1)
    qw1 = torch.empty(B, wl.dk, dtype=torch.bfloat16, device=dev)
    qr1 = torch.empty_like(qw1)
    sdm.sdm_project(cfg, p, xd[0], qw1, qr1, torch.empty(B, wl.d, dtype=torch.bfloat16, device=dev))
    torch.cuda.synchronize()
    out["_sample"] = (DECODE_WORKLOAD, address_sample(qw1, qr1, idx1, list(range(B))))
    del g
    del banks, p, xd, y
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------- the other prefill workloads

def scan_bytes_per_token(wl):
    """Algorithmic HBM bytes of the scan per token: the write set read and written, the
    read set read (disjoint sets on random inputs), v in, y out (fp32), slot ids, weights
    and collision codes of both sets, the two gates."""
    s = wl.elem_bytes
    return (3 * wl.W * wl.d * s + wl.d * s + wl.d * 4 + 2 * wl.W * (4 + 4 + 2) + 8)


def address_sample(q_w, q_r, idx, toks, x=None):
    """What the slot-set check needs of the GPU side, on sampled tokens, copied to the
    host after the timed region: the q bits the addressing scored, the slot sets it
    chose and (optionally) the tokens' x."""
    tt = torch.as_tensor(toks, device=idx.device)
    return {"q_w": q_w[tt].cpu(), "q_r": q_r[tt].cpu(), "idx": idx[tt].cpu().numpy(),
            "x": None if x is None else x[tt].cpu()}


def address_check(wl, p_cpu, smp):
    """Slot sets of the sampled tokens against the oracle scoring the same q bits (the
    CPU-baseline leg; nothing here is timed): mismatches a near-tie does not excuse, and
    mismatches excused because the oracle's gap between the W-th and (W+1)-th combined
    score is below 1e-5. With the tokens' x, also the oracle's own projections and
    addressing (free-running: a one-ulp bf16 difference in q can flip a boundary slot)."""
    import numpy as np
    import oracle
    gi = smp["idx"]
    free_x = smp["x"]
    out = {"sampled_tokens": int(gi.shape[0])}
    for kind, q in ((0, smp["q_w"]), (1, smp["q_r"])):
        S, _, _, gaps = oracle.address(q, p_cpu["K1"], p_cpu["K2"], wl.W)
        bad = np.any(np.sort(gi[:, kind], -1) != np.sort(S, -1), axis=1)
        tie = bad & (gaps < 1e-5)
        key = ("write", "read")[kind]
        out[key] = {"unexcused_mismatches": int((bad & ~tie).sum()),
                    "near_tie_mismatches": int(tie.sum())}
        if free_x is not None:
            wm = p_cpu["W_qw" if kind == 0 else "W_qr"]
            S2, _, _, g2 = oracle.address(oracle.project(free_x, wm), p_cpu["K1"], p_cpu["K2"],
                                          wl.W)
            bad2 = np.any(np.sort(gi[:, kind], -1) != np.sort(S2, -1), axis=1)
            out[key]["free_running_mismatches"] = int(bad2.sum())
            out[key]["free_running_near_ties"] = int((bad2 & (g2 < 1e-5)).sum())
    return out


def prefill_line(sdm, name, steps, warmup):
    """One of the pages' other prefill shapes, timed like the main step: projections,
    addressing, codes, first-touch table, the scan from M0 and the fill. The workload's
    query substitution (a pool of repeated queries, or the inserted key/value pattern) is
    a property of its inputs: it is applied once to projected queries before the timed
    steps, and each step's addressing and scan take those; each step's projection still
    runs in full (into buffers of its own)."""
    import numpy as np
    wl = synth.WORKLOADS[name]
    dev = "cuda"
    cfg = sdm.make_cfg(wl.d, wl.n, wl.dk, wl.W, wl.dtype)
    p_cpu = synth.make_params(wl)
    tok = synth.make_tokens(wl)
    p = {k: v_.to(dev) for k, v_ in p_cpu.items()}
    B, T, d = wl.B, wl.T, wl.d
    ntok = B * T
    x = tok["x"].to(dev)
    alpha = tok["alpha"].to(dev)
    beta = tok["beta"].to(dev)
    q_w = torch.empty(ntok, wl.dk, dtype=torch.bfloat16, device=dev)
    q_r = torch.empty_like(q_w)
    v = torch.empty(ntok, d, dtype=torch.bfloat16, device=dev)
    sdm.sdm_project(cfg, p, x, q_w, q_r, v)
    pool, pattern = synth.make_pool(wl), synth.make_pattern(wl)
    synth.inject_queries(wl, q_w.view(B, T, -1), q_r.view(B, T, -1), v.view(B, T, -1),
                         pool=pool, pattern=pattern)
    qs_w, qs_r, vs = torch.empty_like(q_w), torch.empty_like(q_r), torch.empty_like(v)
    banks = torch.empty(B, wl.N, d, dtype=torch.bfloat16, device=dev)
    idx = torch.empty(ntok, 2, wl.W, dtype=torch.int32, device=dev)
    wsel = torch.empty(ntok, 2, wl.W, dtype=torch.float32, device=dev)
    y = torch.empty(ntok, d, dtype=torch.float32, device=dev)
    ws_a = sdm.alloc_workspace(sdm.address_workspace_bytes(cfg, ntok))
    ws_s = sdm.alloc_workspace(sdm.scan_workspace_bytes(cfg, B, T))
    first_write = torch.empty(B, wl.N, dtype=torch.int32, device=dev)
    st = sdm.new_status()
    stream = torch.cuda.current_stream()
    # the projections are timed into scratch (qs_w, qs_r, vs); the addressing and the scan
    # take the injected queries and values
    step = make_staged_step(sdm, cfg, p, x, q_w, q_r, vs, alpha, beta, idx, wsel, v, banks, y, B,
                            T, ws_a, ws_s, first_write, st, stream, q_out=(qs_w, qs_r))

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(9)] for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        step(ev[i])
    t1.record(stream)
    torch.cuda.synchronize()
    if sdm.read_status(st) != 0:
        raise RuntimeError("device status %d in %s" % (sdm.read_status(st), name))
    ms = t0.elapsed_time(t1) / steps
    stage_ms = stage_times(ev)
    peak, _ = measured_peaks()
    per_tok = scan_bytes_per_token(wl)
    achieved = per_tok * ntok / (stage_ms["scan"] / 1e3) / 1e9
    line = {"workload": name, "B": B, "T": T, "d": d, "value": round(ntok / (ms / 1e3), 1),
            "unit": "tokens/s", "steps": steps, "ms_per_step": round(ms, 4),
            "stages_ms": {k: round(v_, 4) for k, v_ in stage_ms.items()},
            "scan_tokens_per_s": round(ntok / (stage_ms["scan"] / 1e3), 1),
            "scan_roofline": {"bound": "hbm", "bytes_per_token": per_tok,
                              "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                              "frac": round(achieved / peak, 4),
                              "vs_8tbs": round(achieved / 8000.0, 4)},
            "gpu_launches_per_step": 7}
    gi = idx.cpu().numpy()
    if pattern is not None:
        L, wa, ra = wl.pattern_len, wl.pattern_write_at, wl.pattern_read_at
        line["needle"] = {
            "what": "slots read by the %d pattern queries at %d.. equal the slots written at "
                    "%d.. (blog, needle-in-a-haystack access pattern)" % (L, ra, wa),
            "slot_sets_equal": bool(all(np.array_equal(gi[ra + i, 1], gi[wa + i, 0])
                                        for i in range(L)))}
    if pool is not None:
        m = pool["mask"].reshape(-1).numpy()
        pw = pool["pick_w"].reshape(-1).numpy()
        same = [np.all(gi[np.nonzero(m & (pw == vec))[0], 0] ==
                       gi[np.nonzero(m & (pw == vec))[0][0], 0]) for vec in range(wl.pool_size)
                if np.any(m & (pw == vec))]
        line["pool"] = {"tokens_from_pool": int(m.sum()),
                        "identical_sets_per_pool_vector": bool(all(same))}
    toks = np.sort(np.random.default_rng(7).choice(ntok, 128, replace=False))
    line["_sample"] = (name, address_sample(q_w, q_r, idx, toks))
    del banks, q_w, q_r, v, qs_w, qs_r, vs, idx, wsel, y, ws_a, ws_s, first_write, p, x
    torch.cuda.empty_cache()
    return line


# ------------------------------------------------------------- the CPU oracle

def address_checks(samples):
    """The slot-set check of every sampled workload, and the tiny fp32 workload run whole
    (its 256 tokens) free-running against the oracle."""
    import numpy as np
    import oracle
    import sparse_memory_linear_key_b300 as sdm
    out = {}
    for name, smp in samples:
        wl = synth.WORKLOADS[name]
        out[name] = address_check(wl, synth.make_params(wl, with_m0=False), smp)
    wl = synth.WORKLOADS["tiny-f32"]
    p = synth.make_params(wl)
    tok = synth.make_tokens(wl)
    cfg = sdm.make_cfg(wl.d, wl.n, wl.dk, wl.W, wl.dtype)
    pd = {k: v.cuda() for k, v in p.items()}
    banks = torch.empty(wl.B, wl.N, wl.d, device="cuda")
    sdm.sdm_init_bank(cfg, pd["M0"], banks)
    y = torch.empty(wl.B, wl.T, wl.d, device="cuda")
    idx = torch.empty(wl.B * wl.T, 2, wl.W, dtype=torch.int32, device="cuda")
    st = sdm.new_status()
    ws = sdm.alloc_workspace(sdm.workspace_bytes(cfg, wl.B, wl.T))
    sdm.sdm_prefill(cfg, pd, tok["x"].cuda(), tok["alpha"].cuda(), tok["beta"].cuda(), banks, y,
                    ws, st, idx_out=idx)
    gi = idx.cpu().numpy()
    ref = oracle.prefill_sequence(tok["x"][0], p, tok["alpha"][0], tok["beta"][0], wl.W)
    tiny = {"sampled_tokens": wl.T, "mode": "free-running (the oracle's own projections)"}
    for kind, S, g in ((0, ref["S"], ref["gap_w"]), (1, ref["R"], ref["gap_r"])):
        bad = np.any(np.sort(gi[:, kind], -1) != np.sort(S, -1), axis=1)
        tiny[("write", "read")[kind]] = {"mismatches": int(bad.sum()),
                                         "near_tie_mismatches": int((bad & (g < 1e-5)).sum())}
    tiny["max_abs_y_err"] = float(np.abs(y[0].cpu().numpy() - ref["y"]).max())
    out["tiny-f32"] = tiny
    return out


def oracle_sample(p_cpu, tok_cpu, n_tokens):
    """The oracle (as it stands) on sequence 0's first n_tokens of the workload, all
    rows: projections, exhaustive addressing and the recurrence. The bank it updates is a
    copy of M0 made before the clock starts (a 0.94 GB copy is set-up, not per-token
    work). Returns seconds."""
    import oracle
    wl = synth.WORKLOADS[WORKLOAD]
    M = oracle.storage(p_cpu["M0"])[0].copy()
    t = time.perf_counter()
    oracle.prefill_sequence(tok_cpu["x"][0, :n_tokens], p_cpu, tok_cpu["alpha"][0, :n_tokens],
                            tok_cpu["beta"][0, :n_tokens], wl.W, M=M)
    return time.perf_counter() - t


def oracle_threads():
    v = os.environ.get("OMP_NUM_THREADS")
    return int(v) if v else (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                             else os.cpu_count())


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _omp_threads(n):
    """Set the OpenMP thread count of the oracle's runtime (libgomp); returns the old one."""
    import ctypes
    import oracle
    oracle.lib()
    gomp = ctypes.CDLL("libgomp.so.1")
    old = gomp.omp_get_max_threads()
    gomp.omp_set_num_threads(int(n))
    return old


def cpu_baseline(p_cpu, tok_cpu):
    n = ORACLE_SAMPLE_TOKENS
    secs = oracle_sample(p_cpu, tok_cpu, n)
    n1 = 256
    old = _omp_threads(1)
    try:
        secs1 = oracle_sample(p_cpu, tok_cpu, n1)
    finally:
        _omp_threads(old)
    return {"value": round(n / secs, 2), "unit": "tokens/s", "cores": oracle_threads(),
            "kind": "oracle", "cpu_model": cpu_model(),
            "sample": "sequence 0, first %d tokens of %s, all 2048 rows (fp64 C oracle: "
                      "projections, exhaustive top-W over 230,400 slots, recurrence; the bank "
                      "copy of M0 made before the clock starts); %.1f s" % (n, WORKLOAD, secs),
            "single_thread": {"value": round(n1 / secs1, 2), "unit": "tokens/s", "cores": 1,
                              "sample": "the first %d tokens of the same sequence; %.1f s"
                                        % (n1, secs1)}}


REFERENCE_SAMPLE_TOKENS = 2048


def reference_arm(args, world, rank):
    """The oracle as the reference arm: each step one bounded sample of the workload
    (sequence 0's first 2,048 tokens, all rows, the bank copied from M0 before the clock
    starts), at most three timed steps."""
    if rank != 0:
        return None
    wl = synth.WORKLOADS[WORKLOAD]
    p_cpu = synth.make_params(wl)
    tok_cpu = synth.make_tokens(wl)
    n = REFERENCE_SAMPLE_TOKENS
    for _ in range(min(args.warmup, 1)):
        oracle_sample(p_cpu, tok_cpu, 16)
    times = [oracle_sample(p_cpu, tok_cpu, n) for _ in range(args.steps if args.steps <= 3 else 3)]
    secs = sum(times)
    value = n * len(times) / secs
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s",
        "n_gpus": world, "steps": len(times), "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / len(times), 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "B": wl.B, "T": wl.T, "d": wl.d, "N": wl.N, "W": wl.W,
                   "dk": wl.dk, "state": "bf16"},
        "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": oracle_threads(),
                         "kind": "oracle", "cpu_model": cpu_model(),
                         "sample": "per step: sequence 0, first %d tokens, all rows; the bank "
                                   "copy of M0 made before the clock starts" % n},
        "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        res = reference_arm(args, world, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if args.only_decode:
        import sparse_memory_linear_key_b300 as sdm
        from sparse_memory_linear_key_b300 import build
        build.build()
        res = {"metric": METRIC, "decode": decode_arm(sdm, args, world)}
        res["decode"].pop("_sample", None)
        if rank == 0:
            print(json.dumps(res), flush=True)
        barrier(world)
        return
    res, p_cpu, tok_cpu, samples = gpu_arm(args, world, rank)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(p_cpu, tok_cpu)
            res["address_check"] = address_checks(samples)
        print(json.dumps(res), flush=True)
    barrier(world)


if __name__ == "__main__":
    main()
