"""CPU oracle for one Sparse Delta Memory (SDM) layer forward pass.

TEST INFRASTRUCTURE ONLY: only `tests/`, `__graft_entry__.smoke()` and the
benchmark's CPU-baseline leg may import this package. The CUDA library never
imports, links or calls it, and it shares no code with the CUDA library.

The arithmetic lives in `sdm_oracle.c` (plain C, fp64, OpenMP over independent
rows/queries). This module builds it with gcc on first use and wraps it for numpy /
CPU torch tensors. The steps follow the Sparse Delta Memory blog post ("How does SDM
work?", "Write & Read") and the frozen readings:

- `project`:  q^w = x W_qw, q^r = x W_qr, v = x W_v, fp64 sums rounded once;
- `address`:  product-key scores s1, s2, exhaustive top-W of the outer sum with
  ties broken by smaller slot id, temperature-1 softmax over the kept scores;
- `scan`:     per token decay then delta rule on the write slots, then the
  softmax-weighted read of the read slots from the post-write bank.

Every function is pinned by tests/test_oracle_pins.py against closed forms,
hand-worked values, brute force on tiny inputs and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, BF16, F64 = 0, 1, 2
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile sdm_oracle.c into liboracle.so beside it (gcc, fp-contract off)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            P, I, L, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            _lib.orc_bf16_from_double.argtypes = [D]
            _lib.orc_bf16_from_double.restype = ctypes.c_uint16
            _lib.orc_round_store.argtypes = [P, L, I, P]
            _lib.orc_project.argtypes = [P, P, I, L, I, I, P]
            _lib.orc_subkey_scores.argtypes = [P, I, I, P, P, I, P, P]
            _lib.orc_topw.argtypes = [P, P, I, I, P, P, P]
            _lib.orc_softmax.argtypes = [P, I, P]
            _lib.orc_address.argtypes = [P, I, L, I, P, P, I, I, P, P, P, P]
            _lib.orc_scan.argtypes = [I, I, L, I, L, I, P, P, P, P, P, P, P, P, P]
            _lib.orc_scan.restype = I
            _lib.orc_init_bank.argtypes = [P, L, I, P]
    return _lib


# ------------------------------------------------------------------ conversions

def storage(a):
    """Return (contiguous numpy array, storage type) for a numpy array or CPU torch
    tensor. bf16 tensors become uint16 bit patterns."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                return a.view(torch.int16).numpy().view(np.uint16), BF16
            a = a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, BF16
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.float64:
        return a, F64
    raise TypeError("unsupported dtype %s" % a.dtype)


def to_f64(a) -> np.ndarray:
    """Exact fp64 values of a storage array (numpy/torch; bf16 as uint16 or torch)."""
    arr, t = storage(a)
    if t == BF16:
        return (arr.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return arr.astype(np.float64)


def _empty(shape, type_):
    return np.empty(shape, dtype={F32: np.float32, BF16: np.uint16, F64: np.float64}[type_])


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def round_to(values, type_) -> np.ndarray:
    """Round fp64 values once to a storage type (bf16 RNE / fp32 / fp64)."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = _empty(v.shape, type_)
    lib().orc_round_store(_p(v), v.size, type_, _p(out))
    return out


# ------------------------------------------------------------------- the steps

def project(x, Wm) -> np.ndarray:
    """x [rows, din] @ Wm [din, dout], fp64 sum, rounded once to the storage type."""
    xa, t = storage(x)
    wa, tw = storage(Wm)
    assert t == tw
    rows, din = xa.reshape(-1, xa.shape[-1]).shape
    dout = wa.shape[1]
    out = _empty((rows, dout), t)
    lib().orc_project(_p(xa), _p(wa), t, rows, din, dout, _p(out))
    return out.reshape(xa.shape[:-1] + (dout,))


def subkey_scores(q, K1, K2):
    """Sub-key scores of one query: (s1 [n], s2 [n]) in fp64."""
    qa, t = storage(q)
    k1, _ = storage(K1)
    k2, _ = storage(K2)
    n = k1.shape[0]
    s1 = np.empty(n)
    s2 = np.empty(n)
    lib().orc_subkey_scores(_p(qa), t, qa.shape[-1], _p(k1), _p(k2), n, _p(s1), _p(s2))
    return s1, s2


def topw(s1, s2, W):
    """Exhaustive top-W of the outer sum: (slots [W], scores [W], gap)."""
    s1 = np.ascontiguousarray(s1, dtype=np.float64)
    s2 = np.ascontiguousarray(s2, dtype=np.float64)
    slots = np.empty(W, dtype=np.int32)
    scores = np.empty(W)
    gap = np.empty(1)
    lib().orc_topw(_p(s1), _p(s2), len(s1), W, _p(slots), _p(scores), _p(gap))
    return slots, scores, float(gap[0])


def softmax(c) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.float64)
    w = np.empty_like(c)
    lib().orc_softmax(_p(c), len(c), _p(w))
    return w


def address(q, K1, K2, W):
    """Addressing of queries q [..., dk]: slots, weights, scores ([..., W]) and the
    boundary gap [...] between the W-th and (W+1)-th combined score."""
    qa, t = storage(q)
    k1, t1 = storage(K1)
    k2, _ = storage(K2)
    assert t == t1
    dk = qa.shape[-1]
    lead = qa.shape[:-1]
    nq = int(np.prod(lead)) if lead else 1
    n = k1.shape[0]
    slots = np.empty((nq, W), dtype=np.int32)
    weights = np.empty((nq, W))
    scores = np.empty((nq, W))
    gaps = np.empty(nq)
    lib().orc_address(_p(qa), t, nq, dk, _p(k1), _p(k2), n, W, _p(slots), _p(weights),
                      _p(scores), _p(gaps))
    return (slots.reshape(lead + (W,)), weights.reshape(lead + (W,)),
            scores.reshape(lead + (W,)), gaps.reshape(lead))


def scan(M, v, alpha, beta, S, k, Rd, r):
    """Recurrence of one sequence on a subset of rows.

    M [N, R] (storage array, updated IN PLACE; the selected rows of every slot),
    v [T, R] storage array, alpha/beta [T], S/Rd [T, W] int slot ids, k/r [T, W]
    weights. Returns y [T, R] (fp64)."""
    if not (isinstance(M, np.ndarray) and M.flags["C_CONTIGUOUS"]):
        raise ValueError("M must be a C-contiguous numpy array (it is updated in place)")
    Ma, tm = storage(M)
    va, tv = storage(v)
    N, R = Ma.shape
    T, W = np.asarray(S).shape
    al = np.ascontiguousarray(to_f64(alpha).reshape(T))
    be = np.ascontiguousarray(to_f64(beta).reshape(T))
    Sa = np.ascontiguousarray(S, dtype=np.int32)
    Ra = np.ascontiguousarray(Rd, dtype=np.int32)
    ka = np.ascontiguousarray(to_f64(k).reshape(T, W))
    ra = np.ascontiguousarray(to_f64(r).reshape(T, W))
    y = np.empty((T, R))
    rc = lib().orc_scan(tm, tv, N, R, T, W, _p(Ma), _p(va), _p(al), _p(be), _p(Sa), _p(ka),
                        _p(Ra), _p(ra), _p(y))
    if rc != 0:
        raise ValueError("oracle scan: slot id out of range or repeated within a set")
    return y


def init_bank(M0, B):
    """B copies of the learned initial state, [B, N, d] (storage array)."""
    m, t = storage(M0)
    banks = _empty((B,) + m.shape, t)
    lib().orc_init_bank(_p(m), m.nbytes, B, _p(banks))
    return banks


def prefill_sequence(x, params, alpha, beta, W, rows=None, M=None):
    """Whole layer for ONE sequence: project, address, scan.

    x [T, d]; params: W_qw, W_qr, W_v, K1, K2, M0 (storage tensors); alpha, beta [T];
    W active slots. rows: optional list of bank rows to carry (default all).
    M: optional starting bank rows [N, len(rows)] (default: M0 restricted to rows),
    updated in place. Returns q_w, q_r, v, write/read slots, weights and gaps, y, M."""
    q_w = project(x, params["W_qw"])
    q_r = project(x, params["W_qr"])
    v = project(x, params["W_v"])
    Sw, kw, _, gw = address(q_w, params["K1"], params["K2"], W)
    Sr, kr, _, gr = address(q_r, params["K1"], params["K2"], W)
    m0, _ = storage(params["M0"])
    d = m0.shape[1]
    all_rows = rows is None
    rows = np.arange(d) if all_rows else np.asarray(rows)
    if M is None:
        M = m0.copy() if all_rows else np.ascontiguousarray(m0[:, rows])
    vr = v if all_rows else np.ascontiguousarray(v[:, rows])
    y = scan(M, vr, alpha, beta, Sw, kw, Sr, kr)
    return {"q_w": q_w, "q_r": q_r, "v": v, "S": Sw, "k": kw, "gap_w": gw,
            "R": Sr, "r": kr, "gap_r": gr, "y": y, "M": M, "rows": rows}


# --------------------------------------------------------- slot-access statistics
# The pages' diagnostic of memory use (Sparse Delta Memory blog, "Memory Access Patterns
# on a Needle-in-a-Haystack Task": the slots written and read at each token position,
# and the write-read bucket overlap). Written as the set definitions, with numpy.

def slot_counts(idx, B, T, N, kind, t0, t1) -> np.ndarray:
    """counts[b, s] = number of tokens t in [t0, t1) of sequence b whose write (kind 0)
    or read (kind 1) set holds slot s. idx: [B*T, 2, W] int."""
    idx = np.asarray(idx).reshape(B, T, 2, -1)
    counts = np.zeros((B, N), np.int64)
    for b in range(B):
        for t in range(t0, t1):
            for s in set(int(v) for v in idx[b, t, kind]):
                if 0 <= s < N:
                    counts[b, s] += 1
    return counts


def slot_overlap(idx, B, T, N, w0, w1, r0, r1) -> np.ndarray:
    """Per sequence: [|written in [w0, w1)|, |read in [r0, r1)|, |both|] over distinct
    slot ids in [0, N)."""
    idx = np.asarray(idx).reshape(B, T, 2, -1)
    out = np.zeros((B, 3), np.int64)
    for b in range(B):
        wr = {int(s) for s in idx[b, w0:w1, 0].ravel() if 0 <= s < N}
        rd = {int(s) for s in idx[b, r0:r1, 1].ravel() if 0 <= s < N}
        out[b] = (len(wr), len(rd), len(wr & rd))
    return out


# ------------------------------------------------------- dense-state comparator
# The same gated delta rule on a dense state of W columns that every token updates
# (Sparse Delta Memory blog, "Background": SDM's W active slot vectors are the size of a
# gated-delta-net's whole dense state at identical FLOPs per token). Written out per
# token in fp64 with numpy, no rounding of the state.

def gdn_dense(S0, kw, kr, v, alpha, beta):
    """S0 [d, W] initial state (None: zeros); kw, kr [T, W] write / read weights; v [T, d];
    alpha, beta [T]. Per token: u = S k; S <- alpha S + beta (v - alpha u) k^T; y = S r.
    Returns (y [T, d], final S [d, W]), fp64."""
    kw = to_f64(kw)
    kr = to_f64(kr)
    v = to_f64(v)
    al = to_f64(alpha).reshape(-1)
    be = to_f64(beta).reshape(-1)
    T, W = kw.shape
    d = v.shape[1]
    S = np.zeros((d, W)) if S0 is None else to_f64(S0).reshape(d, W).copy()
    y = np.empty((T, d))
    for t in range(T):
        u = S @ kw[t]
        S = al[t] * S + be[t] * np.outer(v[t] - al[t] * u, kw[t])
        y[t] = S @ kr[t]
    return y, S


# ------------------------------------------------------------- backward (a5 + a6)
# Gradients of the recurrence by automatic differentiation of the per-token definition,
# written with plain PyTorch CPU ops in fp64. The state is stored once per token in the
# storage type (bf16 RNE or fp32) as the forward does; the rounding passes the gradient
# through unchanged (its derivative is taken as 1), which is what a backward pass that
# reuses the stored forward values computes.

def scan_backward(M_init, v, alpha, beta, S, k, Rd, r, dy, dM_final=None, type_=F32):
    """One sequence, a subset of rows. M_init [N, R] fp64 values, v [T, R], alpha/beta [T],
    S/Rd [T, W] slot ids, k/r [T, W] weights, dy [T, R]; dM_final [N, R] or None.
    Returns dict of fp64 numpy arrays: dM_init [N, R], dv [T, R], dalpha [T], dbeta [T],
    dk [T, W], dr [T, W]."""
    import torch
    f = torch.float64

    def store(x):
        if type_ == F64:
            return x
        if type_ == F32:
            q = x.detach().to(torch.float32).to(f)
        else:
            q = x.detach().to(torch.float32).to(torch.bfloat16).to(f)
        return x + (q - x).detach()

    M0 = torch.tensor(np.asarray(M_init, np.float64), dtype=f, requires_grad=True)
    vv = torch.tensor(to_f64(v), dtype=f, requires_grad=True)
    al = torch.tensor(to_f64(alpha).reshape(-1), dtype=f, requires_grad=True)
    be = torch.tensor(to_f64(beta).reshape(-1), dtype=f, requires_grad=True)
    kk = torch.tensor(to_f64(k), dtype=f, requires_grad=True)
    rr = torch.tensor(to_f64(r), dtype=f, requires_grad=True)
    S = np.asarray(S)
    Rd = np.asarray(Rd)
    T = S.shape[0]
    M = M0.clone()
    ys = []
    for t in range(T):
        s_idx = torch.as_tensor(S[t], dtype=torch.long)
        r_idx = torch.as_tensor(Rd[t], dtype=torch.long)
        old = M[s_idx]                                   # [W, R]
        u = kk[t] @ old                                  # [R]
        new = al[t] * old + be[t] * kk[t][:, None] * (vv[t] - al[t] * u)[None, :]
        M = M.index_copy(0, s_idx, store(new))
        ys.append(rr[t] @ M[r_idx])
    y = torch.stack(ys)
    loss = (y * torch.tensor(to_f64(dy), dtype=f)).sum()
    if dM_final is not None:
        loss = loss + (M * torch.tensor(np.asarray(dM_final, np.float64), dtype=f)).sum()
    loss.backward()
    return {"dM_init": M0.grad.numpy(), "dv": vv.grad.numpy(), "dalpha": al.grad.numpy(),
            "dbeta": be.grad.numpy(), "dk": kk.grad.numpy(), "dr": rr.grad.numpy(),
            "y": y.detach().numpy(), "M_final": M.detach().numpy()}


def address_backward(q, K1, K2, slots, dw):
    """Gradients of the selection weights with respect to the queries and sub-keys,
    the kept slots held fixed (the top-W selection is piecewise constant; the weights
    are a softmax of the kept combined scores c_j = <K1[i_j], q1> + <K2[l_j], q2>, slot
    i_j * n + l_j). q [ntok, dk], K1/K2 [n, dk/2], slots [ntok, W], dw [ntok, W].
    Autograd in fp64 with plain PyTorch CPU ops. Returns (w, dq, dK1, dK2) as numpy."""
    import torch
    f = torch.float64
    qq = torch.tensor(to_f64(q), dtype=f, requires_grad=True)
    k1 = torch.tensor(to_f64(K1), dtype=f, requires_grad=True)
    k2 = torch.tensor(to_f64(K2), dtype=f, requires_grad=True)
    n = k1.shape[0]
    h = k1.shape[1]
    sl = torch.as_tensor(np.asarray(slots), dtype=torch.long)
    i_idx, l_idx = sl // n, sl % n
    s1 = qq[:, :h] @ k1.T                          # [ntok, n]
    s2 = qq[:, h:] @ k2.T
    c = torch.gather(s1, 1, i_idx) + torch.gather(s2, 1, l_idx)
    w = torch.softmax(c, dim=1)
    (w * torch.tensor(np.asarray(dw, np.float64), dtype=f)).sum().backward()
    return w.detach().numpy(), qq.grad.numpy(), k1.grad.numpy(), k2.grad.numpy()


def project_backward(x, W_qw, W_qr, W_v, dq_w, dq_r, dv):
    """Gradients of q_w = x W_qw, q_r = x W_qr, v = x W_v (the rounding of the outputs
    passed through): dx = dq_w W_qw^T + dq_r W_qr^T + dv W_v^T, dW = x^T dout. fp64."""
    xx = to_f64(x)
    dqw, dqr, dvv = to_f64(dq_w), to_f64(dq_r), to_f64(dv)
    dx = dqw @ to_f64(W_qw).T + dqr @ to_f64(W_qr).T + dvv @ to_f64(W_v).T
    return dx, xx.T @ dqw, xx.T @ dqr, xx.T @ dvv
