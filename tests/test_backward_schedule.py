"""The order of operations of the backward walk, pinned on the CPU.

The walk's kernel gathers a token's rows one token ahead: before the token processed
just before it (the next token in sequence order) has stored anything. It then takes
over, for every slot that token touched, the value that token left behind. Three things
come from a per-slot descriptor built beforehand:

- the position of the same slot in the next token;
- for a write slot, the read position of the same slot in its own token;
- whether the previous token in sequence order takes a position's value.

This file restates that schedule in numpy and checks it against the plain walk: each
token read and written in turn, in reverse. The plain walk is the per-token backward of
the gated-delta write and the weighted read ("Sparse Delta Memory" blog, "Write &
Read"). Inputs are crowded, every slot drawn from a small pool, so that nearly every
token needs the takeover. It also pins the index rule of the lane-exchange sum that the
kernel uses for its per-slot sums over rows.
"""
import numpy as np
import pytest


def plain_walk(idx, w, v, al, be, tape, bank, dy, G):
    T, _, W = idx.shape
    bank, G = bank.copy(), G.copy()
    out = {k: np.zeros(s) for k, s in (("dk", (T, W)), ("dr", (T, W)), ("da", T), ("db", T),
                                       ("dv", v.shape))}
    for t in range(T - 1, -1, -1):
        S, R, k, r = idx[t, 0], idx[t, 1], w[t, 0], w[t, 1]
        for j in range(W):
            out["dr"][t, j] = bank[R[j]] @ dy[t]
            G[R[j]] += r[j] * dy[t]
        old, gj = tape[t], G[S].copy()
        g, u = k @ gj, k @ old
        c = v[t] - al[t] * u
        out["dv"][t] = be[t] * g
        out["db"][t] = g @ c
        out["da"][t] = sum(gj[j] @ (old[j] - be[t] * k[j] * u) for j in range(W))
        out["dk"][t] = be[t] * gj @ c - al[t] * be[t] * old @ g
        for j in range(W):
            G[S[j]] = al[t] * (gj[j] - be[t] * k[j] * g)
            bank[S[j]] = old[j]
    return bank, G, out


def descriptors(idx):
    """Per token and position p (write p < W, read W + p): nxt[p], the position of p's slot in
    token t+1 (its write position if it has both) or -1; rm[j], the read position of write
    j's slot in token t or -1; rw[j], whether read j's slot is written by token t; need[p],
    whether token t-1 takes position p's final value from token t."""
    T, _, W = idx.shape
    nxt = np.full((T, 2 * W), -1)
    rm = np.full((T, W), -1)
    rw = np.zeros((T, W), bool)
    need = np.zeros((T, 2 * W), bool)
    for t in range(T):
        pos = list(np.concatenate([idx[t, 0], idx[t, 1]]))
        S, R = list(idx[t, 0]), list(idx[t, 1])
        if t + 1 < T:
            nx = list(np.concatenate([idx[t + 1, 0], idx[t + 1, 1]]))
            nxt[t] = [nx.index(s) if s in nx else -1 for s in pos]
        for j in range(W):
            rm[t, j] = R.index(S[j]) if S[j] in R else -1
            rw[t, j] = R[j] in S
        if t >= 1:
            prev = set(np.concatenate([idx[t - 1, 0], idx[t - 1, 1]]))
            for p, s in enumerate(pos):
                need[t, p] = s in prev and (p < W or s not in S)
    return nxt, rm, rw, need


def scheduled_walk(idx, w, v, al, be, tape, bank, dy, G):
    T, _, W = idx.shape
    bank, G = bank.copy(), G.copy()
    nxt, rm, rw, need = descriptors(idx)
    out = {k: np.zeros(s) for k, s in (("dk", (T, W)), ("dr", (T, W)), ("da", T), ("db", T),
                                       ("dv", v.shape))}

    def gather(t):   # before token t + 1 stores anything
        S, R = idx[t, 0], idx[t, 1]
        m = [tape[t + 1][nxt[t, W + j]] if 0 <= nxt[t, W + j] < W else bank[R[j]]
             for j in range(W)]
        return {"gw": G[S].copy(), "gr": G[R].copy(), "mr": np.stack(m)}

    ahead, left = gather(T - 1), None
    for t in range(T - 1, -1, -1):
        cur = ahead
        if t > 0:
            ahead = gather(t - 1)
        S, R, k, r = idx[t, 0], idx[t, 1], w[t, 0], w[t, 1]
        for j in range(W):   # values token t + 1 left behind
            if nxt[t, j] >= 0:
                cur["gw"][j] = left[nxt[t, j]]
            if nxt[t, W + j] >= 0:
                cur["gr"][j] = left[nxt[t, W + j]]
        new_r = cur["gr"] + r[:, None] * dy[t][None]
        for j in range(W):
            out["dr"][t, j] = cur["mr"][j] @ dy[t]
            if not rw[t, j]:
                G[R[j]] = new_r[j]
        gj = cur["gw"] + np.array([r[rm[t, j]] if rm[t, j] >= 0 else 0.0 for j in range(W)])[:, None] * dy[t][None]
        old = tape[t]
        g, u = k @ gj, k @ old
        c = v[t] - al[t] * u
        out["dv"][t] = be[t] * g
        out["db"][t] = g @ c
        out["da"][t] = sum(gj[j] @ (old[j] - be[t] * k[j] * u) for j in range(W))
        out["dk"][t] = be[t] * gj @ c - al[t] * be[t] * old @ g
        new_w = al[t] * (gj - be[t] * k[:, None] * g[None])
        left = np.full((2 * W, v.shape[1]), np.nan)   # only what token t - 1 takes
        for j in range(W):
            G[S[j]] = new_w[j]
            bank[S[j]] = old[j]
            if need[t, j]:
                left[j] = new_w[j]
            if need[t, W + j]:
                left[W + j] = new_r[j]
    return bank, G, out


@pytest.mark.parametrize("seed", range(6))
def test_scheduled_walk_equals_plain_walk(seed):
    rng = np.random.default_rng(seed)
    W, d = 8, 5
    N = int(rng.integers(W, 3 * W))           # a small pool: slots shared all the time
    T = int(rng.integers(1, 24))
    idx = np.stack([np.stack([rng.choice(N, W, replace=False), rng.choice(N, W, replace=False)])
                    for _ in range(T)])
    w = rng.random((T, 2, W))
    v = rng.standard_normal((T, d))
    al, be = rng.random(T), rng.random(T)
    bank0 = rng.standard_normal((N, d))
    bank, tape = bank0.copy(), np.zeros((T, W, d))
    for t in range(T):                        # the forward, recording the tape
        S, k = idx[t, 0], w[t, 0]
        tape[t] = bank[S]
        u = k @ tape[t]
        bank[S] = al[t] * tape[t] + be[t] * k[:, None] * (v[t] - al[t] * u)[None]
    dy, G0 = rng.standard_normal((T, d)), rng.standard_normal((N, d))
    b1, g1, o1 = plain_walk(idx, w, v, al, be, tape, bank, dy, G0)
    b2, g2, o2 = scheduled_walk(idx, w, v, al, be, tape, bank, dy, G0)
    assert np.array_equal(b1, bank0) and np.array_equal(b2, bank0)
    np.testing.assert_allclose(g2, g1, rtol=1e-12, atol=1e-12)   # a NaN here: a value not left
    for key in o1:
        np.testing.assert_allclose(o2[key], o1[key], rtol=1e-12, atol=1e-12, err_msg=key)


@pytest.mark.parametrize("V", [1, 2, 4, 8, 16])
def test_lane_exchange_sum_index_rule(V):
    """Each of V values summed over 32 lanes: at each step a lane keeps half of its values
    and trades the other half with the lane o = 32 h / V away (h the half), then plain
    exchanges finish; lane L ends with the sum of value L // (32 // V)."""
    rng = np.random.default_rng(V)
    x = rng.standard_normal((32, V))
    want = x.sum(0)
    y, h = x.copy(), V // 2
    while h >= 1:
        o, z = 32 * h // V, y.copy()
        for L in range(32):
            P, hi = L ^ o, bool(L & o)
            for k in range(h):
                keep = y[L, k + h] if hi else y[L, k]
                recv = y[P, k] if (P & o) else y[P, k + h]
                z[L, k] = keep + recv
        y, h = z, h // 2
    s, o = y[:, 0].copy(), 16 // V
    while o >= 1:
        s, o = s + s[np.arange(32) ^ o], o // 2
    for L in range(32):
        assert abs(s[L] - want[L // (32 // V)]) < 1e-12
