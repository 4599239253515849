"""Pins of the CPU oracle against facts that do not come from the oracle itself:
hand-worked examples (tests/golden/), closed forms, invariants, and brute force on
tiny inputs written in a different form (dense matrices, full sorts).

Each test names the passage of the Sparse Delta Memory pages, or the property of
the frozen specification, that it pins."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- bf16 storage

def test_bf16_rounding_matches_fp32_cast_on_floats():
    """Storage rounding (the state is stored in bf16, each written value rounded once to
nearest, ties to even): for values that are already fp32, rounding
    to bf16 must equal the standard fp32 -> bf16 round-to-nearest-even cast."""
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    got = oracle.round_to(f.astype(np.float64), oracle.BF16)
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # values that overflow past the largest bf16 go to inf in both
    assert np.array_equal(got, want)


def test_bf16_rounding_single_step_and_ties():
    r = oracle.lib().orc_bf16_from_double
    assert r(1.0) == 0x3F80
    assert r(1.0 + 2.0**-8) == 0x3F80            # halfway -> even (down)
    assert r(1.0 + 3 * 2.0**-8) == 0x3F82        # halfway -> even (up)
    # just above halfway: one rounding step gives 0x3F81; rounding through fp32
    # first would give 0x3F80, so this pins the single rounding from fp64.
    assert r(1.0 + 2.0**-8 + 2.0**-40) == 0x3F81
    assert r(-1.0 - 2.0**-8 - 2.0**-40) == 0xBF81
    assert r(2.0**-133) == 0x0001                 # smallest subnormal
    assert r(2.0**-134) == 0x0000                 # halfway to zero -> even
    assert r(3.0 * 2.0**-134) == 0x0002           # 1.5 ulp -> even (2)
    assert r(3.4e38) == 0x7F80                    # beyond the largest finite -> inf
    assert r(0.0) == 0x0000 and r(-0.0) == 0x8000


# ---------------------------------------------------------------- projections

def test_project_exact_on_integers():
    """Step P is a plain matrix product: with small integers every product and sum
    is exact, so the result must equal integer matrix multiplication."""
    rng = np.random.default_rng(1)
    x = rng.integers(-8, 9, size=(7, 33)).astype(np.float32)
    w = rng.integers(-8, 9, size=(33, 19)).astype(np.float32)
    want = (x.astype(np.int64) @ w.astype(np.int64)).astype(np.float32)
    got = oracle.project(x, w)
    assert got.dtype == np.float32 and np.array_equal(got, want)
    # bf16 inputs: integers up to 8 are exact in bf16; sums up to 33*64 = 2112 need
    # 12 bits, so the stored bf16 value is the sum rounded once (RNE)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    wb = torch.from_numpy(w).to(torch.bfloat16)
    gotb = oracle.to_f64(oracle.project(xb, wb))
    wantb = torch.from_numpy(want).to(torch.bfloat16).float().numpy()   # exact int -> RNE
    assert np.array_equal(gotb, wantb.astype(np.float64))


# ---------------------------------------------------------------- addressing

def test_product_key_hand_example():
    g = _load("product_key_3x3.json")
    q = np.array(g["q"], dtype=np.float32)
    K1 = np.array(g["K1"], dtype=np.float32)
    K2 = np.array(g["K2"], dtype=np.float32)
    s1, s2 = oracle.subkey_scores(q, K1, K2)
    assert np.array_equal(s1, g["s1"]) and np.array_equal(s2, g["s2"])
    for case in g["cases"]:
        slots, scores, gap = oracle.topw(s1, s2, case["W"])
        assert slots.tolist() == case["slots"]
        assert scores.tolist() == case["scores"]
        assert gap == case["gap"]
        if "weights" in case:
            S, w, sc, gp = oracle.address(q[None], K1, K2, case["W"])
            assert S[0].tolist() == case["slots"]
            np.testing.assert_allclose(w[0], case["weights"], rtol=0, atol=1e-15)


def _brute_topw(s1, s2, W):
    """Exhaustive top-W by a full sort of all n*n sums: larger first, ties by id."""
    n = len(s1)
    c = np.add.outer(s1, s2).ravel()
    ids = np.arange(n * n)
    order = np.lexsort((ids, -c))
    return ids[order[:W]], c[order[:W]], (c[order[W - 1]] - c[order[W]]) if n * n > W else math.inf


@pytest.mark.parametrize("n,W,seed,integer", [(4, 3, 0, False), (8, 8, 1, False),
                                              (16, 5, 2, True), (32, 32, 3, True),
                                              (64, 64, 4, False), (20, 16, 5, True)])
def test_topw_matches_full_sort(n, W, seed, integer):
    """Step A.4: the selected set is the top-W of all n^2 outer sums (brute force on
    tiny n, with many exact ties when the scores are small integers)."""
    rng = np.random.default_rng(seed)
    if integer:
        s1 = rng.integers(-3, 4, n).astype(np.float64)
        s2 = rng.integers(-3, 4, n).astype(np.float64)
    else:
        s1, s2 = rng.standard_normal(n), rng.standard_normal(n)
    slots, scores, gap = oracle.topw(s1, s2, W)
    bs, bc, bg = _brute_topw(s1, s2, W)
    assert slots.tolist() == bs.tolist()
    assert np.array_equal(scores, bc)
    assert gap == bg


def _pruned_topw(s1, s2, W):
    """The product-key route the CUDA path uses: top-W of each half (sorted, ties by
    index), candidates with 1-based ranks a*b <= W, top-W of those."""
    n = len(s1)
    o1 = np.lexsort((np.arange(n), -s1))[:W]
    o2 = np.lexsort((np.arange(n), -s2))[:W]
    cand = [(s1[i] + s2[j], i * n + j) for a, i in enumerate(o1) for b, j in enumerate(o2)
            if (a + 1) * (b + 1) <= W]
    cand.sort(key=lambda t: (-t[0], t[1]))
    return [c[1] for c in cand[:W]]


@pytest.mark.parametrize("seed", range(12))
def test_product_key_route_is_exact(seed):
    """The product-key route ("Write & Read": two sub-keys -> outer sum -> top-k): with
    W <= n, pruning to per-half top-W and rank products
    a*b <= W keeps the exact top-W of all n^2 sums (continuous scores, no ties)."""
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(8, 65))
    W = int(rng.integers(1, n + 1))
    s1, s2 = rng.standard_normal(n), rng.standard_normal(n)
    slots, _, _ = oracle.topw(s1, s2, W)
    assert sorted(slots.tolist()) == sorted(_pruned_topw(s1, s2, W))


def test_subkey_scores_exact_on_integers():
    rng = np.random.default_rng(7)
    n, h = 24, 16
    K1 = rng.integers(-4, 5, (n, h)).astype(np.float32)
    K2 = rng.integers(-4, 5, (n, h)).astype(np.float32)
    q = rng.integers(-4, 5, 2 * h).astype(np.float32)
    s1, s2 = oracle.subkey_scores(q, K1, K2)
    assert np.array_equal(s1, K1.astype(np.int64) @ q[:h].astype(np.int64))
    assert np.array_equal(s2, K2.astype(np.int64) @ q[h:].astype(np.int64))


def test_softmax_properties():
    rng = np.random.default_rng(3)
    for W in (1, 2, 8, 64):
        c = np.sort(rng.standard_normal(W) * 3)[::-1].copy()
        w = oracle.softmax(c)
        assert abs(w.sum() - 1.0) < 1e-12
        assert np.all(np.diff(w) <= 0)          # monotone with the score
        # closed form of each ratio: w_i / w_j = exp(c_i - c_j)
        np.testing.assert_allclose(w[:-1] / w[1:] if W > 1 else [1.0],
                                   np.exp(c[:-1] - c[1:]) if W > 1 else [1.0], rtol=1e-12)
    assert oracle.softmax(np.array([5.0]))[0] == 1.0
    # shift invariance (max-subtracted): adding a constant leaves the weights
    c = rng.standard_normal(16)
    np.testing.assert_allclose(oracle.softmax(c), oracle.softmax(c + 1000.0), rtol=1e-12)


# ---------------------------------------------------------------- the recurrence

def _scan1(M, v, alpha, beta, S, k, R, r):
    T = 1
    return oracle.scan(M, np.asarray(v)[None], np.array([alpha]), np.array([beta]),
                       np.asarray(S, dtype=np.int32)[None], np.asarray(k, dtype=np.float64)[None],
                       np.asarray(R, dtype=np.int32)[None], np.asarray(r, dtype=np.float64)[None])


def test_delta_rule_hand_example():
    g = _load("delta_rule_2slot.json")
    for case in g["cases"]:
        M = np.eye(2, dtype=np.float64)               # slot-major: M[slot] = column
        y = _scan1(M, np.array(g["v"]), case["alpha"], g["beta"], g["slots"], g["k"],
                   g["slots"], g["k"])
        np.testing.assert_allclose(M, case["M_S_columns"], rtol=0, atol=1e-14)
        np.testing.assert_allclose(y[0], case["read_with_k"], rtol=0, atol=1e-14)


def _rand_bank(rng, N, R, dtype=np.float64):
    return np.ascontiguousarray(rng.standard_normal((N, R)).astype(dtype))


def test_decay_only_invariant():
    """beta = 0: the selected columns scale by alpha, nothing else changes (bits)."""
    rng = np.random.default_rng(11)
    N, R, W = 40, 6, 5
    M = _rand_bank(rng, N, R)
    M0 = M.copy()
    S = rng.choice(N, W, replace=False)
    Rd = rng.choice(N, W, replace=False)
    alpha = 0.731
    _scan1(M, rng.standard_normal(R), alpha, 0.0, S, oracle.softmax(rng.standard_normal(W)),
           Rd, oracle.softmax(rng.standard_normal(W)))
    assert np.array_equal(M[S], alpha * M0[S])
    rest = np.setdiff1d(np.arange(N), S)
    assert np.array_equal(M[rest], M0[rest])


def test_idempotence_invariant():
    """beta = 1, |k| = 1, R = S, r = k: the read returns v (up to fp64 rounding of
    a + (v - a), i.e. one ulp, for one-hot k)."""
    rng = np.random.default_rng(12)
    N, R = 30, 8
    v = rng.standard_normal(R)
    for alpha in (1.0, 0.5, 0.93):
        M = _rand_bank(rng, N, R)
        S = [4, 17, 22]
        k = [0.0, 1.0, 0.0]
        y = _scan1(M, v, alpha, 1.0, S, k, S, k)
        # the rounding error of a + (v - a) is one ulp of max(|a|, |v|) (|a| < 5 here)
        np.testing.assert_allclose(y[0], v, rtol=0, atol=5 * 2.3e-16)
        M = _rand_bank(rng, N, R)
        y = _scan1(M, v, alpha, 1.0, [3, 9], [0.6, 0.8], [3, 9], [0.6, 0.8])
        np.testing.assert_allclose(y[0], v, rtol=0, atol=1e-13)


def test_read_after_write_closed_form():
    """R = S, r = k: y = alpha (1 - beta |k|^2) u + beta |k|^2 v, u = M_S k before
    the write (the read follows this token's write, "How does SDM work?"; softmax weights,
    so |k| < 1)."""
    rng = np.random.default_rng(13)
    N, R, W = 200, 10, 16
    for _ in range(5):
        M = _rand_bank(rng, N, R)
        S = rng.choice(N, W, replace=False)
        k = oracle.softmax(rng.standard_normal(W) * 2)
        v = rng.standard_normal(R)
        a, b = rng.uniform(0.5, 1), rng.uniform(0, 1)
        u = k @ M[S]
        y = _scan1(M, v, a, b, S, k, S, k)
        kk = float(k @ k)
        np.testing.assert_allclose(y[0], a * (1 - b * kk) * u + b * kk * v, rtol=0, atol=1e-12)


def test_repeated_identical_query_closed_form():
    """The same (S, k, v, alpha, beta) for T tokens: M_S(T) = M_S(0) A^T + B sum A^i
    with A = alpha (I - beta k k^T), B = beta v k^T (column-matrix form)."""
    rng = np.random.default_rng(14)
    N, R, W, T = 50, 7, 6, 9
    M = _rand_bank(rng, N, R)
    S = rng.choice(N, W, replace=False)
    k = oracle.softmax(rng.standard_normal(W))
    v = rng.standard_normal(R)
    a, b = 0.9, 0.6
    MS0 = M[S].T.copy()                                       # d x W column form
    A = a * (np.eye(W) - b * np.outer(k, k))
    Bm = b * np.outer(v, k)
    want = MS0 @ np.linalg.matrix_power(A, T) + Bm @ sum(np.linalg.matrix_power(A, i)
                                                          for i in range(T))
    oracle.scan(M, np.tile(v, (T, 1)), np.full(T, a), np.full(T, b), np.tile(S, (T, 1)),
                np.tile(k, (T, 1)), np.tile(S, (T, 1)), np.tile(k, (T, 1)))
    np.testing.assert_allclose(M[S].T, want, rtol=0, atol=1e-12)


def test_disjoint_tokens_commute():
    rng = np.random.default_rng(15)
    N, R, W, T = 300, 5, 4, 6
    perm = rng.permutation(N)
    S = perm[:T * W].reshape(T, W)
    Rd = rng.choice(N, (T, W))
    Rd = np.stack([rng.choice(N, W, replace=False) for _ in range(T)])
    k = np.stack([oracle.softmax(rng.standard_normal(W)) for _ in range(T)])
    r = np.stack([oracle.softmax(rng.standard_normal(W)) for _ in range(T)])
    v = rng.standard_normal((T, R))
    al, be = rng.uniform(0.5, 1, T), rng.uniform(0, 1, T)
    M0 = _rand_bank(rng, N, R)
    M1 = M0.copy()
    oracle.scan(M1, v, al, be, S, k, Rd, r)
    o = rng.permutation(T)
    M2 = M0.copy()
    oracle.scan(M2, v[o], al[o], be[o], S[o], k[o], Rd[o], r[o])
    assert np.array_equal(M1, M2)


def test_row_subset_is_independent():
    """Rows of M and y evolve independently: the delta rule and the read act on each row
    of the selected slot vectors separately (bits, bf16 storage)."""
    rng = np.random.default_rng(16)
    N, d, W, T = 64, 24, 8, 20
    M0 = torch.randn(N, d, generator=torch.Generator().manual_seed(1)).mul(0.1).to(torch.bfloat16)
    v = torch.randn(T, d, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    S = np.stack([rng.choice(N, W, replace=False) for _ in range(T)])
    Rd = np.stack([rng.choice(N, W, replace=False) for _ in range(T)])
    k = np.stack([oracle.softmax(rng.standard_normal(W)) for _ in range(T)])
    r = np.stack([oracle.softmax(rng.standard_normal(W)) for _ in range(T)])
    al, be = rng.uniform(0.5, 1, T), rng.uniform(0, 1, T)
    Mfull, _ = oracle.storage(M0)
    Mfull = Mfull.copy()
    vfull, _ = oracle.storage(v)
    y_full = oracle.scan(Mfull, vfull, al, be, S, k, Rd, r)
    rows = np.array([0, 5, 6, 23])
    Msub = np.ascontiguousarray(oracle.storage(M0)[0][:, rows])
    y_sub = oracle.scan(Msub, np.ascontiguousarray(vfull[:, rows]), al, be, S, k, Rd, r)
    assert np.array_equal(Msub, Mfull[:, rows])
    assert np.array_equal(y_sub, y_full[:, rows])


def _nearest_bf16(x):
    """Brute-force nearest bf16 of a double (ties to even) from the bracketing
    bit patterns around the fp32 value."""
    f = np.float32(x)
    base = int(np.array([f]).view(np.uint32)[0] >> 16)
    best = None
    for b in range(base - 2, base + 3):
        val = float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0])
        key = (abs(val - x), b & 1)
        if best is None or key < best[0]:
            best = (key, b)
    return best[1]


def test_bf16_state_is_rounded_once_per_write():
    """bf16 storage: each written value is the nearest bf16 of the exact fp64
    update (decay then delta from the stored inputs), unwritten values keep bits."""
    rng = np.random.default_rng(17)
    N, R, W = 20, 6, 4
    Mb = oracle.round_to(rng.standard_normal((N, R)) * 0.3, oracle.BF16)
    M64 = oracle.to_f64(Mb)
    v = oracle.round_to(rng.standard_normal(R), oracle.BF16)
    S = [2, 7, 11, 19]
    k = oracle.softmax(rng.standard_normal(W))
    a, b = 0.87, 0.41
    M = Mb.copy()
    _scan1(M, v, a, b, S, k, S, k)
    vf = oracle.to_f64(v)
    u = k @ (a * M64[S])
    for jj, s in enumerate(S):
        for c in range(R):
            exact = a * M64[s, c] + b * (vf[c] - u[c]) * k[jj]
            assert M[s, c] == _nearest_bf16(exact)
    rest = [i for i in range(N) if i not in S]
    assert np.array_equal(M[rest], Mb[rest])


# ------------------------------------------------------ whole layer, brute force

def _dense_layer(x, Wqw, Wqr, Wv, K1, K2, M0, alpha, beta, W):
    """Dense brute force of one sequence: M is a d x N matrix, the outer sum is
    formed in full, the update is the matrix form alpha M_S (I - beta k k^T) +
    beta v k^T, the read is M_R r (all fp64)."""
    d, N = M0.shape[1], M0.shape[0]
    n = K1.shape[0]
    h = K1.shape[1]
    M = M0.T.copy()
    ys = []
    for t in range(x.shape[0]):
        qw, qr, v = x[t] @ Wqw, x[t] @ Wqr, x[t] @ Wv

        def sel(q):
            c = np.add.outer(K1 @ q[:h], K2 @ q[h:]).ravel()
            o = np.lexsort((np.arange(N), -c))[:W]
            e = np.exp(c[o] - c[o].max())
            return o, e / e.sum()
        S, k = sel(qw)
        R, r = sel(qr)
        M[:, S] = alpha[t] * M[:, S] @ (np.eye(W) - beta[t] * np.outer(k, k)) + \
            beta[t] * np.outer(v, k)
        ys.append(M[:, R] @ r)
    return np.array(ys), M.T


@pytest.mark.parametrize("seed,n,W,d,dk,T", [(0, 6, 4, 5, 4, 12), (1, 8, 8, 7, 6, 20),
                                             (2, 5, 2, 3, 8, 15)])
def test_whole_layer_vs_dense_brute_force(seed, n, W, d, dk, T):
    rng = np.random.default_rng(200 + seed)
    x = rng.standard_normal((T, d))
    Wqw, Wqr = rng.standard_normal((d, dk)), rng.standard_normal((d, dk))
    Wv = rng.standard_normal((d, d))
    K1, K2 = rng.standard_normal((n, dk // 2)), rng.standard_normal((n, dk // 2))
    M0 = rng.standard_normal((n * n, d)) * 0.1
    al, be = rng.uniform(0.5, 1, T), rng.uniform(0, 1, T)
    y_ref, M_ref = _dense_layer(x, Wqw, Wqr, Wv, K1, K2, M0, al, be, W)
    params = {"W_qw": Wqw, "W_qr": Wqr, "W_v": Wv, "K1": K1, "K2": K2, "M0": M0}
    out = oracle.prefill_sequence(x, params, al, be, W)
    np.testing.assert_allclose(out["y"], y_ref, rtol=0, atol=1e-11)
    np.testing.assert_allclose(out["M"], M_ref, rtol=0, atol=1e-11)


def test_init_bank_is_a_copy():
    rng = np.random.default_rng(5)
    M0 = oracle.round_to(rng.standard_normal((30, 8)), oracle.BF16)
    banks = oracle.init_bank(M0, 3)
    assert banks.shape == (3, 30, 8)
    for b in range(3):
        assert np.array_equal(banks[b], M0)


# ------------------------------------------------------------ slot-access statistics

def test_slot_stats_hand_example():
    """Three tokens, two slots each (blog, "Memory Access Patterns": cumulative writes,
    current reads, write-read bucket overlap), worked by hand:
    writes {1,2}, {2,4}, {6,7}; reads {2,3}, {1,5}, {7,1}."""
    idx = np.array([[[1, 2], [2, 3]], [[2, 4], [1, 5]], [[6, 7], [7, 1]]])
    w = oracle.slot_counts(idx, 1, 3, 8, 0, 0, 3)
    assert w.tolist() == [[0, 1, 2, 0, 1, 0, 1, 1]]
    r = oracle.slot_counts(idx, 1, 3, 8, 1, 1, 3)
    assert r.tolist() == [[0, 2, 0, 0, 0, 1, 0, 1]]
    # written in tokens 0-1: {1,2,4}; read in tokens 1-2: {1,5,7}; both: {1}
    assert oracle.slot_overlap(idx, 1, 3, 8, 0, 2, 1, 3).tolist() == [[3, 3, 1]]
    # an empty write window; all reads: {2,3} | {1,5} | {7,1} = {1,2,3,5,7}
    assert oracle.slot_overlap(idx, 1, 3, 8, 1, 1, 0, 3).tolist() == [[0, 5, 0]]


def test_slot_stats_invariants():
    rng = np.random.default_rng(11)
    B, T, W, N = 3, 40, 4, 64
    idx = np.stack([np.stack([rng.choice(N, W, replace=False) for _ in range(2)])
                    for _ in range(B * T)])
    c = oracle.slot_counts(idx, B, T, N, 0, 5, 30)
    assert np.all(c.sum(1) == 25 * W)          # distinct ids: one count per reference
    o = oracle.slot_overlap(idx, B, T, N, 5, 30, 10, 40)
    assert np.all(o[:, 2] <= np.minimum(o[:, 0], o[:, 1]))
    # the distinct written slots are exactly the slots with a nonzero count
    assert np.array_equal(o[:, 0], (c > 0).sum(1))
    # a window against itself with the read sets equal to the write sets: full overlap
    same = idx.copy()
    same[:, 1] = same[:, 0]
    o2 = oracle.slot_overlap(same, B, T, N, 0, T, 0, T)
    assert np.array_equal(o2[:, 0], o2[:, 2]) and np.array_equal(o2[:, 1], o2[:, 2])
    # out-of-range ids are not counted
    bad = idx.copy()
    bad[0, 0, 0] = N
    assert oracle.slot_counts(bad, B, T, N, 0, 0, 1)[0].sum() == W - 1


# ------------------------------------------------------- dense-state comparator

def test_gdn_dense_is_the_scan_on_a_fixed_slot_set():
    """The dense comparator is the SDM recurrence with every token selecting the same
    W slots of a W-slot bank: the numpy dense form against the C scan (fp64 storage, so
    no rounding on either side)."""
    rng = np.random.default_rng(21)
    T, W, d = 40, 8, 12
    S0 = rng.normal(size=(d, W))
    kw = rng.dirichlet(np.ones(W), size=T)
    kr = rng.dirichlet(np.ones(W), size=T)
    v = rng.normal(size=(T, d))
    al = rng.uniform(0.5, 1.0, T)
    be = rng.uniform(0.0, 1.0, T)
    y, S = oracle.gdn_dense(S0, kw, kr, v, al, be)
    M = np.ascontiguousarray(S0.T)                       # [N = W slots, d rows]
    sets = np.tile(np.arange(W, dtype=np.int32), (T, 1))
    y2 = oracle.scan(M, v, al, be, sets, kw, sets, kr)
    np.testing.assert_allclose(y, y2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S, M.T, rtol=0, atol=1e-12)


def test_gdn_dense_closed_forms():
    d, W = 5, 4
    rng = np.random.default_rng(22)
    S0 = rng.normal(size=(d, W))
    e = np.eye(W)
    # beta = 0: pure decay, y = alpha S0 r
    y, S = oracle.gdn_dense(S0, e[[1]], e[[2]], rng.normal(size=(1, d)), [0.5], [0.0])
    np.testing.assert_allclose(S, 0.5 * S0, atol=1e-15)
    np.testing.assert_allclose(y[0], 0.5 * S0[:, 2], atol=1e-15)
    # beta = 1, one-hot k, r = k: the write is read back exactly (idempotence)
    v = rng.normal(size=(1, d))
    y, S = oracle.gdn_dense(S0, e[[3]], e[[3]], v, [0.7], [1.0])
    np.testing.assert_allclose(y[0], v[0], atol=1e-14)
    np.testing.assert_allclose(S[:, :3], 0.7 * S0[:, :3], atol=1e-15)


# ------------------------------------------------------------- backward (a5 + a6)

def _bwd_case(seed, T=6, N=10, W=3, R=4):
    rng = np.random.default_rng(seed)
    M0 = rng.normal(size=(N, R))
    v = rng.normal(size=(T, R))
    al = rng.uniform(0.5, 1.0, T)
    be = rng.uniform(0.1, 0.9, T)
    S = np.stack([np.sort(rng.choice(N, W, replace=False)) for _ in range(T)])
    Rd = np.stack([np.sort(rng.choice(N, W, replace=False)) for _ in range(T)])
    S[2] = Rd[2]                      # a token that reads exactly what it writes
    k = rng.dirichlet(np.ones(W), size=T)
    r = rng.dirichlet(np.ones(W), size=T)
    dy = rng.normal(size=(T, R))
    dMf = rng.normal(size=(N, R))
    return M0, v, al, be, S, k, Rd, r, dy, dMf


def test_scan_backward_forward_values_are_the_scan():
    M0, v, al, be, S, k, Rd, r, dy, dMf = _bwd_case(31)
    g = oracle.scan_backward(M0, v, al, be, S, k, Rd, r, dy, dMf, type_=oracle.F64)
    M = np.ascontiguousarray(M0.copy())
    y = oracle.scan(M, v, al, be, S, k, Rd, r)
    np.testing.assert_allclose(g["y"], y, atol=1e-12)
    np.testing.assert_allclose(g["M_final"], M, atol=1e-12)


def test_scan_backward_matches_finite_differences():
    """Central differences of L = <y, dy> + <M_final, dM> through the C scan (fp64
    storage), against the autograd gradients, for every input family."""
    M0, v, al, be, S, k, Rd, r, dy, dMf = _bwd_case(32)
    g = oracle.scan_backward(M0, v, al, be, S, k, Rd, r, dy, dMf, type_=oracle.F64)

    def loss(M0_, v_, al_, be_, k_, r_):
        M = np.ascontiguousarray(M0_.copy())
        y = oracle.scan(M, v_, al_, be_, S, k_, Rd, r_)
        return float((y * dy).sum() + (M * dMf).sum())

    base = [M0, v, al, be, k, r]
    names = ["dM_init", "dv", "dalpha", "dbeta", "dk", "dr"]
    h = 1e-6
    for a_i, name in enumerate(names):
        arr = base[a_i]
        flat = arr.reshape(-1)
        for e in range(0, flat.size, max(1, flat.size // 7)):
            plus = [b.copy() for b in base]
            minus = [b.copy() for b in base]
            plus[a_i].reshape(-1)[e] += h
            minus[a_i].reshape(-1)[e] -= h
            fd = (loss(*plus) - loss(*minus)) / (2 * h)
            assert abs(fd - g[name].reshape(-1)[e]) <= 1e-6 * max(1.0, abs(fd)), (name, e)


def test_scan_backward_closed_form_single_token():
    """One token, W = 1, R = S: y = alpha m + beta k (v - alpha k m) k-weighted read.
    With k = r = 1 (W = 1): y = alpha m + beta (v - alpha m) = alpha (1 - beta) m + beta v,
    so dy/dv = beta, dy/dm = alpha (1 - beta), dy/dalpha = (1 - beta) m,
    dy/dbeta = v - alpha m."""
    m, vv, a, b = 0.7, -1.3, 0.8, 0.25
    g = oracle.scan_backward(np.array([[m]]), np.array([[vv]]), [a], [b], np.array([[0]]),
                             np.array([[1.0]]), np.array([[0]]), np.array([[1.0]]),
                             np.array([[1.0]]), None, type_=oracle.F64)
    assert abs(g["dv"][0, 0] - b) < 1e-14
    assert abs(g["dM_init"][0, 0] - a * (1 - b)) < 1e-14
    assert abs(g["dalpha"][0] - (1 - b) * m) < 1e-14
    assert abs(g["dbeta"][0] - (vv - a * m)) < 1e-14


def test_address_backward_matches_finite_differences():
    """The selection weights as a function of q and the sub-keys with the kept slots
    fixed, differentiated by central differences of the plain formula."""
    rng = np.random.default_rng(41)
    ntok, n, h, W = 3, 5, 4, 4
    q = rng.normal(size=(ntok, 2 * h))
    K1 = rng.normal(size=(n, h))
    K2 = rng.normal(size=(n, h))
    slots = np.stack([rng.choice(n * n, W, replace=False) for _ in range(ntok)])
    dw = rng.normal(size=(ntok, W))

    def loss(q_, K1_, K2_):
        i, l = slots // n, slots % n
        c = np.einsum("th,tjh->tj", q_[:, :h], K1_[i]) + np.einsum("th,tjh->tj", q_[:, h:], K2_[l])
        e = np.exp(c - c.max(1, keepdims=True))
        return float(((e / e.sum(1, keepdims=True)) * dw).sum())

    w, dq, dK1, dK2 = oracle.address_backward(q, K1, K2, slots, dw)
    i, l = slots // n, slots % n
    c = np.einsum("th,tjh->tj", q[:, :h], K1[i]) + np.einsum("th,tjh->tj", q[:, h:], K2[l])
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-12)
    np.testing.assert_allclose(w, np.stack([oracle.softmax(row) for row in c]), atol=1e-12)
    hh = 1e-6
    for arr, grad, which in ((q, dq, 0), (K1, dK1, 1), (K2, dK2, 2)):
        for e_ in range(arr.size):
            args = [q.copy(), K1.copy(), K2.copy()]
            args[which].reshape(-1)[e_] += hh
            up = loss(*args)
            args[which].reshape(-1)[e_] -= 2 * hh
            fd = (up - loss(*args)) / (2 * hh)
            assert abs(fd - grad.reshape(-1)[e_]) < 1e-7, (which, e_)


def test_project_backward_is_autograd_of_the_projections():
    import torch
    rng = np.random.default_rng(51)
    ntok, d, dk = 5, 6, 4
    x = rng.normal(size=(ntok, d))
    Ws = [rng.normal(size=(d, dk)), rng.normal(size=(d, dk)), rng.normal(size=(d, d))]
    douts = [rng.normal(size=(ntok, dk)), rng.normal(size=(ntok, dk)), rng.normal(size=(ntok, d))]
    xt = torch.tensor(x, requires_grad=True)
    Wt = [torch.tensor(w, requires_grad=True) for w in Ws]
    loss = sum(((xt @ w) * torch.tensor(g)).sum() for w, g in zip(Wt, douts))
    loss.backward()
    dx, dW1, dW2, dW3 = oracle.project_backward(x, *Ws, *douts)
    np.testing.assert_allclose(dx, xt.grad.numpy(), atol=1e-12)
    for got, w in zip((dW1, dW2, dW3), Wt):
        np.testing.assert_allclose(got, w.grad.numpy(), atol=1e-12)
