"""Pins of the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes the oracle module and raises AssertionError if
it disagrees with a closed form, a hand-worked fixture under tests/golden/,
a library routine, brute force on tiny inputs or a Monte-Carlo estimate.
The mutation tests re-run them on deliberately broken copies of the oracle.
"""
from __future__ import annotations

import math
import os

import numpy as np
import scipy.linalg
import scipy.special
from scipy import integrate

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def _signs(d, seed):
    return (1 - 2 * np.random.default_rng(seed).integers(0, 2, d)).astype(np.int8)


# --- rotation ----------------------------------------------------------------

def pin_fwht_golden(o):
    for row in _golden_rows("fwht_worked.txt"):
        a, b = row.split(";")
        x = np.array(a.split(), dtype=np.float64)
        want = np.array(b.split(), dtype=np.float64)
        np.testing.assert_array_equal(o.fwht(x), want)
        np.testing.assert_array_equal(o.fwht(x.astype(np.float32)), want.astype(np.float32))


def pin_fwht_matches_library_hadamard(o):
    rng = np.random.default_rng(1)
    for d in (2, 8, 32, 128, 256):
        H = scipy.linalg.hadamard(d).astype(np.float64)
        y = rng.standard_normal((5, d))
        np.testing.assert_allclose(o.fwht(y), y @ H.T, rtol=0, atol=1e-11)
        np.testing.assert_array_equal(o.sylvester_hadamard(d), H)
        np.testing.assert_array_equal(H @ H, d * np.eye(d))


def pin_srht_orthogonal(o):
    rng = np.random.default_rng(2)
    d = 128
    D = _signs(d, 3)
    R = o.srht_matrix(D)
    np.testing.assert_allclose(R @ R.T, np.eye(d), atol=1e-12)
    x, y = rng.standard_normal((2, d))
    assert abs((R @ x) @ (R @ y) - x @ y) <= 1e-12 * np.linalg.norm(x) * np.linalg.norm(y)
    # float32 FWHT path: <Hx, Hy>/d = <x, y> to 1e-6 of |x||y|, ||Hx||/sqrt(d) = ||x||
    X = rng.standard_normal((64, d)).astype(np.float32)
    Y = rng.standard_normal((64, d)).astype(np.float32)
    zx = o.fwht(X * D.astype(np.float32)).astype(np.float64)
    zy = o.fwht(Y * D.astype(np.float32)).astype(np.float64)
    ip = np.sum(zx * zy, axis=1) / d
    ref = np.sum(X.astype(np.float64) * Y, axis=1)
    scale = np.linalg.norm(X.astype(np.float64), axis=1) * np.linalg.norm(Y.astype(np.float64), axis=1)
    assert np.max(np.abs(ip - ref) / scale) < 1e-6
    nz = np.linalg.norm(zx, axis=1) / math.sqrt(d)
    assert np.max(np.abs(nz / np.linalg.norm(X.astype(np.float64), axis=1) - 1)) < 1e-6


# --- analytic centroids --------------------------------------------------------

def pin_ids_are_nearest_centroids(o):
    """Brute force over all 2^m centroids (max <c, z_b>, ties to the lower id)."""
    rng = np.random.default_rng(4)
    for d, n_sub in ((128, 16), (32, 8), (16, 2)):
        m = d // n_sub
        # small integers so every <c, z> is exact and ties are real ties
        z = rng.integers(-3, 4, size=(200, d)).astype(np.float64)
        z[rng.random(z.shape) < 0.2] = 0.0
        z[0, :] = -0.0
        ids = o.sign_pattern_ids(z, n_sub)
        C = np.array([[-1.0 if (c >> j) & 1 else 1.0 for j in range(m)] for c in range(1 << m)])
        for i in range(z.shape[0]):
            for b in range(n_sub):
                s = C @ z[i, b * m:(b + 1) * m]
                best = int(np.flatnonzero(s == s.max())[0])
                assert ids[i, b] == best, (i, b)
        # the centroid helper is the +-1/sqrt(m) pattern of the same id
        for c in (0, 1, (1 << m) - 1):
            np.testing.assert_allclose(o.centroid(c, m), C[c] / math.sqrt(m))


def pin_top_rho_closed_form(o):
    """Top-rho by enumeration = the query's sign pattern with the cheapest
    coordinate subsets flipped (flipping set F costs 2 * sum_{j in F} |z_j|)."""
    rng = np.random.default_rng(5)
    m, n_sub = 8, 4
    for _ in range(20):
        # distinct powers of two: every subset sum is distinct and exact in float32
        mags = 2.0 ** rng.permutation(np.arange(-4, 4))
        z = np.concatenate([mags * np.where(rng.random(m) < 0.5, -1, 1) for _ in range(n_sub)])
        z = z.astype(np.float32)
        scores = o.centroid_scores_contract(z, n_sub)
        for rho in (1, 2, 4, 8):
            got = o.top_rho(scores, rho)
            for b in range(n_sub):
                zb = z[b * m:(b + 1) * m].astype(np.float64)
                base = sum(1 << j for j in range(m) if zb[j] < 0)
                costs = sorted((sum(abs(zb[j]) for j in range(m) if (f >> j) & 1), f)
                               for f in range(1 << m))
                want = [base ^ f for _, f in costs[:rho]]
                assert list(got[b]) == want
    # exact ties go to the lower centroid id: a zero subvector ties all 2^m
    # centroids; z = e_0 ties every centroid whose bit 0 is clear
    z = np.zeros(m * n_sub, dtype=np.float32)
    z[m] = 1.0
    z[2 * m + 1] = -2.0
    got = o.top_rho(o.centroid_scores_contract(z, n_sub), 4)
    assert list(got[0]) == [0, 1, 2, 3]
    assert list(got[1]) == [0, 2, 4, 6]
    assert list(got[2]) == [2, 3, 6, 7]


# --- quantiser levels -------------------------------------------------------

def _golden_closed_forms():
    out = {}
    for row in _golden_rows("beta_prior_closed_forms.txt"):
        k, v = row.split()
        out[k] = float(v)
    return out


def pin_levels_closed_forms(o):
    g = _golden_closed_forms()
    lev, thr = o.rsq_levels(3)
    np.testing.assert_allclose(lev, [g[f"m3_level_{t}"] for t in range(8)], atol=1e-12)
    np.testing.assert_allclose(thr, np.arange(1, 8) / 8.0, atol=1e-12)
    lev1, thr1 = o.rsq_levels(2, n_mag=1)
    assert abs(lev1[0] - g["m2_single_level"]) < 1e-12 and len(thr1) == 0


def _density(t, m):
    """Independent statement of the |x_j| density on [0, 1]:
    2 Gamma(m/2) / (sqrt(pi) Gamma((m-1)/2)) (1 - t^2)^((m-3)/2)."""
    c = 2 * math.gamma(m / 2) / (math.sqrt(math.pi) * math.gamma((m - 1) / 2))
    return c * (1 - t * t) ** ((m - 3) / 2)


def pin_levels_quadrature(o):
    """Density integrates to 1, E[x^2] = 1/m, and the levels are a Lloyd-Max
    fixed point (cell means, midpoint thresholds) under independent quadrature."""
    for m in (4, 8, 16):
        tot = integrate.quad(lambda t: _density(t, m), 0, 1, epsabs=1e-14)[0]
        ex2 = integrate.quad(lambda t: t * t * _density(t, m), 0, 1, epsabs=1e-14)[0]
        assert abs(tot - 1) < 1e-10 and abs(ex2 - 1 / m) < 1e-10
        lev, thr = o.rsq_levels(m)
        np.testing.assert_allclose(thr, 0.5 * (lev[1:] + lev[:-1]), atol=1e-15)
        edges = np.concatenate([[0.0], thr, [1.0]])
        for t in range(8):
            a, b = edges[t], edges[t + 1]
            mass = integrate.quad(lambda s: _density(s, m), a, b, epsabs=1e-15, epsrel=1e-13)[0]
            mom = integrate.quad(lambda s: s * _density(s, m), a, b, epsabs=1e-15, epsrel=1e-13)[0]
            assert abs(mom / mass - lev[t]) < 1e-10, (m, t)
        cdf = o.abs_coordinate_cdf(np.array([0.3, 0.7]), m)
        for tv, cv in zip((0.3, 0.7), cdf):
            assert abs(integrate.quad(lambda s: _density(s, m), 0, tv, epsabs=1e-14)[0] - cv) < 1e-10


def pin_levels_monte_carlo(o):
    """Sampled sphere directions: empirical cell means match the levels and
    the MSE beats the uniform 8-level quantiser."""
    m = 8
    rng = np.random.default_rng(6)
    g = rng.standard_normal((1_250_000, m))
    x = np.abs((g / np.linalg.norm(g, axis=1, keepdims=True)).ravel())
    assert abs(np.mean(x * x) - 1 / m) < 1e-3
    lev, thr = o.rsq_levels(m)
    t = np.searchsorted(thr, x, side="left")
    for c in range(8):
        assert abs(x[t == c].mean() - lev[c]) < 1.5e-3
    mse = np.mean((x - lev[t]) ** 2)
    uni = (np.minimum(np.floor(x * 8), 7) + 0.5) / 8
    assert mse < np.mean((x - uni) ** 2)


# --- encoding and estimator ---------------------------------------------------

def pin_estimator_exact_when_lossless(o):
    """With v = x the estimator ||q|| sum_b w_b <v_b, q~_b> equals <k, q>."""
    rng = np.random.default_rng(7)
    d, n_sub = 128, 16
    D = _signs(d, 8)
    K = rng.standard_normal((300, d)) * np.exp(0.5 * rng.standard_normal(d))
    K[5] = 0.0
    q = rng.standard_normal(d)
    enc = o.encode_ideal(K, D, n_sub, levels=None)
    qn, qt = o.query_prep_ideal(q, D)
    est = o.estimator_ideal(enc["v"], enc["w"], qn, qt)
    ref = K @ q
    assert np.max(np.abs(est - ref)) <= 1e-9 * np.max(np.abs(ref))
    assert est[5] == 0.0


def pin_estimator_level_scale_invariant(o):
    rng = np.random.default_rng(9)
    d, n_sub = 128, 16
    D = _signs(d, 10)
    K = rng.standard_normal((100, d))
    q = rng.standard_normal(d)
    lev, thr = o.rsq_levels(8)
    qn, qt = o.query_prep_ideal(q, D)
    e1 = o.encode_ideal(K, D, n_sub, lev, thr)
    e2 = o.encode_ideal(K, D, n_sub, 2.5 * lev, thr)
    np.testing.assert_array_equal(e1["nib"], e2["nib"])
    a = o.estimator_ideal(e1["v"], e1["w"], qn, qt)
    b = o.estimator_ideal(e2["v"], e2["w"], qn, qt)
    np.testing.assert_allclose(a, b, rtol=1e-12)
    # the quantised estimator tracks <k, q> (4-bit codes: a few percent)
    ref = K @ q
    assert np.sqrt(np.mean((a - ref) ** 2)) < 0.08 * np.sqrt(np.mean(ref ** 2))


def pin_w_simplified_form(o):
    """w = ||k|| ||u_b|| / <v,x> equals n_b / (sqrt(d) <v,x>) with z = H D k."""
    rng = np.random.default_rng(11)
    d, n_sub = 128, 16
    m = d // n_sub
    D = _signs(d, 12)
    K = rng.standard_normal((50, d))
    lev, thr = o.rsq_levels(m)
    e = o.encode_ideal(K, D, n_sub, lev, thr)
    z = (K * D) @ scipy.linalg.hadamard(d).T
    nb = np.linalg.norm(z.reshape(50, n_sub, m), axis=2)
    vx = np.sum(e["v"] * e["x"], axis=2)
    np.testing.assert_allclose(e["w"], nb / (math.sqrt(d) * vx), rtol=1e-12)


def pin_codes_nearest_level(o):
    """The magnitude index picks the nearest level (Lloyd-Max thresholds are
    midpoints); the sign bit is the coordinate's sign."""
    rng = np.random.default_rng(13)
    lev, thr = o.rsq_levels(8)
    x = rng.random(20000)
    t = o.magnitude_index(x, thr)
    brute = np.argmin(np.abs(x[:, None] - lev[None, :]), axis=1)
    np.testing.assert_array_equal(t, brute)
    # a magnitude exactly on a threshold is equidistant from two levels: the
    # lower level wins (ties to the lower index)
    np.testing.assert_array_equal(o.magnitude_index(thr, thr), np.arange(7))
    nib = np.array([0, 7, 8, 15, 3, 11])
    np.testing.assert_allclose(o.dequantise(nib, lev), [lev[0], lev[7], -lev[0], -lev[7], lev[3], -lev[3]])
    packed = o.pack_codes(np.array([[1, 2, 3, 4]], dtype=np.uint8))
    np.testing.assert_array_equal(packed, [[0x21, 0x43]])
    np.testing.assert_array_equal(o.unpack_codes(packed), [[1, 2, 3, 4]])


def pin_contract_tracks_ideal(o):
    """The float32 contract encoding and rerank agree with float64 within
    float32 rounding (decisions differ only next to a decision boundary)."""
    rng = np.random.default_rng(14)
    d, n_sub = 128, 16
    D = _signs(d, 15)
    K = (rng.standard_normal((4000, d)) * np.exp(0.5 * rng.standard_normal(d))).astype(np.float32)
    lev, thr = o.rsq_levels(8)
    l32, t32 = lev.astype(np.float32), thr.astype(np.float32)
    ec = o.encode_contract(K, D, n_sub, l32, t32)
    ei = o.encode_ideal(K.astype(np.float64), D, n_sub, l32.astype(np.float64), t32.astype(np.float64))
    assert np.mean(ec["ids"] == ei["ids"]) > 0.9999
    same = np.all(ec["nib"].reshape(-1, n_sub, 8) == ei["nib"].reshape(-1, n_sub, 8), axis=2)
    assert same.mean() > 0.999
    # w scale: ideal w carries sqrt(d) ||k|| ||u_b|| / ... in units of k; same definition
    np.testing.assert_allclose(ec["w"][same], ei["w"][same], rtol=2e-5)
    q = (K[17] + 0.5 * rng.standard_normal(d)).astype(np.float32)
    qp = o.query_prep_contract(q, D, n_sub, 4)
    qn, qt = o.query_prep_ideal(q.astype(np.float64), D)
    assert abs(qp["qnorm"] - qn) < 1e-6 * qn
    np.testing.assert_allclose(qp["qt"], qt, atol=1e-6)
    rows = np.flatnonzero(same.all(axis=1))[:500]
    est_c = o.rerank_contract(ec["nib"][rows], ec["w"][rows], qp["qnorm"], qp["qt"], l32, n_sub)
    est_i = o.estimator_ideal(ei["v"][rows], ei["w"][rows], qn, qt)
    assert np.max(np.abs(est_c - est_i)) < 1e-4 * np.max(np.abs(est_i))


# --- votes, candidates, top-k --------------------------------------------------

def pin_votes(o):
    rng = np.random.default_rng(16)
    d, n_sub, m = 128, 16, 8
    D = _signs(d, 17)
    K = rng.standard_normal((500, d)).astype(np.float32)
    lev, thr = o.rsq_levels_f32(m)
    ids = o.encode_contract(K, D, n_sub, lev, thr)["ids"]
    q = rng.standard_normal(d).astype(np.float32)
    # every centroid selected: each key is hit in every subspace
    qp = o.query_prep_contract(q, D, n_sub, 1 << m, "flat")
    assert np.all(o.votes(ids, qp["lut"]) == n_sub)
    qp = o.query_prep_contract(q, D, n_sub, 1 << m, "rank")
    assert np.all(qp["lut"] > 0)
    # rho = 1, flat: count subspaces whose id equals the query's own sign pattern
    qp = o.query_prep_contract(q, D, n_sub, 1, "flat")
    qid = o.sign_pattern_ids(qp["z"][None, :], n_sub)[0]
    np.testing.assert_array_equal(o.votes(ids, qp["lut"]), np.sum(ids == qid[None, :], axis=1))
    # rank weights by explicit loops over the hot lists
    qp = o.query_prep_contract(q, D, n_sub, 4, "rank")
    got = o.votes(ids, qp["lut"])
    for i in range(0, 500, 37):
        s = 0
        for b in range(n_sub):
            for r in range(4):
                if ids[i, b] == qp["hot_ids"][b, r]:
                    s += 4 - r
        assert got[i] == s


def pin_candidate_counts(o):
    for row in _golden_rows("candidate_counts.txt"):
        n, bp, k, c = map(int, row.split())
        assert o.candidate_count(n, bp, k) == c, row


def _check_ordered_selection(keys, chosen, c, listed="index"):
    """chosen must be the c best by (key desc, index asc), listed by ascending
    index or (listed="key") in that order."""
    keys = np.asarray(keys)
    n = len(keys)
    assert len(chosen) == c and len(set(chosen.tolist())) == c
    if listed == "key":
        dk, di = np.diff(keys[chosen].astype(np.float64)), np.diff(chosen)
        assert np.all((dk < 0) | ((dk == 0) & (di > 0)))
        chosen = np.sort(chosen)
    assert np.all(np.diff(chosen) > 0)
    if c == 0 or c == n:
        return
    sel = np.zeros(n, bool)
    sel[chosen] = True
    thr = keys[sel].min()
    assert np.all(keys[~sel] <= thr)
    eq = np.flatnonzero(keys == thr)
    taken = sel[eq]
    # among keys equal to the threshold the lowest indices are taken first
    assert np.all(np.diff(taken.astype(int)) <= 0)


def pin_selection(o):
    rng = np.random.default_rng(18)
    for n in (1, 7, 64, 300):
        for c in sorted({0, 1, n // 3, n}):
            s = rng.integers(0, 5, n)
            _check_ordered_selection(s, o.select_candidates(s, c), c)
            est = rng.integers(-3, 3, n).astype(np.float32) * 0.5
            est[rng.random(n) < 0.1] = -0.0
            cand = np.sort(rng.choice(10 * n, n, replace=False))
            ti, te = o.topk(est, cand, c)
            pos = np.searchsorted(cand, ti)
            _check_ordered_selection(est + 0.0, pos, c, listed="key")
            np.testing.assert_array_equal(te, est[pos])
    assert len(o.select_candidates(np.arange(10), 10)) == 10


def pin_recall_one_at_full_candidates(o):
    """100% candidates and a lossless quantiser: the pipeline's top-k is the
    exact top-k of <k, q> (ideal arithmetic)."""
    rng = np.random.default_rng(19)
    d, n_sub = 128, 16
    D = _signs(d, 20)
    K = rng.standard_normal((2000, d))
    q = K[123] + 0.5 * rng.standard_normal(d)
    enc = o.encode_ideal(K, D, n_sub, levels=None)
    qn, qt = o.query_prep_ideal(q, D)
    cand = np.arange(2000)
    est = o.estimator_ideal(enc["v"], enc["w"], qn, qt)
    top, _ = o.topk(est, cand, 64)
    assert o.recall(top, o.exact_topk(K, q, 64)) == 1.0
    # and listed best first, as a library sort of the exact products lists them
    np.testing.assert_array_equal(top, np.argsort(-(K @ q), kind="stable")[:64])


# --- the composed retrieval (coarse candidates -> rerank -> top-k) -------------

def _keys_with_duplicates(rng, n, d, n_dup):
    """float32 keys [n, d] where n_dup rows repeat earlier rows (equal bucket
    ids and equal estimates), so votes and estimates tie.  Returns the keys
    and the repeated rows."""
    K = rng.standard_normal((n, d)).astype(np.float32)
    dups = rng.choice(np.arange(1, n), size=n_dup, replace=False) if n > 1 else np.zeros(0, np.int64)
    for r in dups:
        K[r] = K[rng.integers(0, r)]
    return K, dups


def _row_estimates(o, enc, q32, D, n_sub, lev):
    """Estimate of every row on its own (a row's estimate does not depend on
    which other rows are candidates), one row per call of the rerank."""
    qp = o.query_prep_contract(q32, D, n_sub, 1, "flat")
    return np.array([o.rerank_contract(enc["nib"][i:i + 1], enc["w"][i:i + 1], qp["qnorm"], qp["qt"], lev, n_sub)[0]
                     for i in range(enc["nib"].shape[0])], dtype=np.float32)


def pin_pipeline_full_candidates(o):
    """Candidates = 100% (cand_bp = 10000): the pipeline's top-k is the first k
    of every row sorted by (estimate desc, index asc), the brute-force top-k of
    the estimator over the whole zone; equal estimates from duplicated keys
    go to the lower index."""
    rng = np.random.default_rng(23)
    d, n_sub, m = 128, 16, 8
    D = _signs(d, 24)
    lev, thr = o.rsq_levels_f32(m)
    for n, k in ((300, 40), (97, 97), (50, 200)):
        K, dups = _keys_with_duplicates(rng, n, d, n // 5)
        enc = o.encode_contract(K, D, n_sub, lev, thr)
        q = (K[dups[0]] + 0.1 * rng.standard_normal(d)).astype(np.float32)  # near a key that has a copy
        r = o.retrieve_contract(enc, q, D, n_sub, 4, 10000, k, lev)
        est = _row_estimates(o, enc, q, D, n_sub, lev)
        want = sorted(range(n), key=lambda i: (-float(est[i]), i))[:min(k, n)]
        assert r["C"] == n and r["k_eff"] == min(k, n)
        np.testing.assert_array_equal(r["cand"], np.arange(n))
        np.testing.assert_array_equal(r["top_idx"], want)
        np.testing.assert_array_equal(r["top_est"].view(np.uint32), est[want].view(np.uint32))
        assert len(set(est[want].tolist())) < len(want), "the case must hold equal estimates in the top-k"


def pin_pipeline_tiny_full_sort(o):
    """N <= 64 with duplicated keys: the votes are the hot-list weights summed
    by explicit loops, the candidates the first C of a full sort by (votes
    desc, index asc), the top-k the first min(k, C) candidates of a full sort
    by (estimate desc, index asc), and k_eff = min(k, C)."""
    rng = np.random.default_rng(25)
    d, n_sub, m = 128, 16, 8
    D = _signs(d, 26)
    lev, thr = o.rsq_levels_f32(m)
    cases = ((64, 2500, 30, 4), (64, 1000, 5, 2), (40, 3000, 100, 8), (17, 10000, 3, 1), (1, 500, 4, 4))
    for n, bp, k, rho in cases:
        K, _ = _keys_with_duplicates(rng, n, d, n // 4)
        enc = o.encode_contract(K, D, n_sub, lev, thr)
        q = (K[n // 2] + 0.5 * rng.standard_normal(d)).astype(np.float32)
        r = o.retrieve_contract(enc, q, D, n_sub, rho, bp, k, lev)
        qp = r["qp"]
        votes = np.zeros(n, dtype=np.int64)
        for i in range(n):
            for b in range(n_sub):
                for rr in range(rho):
                    if enc["ids"][i, b] == qp["hot_ids"][b, rr]:
                        votes[i] += rho - rr
        np.testing.assert_array_equal(r["votes"], votes)
        c = max(-(-bp * n // 10000), min(k, n))
        c = min(c, n)
        cand = sorted(sorted(range(n), key=lambda i: (-int(votes[i]), i))[:c])
        assert r["C"] == c and r["k_eff"] == min(k, c)
        np.testing.assert_array_equal(r["cand"], cand)
        est = _row_estimates(o, enc, q, D, n_sub, lev)
        np.testing.assert_array_equal(r["est"].view(np.uint32), est[cand].view(np.uint32))
        top = sorted(cand, key=lambda i: (-float(est[i]), i))[:min(k, c)]
        np.testing.assert_array_equal(r["top_idx"], top)
        np.testing.assert_array_equal(r["top_est"].view(np.uint32), est[top].view(np.uint32))
    # the cases above must include candidates that are not a prefix of the zone and k > C
    assert any(min(max(-(-bp * n // 10000), min(k, n)), n) < k for n, bp, k, _ in cases)


def pin_recall_hand_made_sets(o):
    """recall = |found intersect truth| / |truth|, each position once."""
    assert o.recall(np.array([1, 2, 3, 4]), np.array([3, 4, 5, 6])) == 0.5
    assert o.recall(np.array([3, 3, 3, 9]), np.array([3, 4])) == 0.5
    assert o.recall(np.array([], dtype=np.int64), np.array([1, 2, 3])) == 0.0
    assert o.recall(np.array([5, 6]), np.array([], dtype=np.int64)) == 1.0
    assert o.recall(np.array([7, 1, 5]), np.array([1, 5, 7])) == 1.0
    assert o.recall(np.array([2]), np.array([1, 2, 3, 4, 5])) == 0.2


# --- attention and zones ---------------------------------------------------

def pin_attention_dense(o):
    rng = np.random.default_rng(21)
    d, T = 128, 300
    K = rng.standard_normal((T, d))
    V = rng.standard_normal((T, d))
    q = rng.standard_normal(d)
    dense = scipy.special.softmax(K @ q / math.sqrt(d)) @ V
    z = o.Zones(16, 64, 32)
    z.prefill(250)
    for _ in range(50):
        z.append()
    rows = np.concatenate([z.sink(), z.retrieval(), z.local(), z.buffer()])
    np.testing.assert_array_equal(np.sort(rows), np.arange(T))
    np.testing.assert_allclose(o.attention(q, K[rows], V[rows]), dense, atol=1e-12)
    perm = rng.permutation(T)
    np.testing.assert_allclose(o.attention(q, K[perm], V[perm]), dense, atol=1e-12)


def pin_zones(o):
    """Against an explicit per-token label list updated by the zone rules."""
    rng = np.random.default_rng(22)
    for S, L, U, T0 in ((16, 64, 32, 500), (4, 8, 4, 3), (0, 5, 2, 0), (16, 512, 128, 100)):
        z = o.Zones(S, L, U)
        z.prefill(T0)
        lab = ["S" if p < S else None for p in range(T0)]
        rest = [p for p in range(T0) if p >= S]
        for p in rest[:len(rest) - min(L, len(rest))]:
            lab[p] = "R"
        for p in rest[len(rest) - min(L, len(rest)):]:
            lab[p] = "L"
        for _ in range(int(rng.integers(50, 400))):
            p = len(lab)
            z.append()
            if p < S:
                lab.append("S")
                continue
            lab.append("B")
            if lab.count("B") == U:
                lab = ["L" if x == "B" else x for x in lab]
                loc = [i for i, x in enumerate(lab) if x == "L"]
                for i in loc[:max(0, len(loc) - L)]:
                    lab[i] = "R"
            for name, want in (("sink", "S"), ("retrieval", "R"), ("local", "L"), ("buffer", "B")):
                np.testing.assert_array_equal(getattr(z, name)(),
                                              [i for i, x in enumerate(lab) if x == want])
            assert z.n_local <= L


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
