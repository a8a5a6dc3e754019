"""ParisKV CPU oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of the ParisKV decode-time
KV-cache retrieval path, written from "ParisKV: Fast and Drift-Robust
KV-Cache Retrieval for Long-Context LLMs" (gist.science summary of arXiv
2602.07721), section "Methodology: the ParisKV framework".  Only the test
suite, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import this module.  The CUDA library never imports it,
shares no code with it and must not fall back to it.

Two arithmetic modes
--------------------
* ideal (float64): the literal definitions -- normalise, rotate with the
  dense orthogonal matrix R = H D / sqrt(d), split, quantise the unit
  subspace direction, calibrate.  Used for the invariants and for recall.
* contract (float32): the same steps with every operation rounded to
  float32 (round to nearest even, no fused multiply-add) in one fixed order.
  The CUDA kernels follow the same order, so every decision that floating
  point turns into an integer (bucket id, 4-bit code, top-rho centroid,
  candidate set, top-k set) is taken in the same precision on both sides and
  agrees bit for bit.  The order of every sum is stated in the docstring of
  the function that computes it.

Readings of points the pages leave open:
R1 SRHT = H_d diag(D) / sqrt(d), no subsampling (d is a power of two), one D
   shared by keys and queries of a layer; D is an input.
R2 normalise-then-rotate equals rotate-then-divide-by-norm; ids and codes
   depend only on the direction of each rotated subvector, so the contract
   mode works on the unnormalised rotation z = H (D * k).
R3 subspace b = coordinates [b*m, (b+1)*m); bucket id bit j = [z_{b,j} < 0]
   (a zero, either sign, counts as positive).
R4 "Beta prior" levels: for x uniform on S^{m-1}, x_j^2 ~ Beta(1/2, (m-1)/2);
   8 magnitude levels by Lloyd-Max on |x_j|, rounded to float32 once.
R5 w_{i,b} = ||k|| ||u_b|| / <v_b, x_b>  (u = R k/||k||, x_b = u_b/||u_b||),
   which is n_b / (sqrt(d) <v_b, x_b>) with n_b = ||z_b||; w = 0 if n_b = 0.
R6 "hierarchical" vote weights: the centroid of rank r (0-based) among the
   query's top-rho of a subspace gives rho - r votes; a flat mode gives 1.
R7 C = max(ceil(p N), min(k, N)) with p in basis points, capped at N.
R8 ties go to the lower index everywhere (token position, centroid id).
R9 attention: scale 1/sqrt(d), softmax over Sink U Local U Buffer U top-k.
R10 zones: prefill puts the first S tokens in Sink, the last L in Local and
   the rest in Retrieval; an append that fills the U-token Update Buffer
   moves the buffer into Local and evicts Local's oldest tokens beyond L.
R11 GQA: retrieval runs per query head; key-side tables are per KV head.
R13 a zero query (||z_q|| = 0) has q_tilde = 0, so every estimate is 0.

Pins (tests/test_oracle_pins.py): the FWHT against the Sylvester matrix,
orthogonality and inner-product preservation of R; nearest-centroid ids by
brute force over all 2^m centroids; the Lloyd-Max levels against closed
forms (m = 3 gives the uniform quantiser, m = 2 with one level gives 2/pi),
against Monte-Carlo samples of the sphere and against independent
quadrature; the estimator exact under a lossless quantiser; rho = 2^m giving
uniform votes; candidate selection and top-k against a full sort;
sparse attention with everything retrieved against dense softmax attention;
the zone bookkeeping against a brute-force token list; each float32 contract
function against its float64 counterpart within float32 rounding bounds.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import beta as beta_fn
from scipy.special import betainc, betaincinv

F32 = np.float32

# ----------------------------------------------------------------------------
# Rotation (ParisKV, Methodology 1: "Normalization and Rotation" -- keys and
# queries are l2-normalised and share a random orthogonal rotation realised as
# an SRHT).
# ----------------------------------------------------------------------------


def fwht(y: np.ndarray) -> np.ndarray:
    """Unnormalised Walsh-Hadamard transform along the last axis (Sylvester order).

    Stage order h = 1, 2, 4, ..., d/2; in stage h every pair (i, i + h) with
    i & h == 0 becomes (y_i + y_{i+h}, y_i - y_{i+h}).  The dtype of ``y`` is
    kept, so a float32 input is rounded after every add and subtract.
    """
    y = np.array(y, copy=True)
    d = y.shape[-1]
    if d & (d - 1):
        raise ValueError("length must be a power of two")
    lead = y.shape[:-1]
    h = 1
    while h < d:
        v = y.reshape(lead + (d // (2 * h), 2, h))
        a = v[..., 0, :].copy()
        b = v[..., 1, :].copy()
        v[..., 0, :] = a + b
        v[..., 1, :] = a - b
        h *= 2
    return y


def sylvester_hadamard(d: int) -> np.ndarray:
    """H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]] as float64 [d, d]."""
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    if h.shape[0] != d:
        raise ValueError("d must be a power of two")
    return h


def srht_matrix(signs: np.ndarray) -> np.ndarray:
    """R = H_d diag(D) / sqrt(d), float64 [d, d] (reading R1)."""
    d = len(signs)
    return sylvester_hadamard(d) * np.asarray(signs, dtype=np.float64)[None, :] / math.sqrt(d)


# ----------------------------------------------------------------------------
# Quantiser levels (ParisKV, Methodology 2, "Candidate reranking (RSQ-IP)":
# 4-bit codes, 1 sign bit + 3 magnitude bits, levels from the rotation-induced
# Beta prior).
# ----------------------------------------------------------------------------


def abs_coordinate_cdf(t, m: int):
    """P(|x_j| <= t) for x uniform on S^{m-1}: x_j^2 ~ Beta(1/2, (m-1)/2)."""
    t = np.asarray(t, dtype=np.float64)
    return betainc(0.5, (m - 1) / 2.0, t * t)


def abs_coordinate_partial_mean(lo, hi, m: int):
    """E[|x_j| ; lo < |x_j| <= hi].

    With u = x_j^2 ~ Beta(1/2, b), b = (m-1)/2:  sqrt(u) * u^{-1/2} (1-u)^{b-1}
    / B(1/2, b) = (B(1, b) / B(1/2, b)) * [Beta(1, b) density], so the partial
    mean is B(1, b)/B(1/2, b) * (I_{hi^2}(1, b) - I_{lo^2}(1, b)).
    """
    b = (m - 1) / 2.0
    c = beta_fn(1.0, b) / beta_fn(0.5, b)
    return c * (betainc(1.0, b, hi * hi) - betainc(1.0, b, lo * lo))


def rsq_levels(m: int, n_mag: int = 8, tol: float = 1e-15, max_iter: int = 200000):
    """Lloyd-Max quantiser of |x_j| under the Beta prior, float64.

    Returns (levels[n_mag], thresholds[n_mag - 1]), levels ascending in (0, 1),
    thresholds the midpoints of adjacent levels.  Starts at the mid-quantiles
    (t + 1/2)/n_mag and alternates "thresholds = midpoints" and "levels =
    conditional means of their cells" until no level moves by more than tol.
    """
    if m < 2:
        raise ValueError("subspace width m must be >= 2")
    b = (m - 1) / 2.0
    lev = np.sqrt(betaincinv(0.5, b, (np.arange(n_mag) + 0.5) / n_mag))
    for _ in range(max_iter):
        edges = np.concatenate([[0.0], 0.5 * (lev[1:] + lev[:-1]), [1.0]])
        mass = abs_coordinate_cdf(edges[1:], m) - abs_coordinate_cdf(edges[:-1], m)
        new = abs_coordinate_partial_mean(edges[:-1], edges[1:], m) / mass
        change = np.max(np.abs(new - lev))
        lev = new
        if change < tol:
            break
    return lev, 0.5 * (lev[1:] + lev[:-1])


def rsq_levels_f32(m: int, n_mag: int = 8):
    """The float32 tables used by the contract mode: levels and midpoints,
    each rounded from float64 once (reading R4)."""
    lev, thr = rsq_levels(m, n_mag)
    return lev.astype(F32), thr.astype(F32)


# ----------------------------------------------------------------------------
# Key encoding (ParisKV, Methodology 2: bucket ids by nearest analytic
# centroid, RSQ-IP codes, calibration w_{i,b} precomputed at prefill).
# ----------------------------------------------------------------------------


def sign_pattern_ids(z: np.ndarray, n_sub: int) -> np.ndarray:
    """Bucket id per subspace: bit j set iff coordinate j of the subvector is < 0.

    z: [..., d] -> uint8/uint16 [..., n_sub].  This is the index of the nearest
    analytic centroid (+-1/sqrt(m))^m, the pinned claim of ParisKV,
    Methodology 1 ("Analytic Centroids").
    """
    d = z.shape[-1]
    m = d // n_sub
    zb = z.reshape(z.shape[:-1] + (n_sub, m))
    ids = np.zeros(zb.shape[:-1], dtype=np.int64)
    for j in range(m):
        ids |= (zb[..., j] < 0).astype(np.int64) << j
    return ids.astype(np.uint8 if m <= 8 else np.uint16)


def table_scores(z: np.ndarray, n_sub: int, table: np.ndarray) -> np.ndarray:
    """float32 [..., n_sub, C]: score of centroid c of subspace b against the
    subvector z_b, ((0 + z_0 c_0) + z_1 c_1) + ... + z_{m-1} c_{m-1}, each
    product and sum rounded to float32 (the learned-centroid baseline;
    table: float32 [n_sub, C, m])."""
    z = np.asarray(z, dtype=F32)
    table = np.asarray(table, dtype=F32)
    m = table.shape[-1]
    zb = z.reshape(z.shape[:-1] + (n_sub, 1, m))
    acc = (zb[..., 0] * table[..., 0]).astype(F32)
    for j in range(1, m):
        acc = (acc + (zb[..., j] * table[..., j]).astype(F32)).astype(F32)
    return acc


def table_ids(z: np.ndarray, n_sub: int, table: np.ndarray) -> np.ndarray:
    """Bucket id per subspace against a table of learned centroids: the
    centroid with the largest table_scores, the lowest id on ties (the
    nearest centroid by inner product, as ParisKV assigns keys)."""
    sc = table_scores(z, n_sub, table)
    return np.argmax(sc, axis=-1).astype(np.uint8 if table.shape[-2] <= 256 else np.uint16)


def kmeans_table(zb_keys: np.ndarray, n_centroids: int, iters: int, seed: int) -> np.ndarray:
    """Learned centroids for the baseline: spherical k-means in float64 on the
    unit subvectors of the prefill keys, per subspace.  zb_keys: [N, n_sub, m]
    rotated key subvectors; start: n_centroids distinct keys drawn with the
    seeded generator; each iteration assigns every key to the centroid of
    largest inner product (lowest index on ties) and replaces each centroid
    by the normalised mean of its keys (an empty centroid keeps its place).
    Returns float32 [n_sub, n_centroids, m] of unit vectors."""
    zb = np.asarray(zb_keys, dtype=np.float64)
    N, n_sub, m = zb.shape
    nrm = np.linalg.norm(zb, axis=-1, keepdims=True)
    u = np.divide(zb, nrm, out=np.zeros_like(zb), where=nrm > 0)
    rng = np.random.default_rng(seed)
    out = np.empty((n_sub, n_centroids, m))
    for b in range(n_sub):
        c = u[rng.choice(N, size=n_centroids, replace=False), b].copy()
        for _ in range(iters):
            a = np.argmax(u[:, b] @ c.T, axis=1)
            sums = np.zeros_like(c)
            np.add.at(sums, a, u[:, b])
            nm = np.linalg.norm(sums, axis=1)
            keep = nm > 0
            c[keep] = sums[keep] / nm[keep, None]
        out[b] = c
    return out.astype(F32)


def centroid(cid: int, m: int) -> np.ndarray:
    """Analytic centroid number cid: coordinate j is -1/sqrt(m) if bit j is set."""
    bits = (cid >> np.arange(m)) & 1
    return np.where(bits == 1, -1.0, 1.0) / math.sqrt(m)


def magnitude_index(ax: np.ndarray, thresholds: np.ndarray) -> np.ndarray:
    """t = #{thresholds strictly below |x|}: the 3 magnitude bits."""
    t = np.zeros(ax.shape, dtype=np.int64)
    for thr in thresholds:
        t += (thr < ax).astype(np.int64)
    return t


def encode_ideal(K: np.ndarray, signs: np.ndarray, n_sub: int, levels=None, thresholds=None):
    """Literal float64 encoding of keys K [N, d] (readings R1-R5).

    k_hat = k/||k||, u = R k_hat, u_b its subvectors, x_b = u_b/||u_b||.
    ids from the sign pattern of u_b; codes: sign bit [x < 0] and magnitude
    index from ``thresholds``; v = dequantised x; w = ||k|| ||u_b|| / <v_b, x_b>.
    With levels=None the quantiser is lossless (v = x), used by the pins.
    Returns a dict with ids, nib (4-bit codes [N, d]), w, x, v, u, knorm.
    """
    K = np.asarray(K, dtype=np.float64)
    N, d = K.shape
    m = d // n_sub
    R = srht_matrix(signs)
    knorm = np.sqrt(np.sum(K * K, axis=1))
    safe = np.where(knorm > 0, knorm, 1.0)
    u = (K / safe[:, None]) @ R.T
    ub = u.reshape(N, n_sub, m)
    un = np.sqrt(np.sum(ub * ub, axis=2))
    x = np.where(un[..., None] > 0, ub / np.where(un > 0, un, 1.0)[..., None], 0.0)
    ids = sign_pattern_ids(u, n_sub)
    s = (x < 0).astype(np.int64)
    if levels is None:
        t = np.zeros_like(s)
        v = x.copy()
    else:
        t = magnitude_index(np.abs(x), thresholds)
        v = np.where(s == 1, -1.0, 1.0) * np.asarray(levels, dtype=np.float64)[t]
    vx = np.sum(v * x, axis=2)
    w = np.where(un > 0, knorm[:, None] * un / np.where(vx != 0, vx, 1.0), 0.0)
    nib = ((s << 3) | t).reshape(N, d).astype(np.uint8)
    return dict(ids=ids, nib=nib, w=w, x=x, v=v, u=u, knorm=knorm)


def encode_contract(K32: np.ndarray, signs: np.ndarray, n_sub: int,
                    lev32: np.ndarray, thr32: np.ndarray, table: np.ndarray = None):
    """float32 encoding of keys K32 [N, d] in the contract order.

    z = fwht(D * k) (exact sign flips, then the FWHT in its stage order);
    per subspace b: n_b = sqrt(sequential sum over j of z_j * z_j);
    x_j = z_j / n_b; s_j = [z_j < 0]; t_j = #{tau < |x_j|};
    v_j = (-1)^s_j * lev[t_j]; vx = sequential sum over j of v_j * x_j;
    w = n_b / (float32(sqrt(d)) * vx), and w = 0, codes 0 where n_b = 0.
    Returns dict ids uint8 [N, n_sub], nib uint8 [N, d], w float32 [N, n_sub].
    table (learned-centroid baseline): ids from table_ids instead of the sign
    patterns; everything else the same.
    """
    K32 = np.asarray(K32, dtype=F32)
    N, d = K32.shape
    m = d // n_sub
    z = fwht(K32 * np.asarray(signs, dtype=F32)[None, :])
    zb = z.reshape(N, n_sub, m)
    ids = sign_pattern_ids(z, n_sub) if table is None else table_ids(z, n_sub, table)
    acc = np.zeros((N, n_sub), dtype=F32)
    for j in range(m):
        acc = acc + zb[..., j] * zb[..., j]
    n = np.sqrt(acc)
    live = n > 0
    x = np.zeros_like(zb)
    np.divide(zb, n[..., None], out=x, where=live[..., None])
    s = (zb < 0) & live[..., None]
    t = magnitude_index(np.abs(x), thr32) * live[..., None]
    lev_t = np.asarray(lev32, dtype=F32)[t]
    v = np.where(s, -lev_t, lev_t).astype(F32)
    vx = np.zeros((N, n_sub), dtype=F32)
    for j in range(m):
        vx = vx + v[..., j] * x[..., j]
    sqrtd = F32(np.sqrt(F32(d)))
    w = np.zeros((N, n_sub), dtype=F32)
    np.divide(n, sqrtd * vx, out=w, where=live)
    nib = ((s.astype(np.uint8) << 3) | t.astype(np.uint8)).reshape(N, d)
    return dict(ids=ids, nib=nib, w=w)


def pack_codes(nib: np.ndarray) -> np.ndarray:
    """[N, d] nibbles -> [N, d/2] bytes; coordinate c in byte c//2, even c low."""
    nib = np.asarray(nib, dtype=np.uint8)
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def dequantise(nib: np.ndarray, levels: np.ndarray) -> np.ndarray:
    """v_j = (-1)^{sign bit} * levels[magnitude bits], in the dtype of levels."""
    nib = np.asarray(nib, dtype=np.int64)
    lv = np.asarray(levels)[nib & 7]
    return np.where(nib >> 3 == 1, -lv, lv).astype(lv.dtype)


# ----------------------------------------------------------------------------
# Query side (ParisKV, Methodology 2: the query's top-rho centroids per
# subspace; the rotated query q_tilde and ||q||_2 of the estimator).
# ----------------------------------------------------------------------------


def query_prep_contract(q32: np.ndarray, signs: np.ndarray, n_sub: int, rho: int,
                        weighting: str = "rank", table: np.ndarray = None):
    """float32 query preparation for one query q32 [d].

    ||q|| = sqrt(sequential sum over j = 0..d-1 of q_j * q_j);
    z = fwht(D * q); ||z|| likewise sequential; q_tilde = z / ||z|| (0 if ||z|| = 0);
    centroid score of id c in subspace b = sequential sum over j of
    (-z_{b,j} if bit j of c else +z_{b,j}); the top rho ids per subspace by
    (score desc, id asc) get weight rho - r (rank r) or 1 (flat).
    Returns dict qnorm, qt [d], hot_ids [n_sub, rho], hot_w [n_sub, rho],
    lut int [n_sub, 2^m] (the vote each bucket gives).  table: the learned
    centroids' table_scores replace the sign-pattern scores.
    """
    q32 = np.asarray(q32, dtype=F32)
    d = q32.shape[0]
    m = d // n_sub
    acc = F32(0)
    for j in range(d):
        acc = F32(acc + q32[j] * q32[j])
    qnorm = F32(np.sqrt(acc))
    z = fwht(q32 * np.asarray(signs, dtype=F32))
    acc = F32(0)
    for j in range(d):
        acc = F32(acc + z[j] * z[j])
    zn = F32(np.sqrt(acc))
    qt = (z / zn).astype(F32) if zn > 0 else np.zeros(d, dtype=F32)
    scores = centroid_scores_contract(z, n_sub) if table is None else table_scores(z, n_sub, table)
    hot_ids = top_rho(scores, rho)
    if weighting == "rank":
        hot_w = np.broadcast_to(rho - np.arange(rho), hot_ids.shape).astype(np.int64)
    elif weighting == "flat":
        hot_w = np.ones(hot_ids.shape, dtype=np.int64)
    else:
        raise ValueError(weighting)
    lut = np.zeros((n_sub, 1 << m), dtype=np.int64)
    for b in range(n_sub):
        lut[b, hot_ids[b]] = hot_w[b]
    return dict(qnorm=qnorm, qt=qt, z=z, hot_ids=hot_ids, hot_w=hot_w, lut=lut, scores=scores)


def centroid_scores_contract(z: np.ndarray, n_sub: int) -> np.ndarray:
    """float32 [n_sub, 2^m]: score of every analytic centroid per subspace,
    as the sequential sum over j of +-z_{b,j} (the common 1/sqrt(m) factor of
    the centroids is dropped; it does not change the order)."""
    z = np.asarray(z, dtype=F32)
    m = z.shape[0] // n_sub
    zb = z.reshape(n_sub, m)
    ids = np.arange(1 << m)
    acc = np.zeros((n_sub, 1 << m), dtype=F32)
    for j in range(m):
        neg = ((ids >> j) & 1).astype(bool)
        term = np.where(neg[None, :], -zb[:, j:j + 1], zb[:, j:j + 1]).astype(F32)
        acc = acc + term
    return acc


def top_rho(scores: np.ndarray, rho: int) -> np.ndarray:
    """Per row, the rho column ids with the largest score, ties to the lower id."""
    out = np.empty((scores.shape[0], rho), dtype=np.int64)
    ids = np.arange(scores.shape[1])
    for b in range(scores.shape[0]):
        order = np.lexsort((ids, -scores[b].astype(np.float64)))
        out[b] = order[:rho]
    return out


def query_prep_ideal(q: np.ndarray, signs: np.ndarray):
    """float64: ||q|| and q_tilde = R q / ||q||."""
    q = np.asarray(q, dtype=np.float64)
    qnorm = math.sqrt(float(np.dot(q, q)))
    if qnorm == 0:
        return qnorm, np.zeros_like(q)
    return qnorm, srht_matrix(signs) @ (q / qnorm)


# ----------------------------------------------------------------------------
# Coarse candidates (ParisKV, Methodology 2, "Coarse candidate generation
# (collision-based)").
# ----------------------------------------------------------------------------


def votes(ids: np.ndarray, lut: np.ndarray) -> np.ndarray:
    """score_i = sum over subspaces b of lut[b, ids[i, b]] (integer)."""
    ids = np.asarray(ids, dtype=np.int64)
    n_sub = ids.shape[1]
    return lut[np.arange(n_sub)[None, :], ids].sum(axis=1)


def candidate_count(n: int, cand_bp: int, k: int) -> int:
    """C = max(ceil(cand_bp * n / 10000), min(k, n)), at most n (reading R7)."""
    c = max((cand_bp * n + 9999) // 10000, min(k, n))
    return min(c, n)


def select_candidates(scores: np.ndarray, c: int) -> np.ndarray:
    """The first c indices by (score desc, index asc), returned ascending."""
    idx = np.arange(len(scores))
    order = np.lexsort((idx, -np.asarray(scores, dtype=np.int64)))
    return np.sort(order[:c])


# ----------------------------------------------------------------------------
# Rerank and top-k (ParisKV, Methodology 2, "Estimation":
# <k, q> ~ ||q||_2 sum_b w_{i,b} <v_{i,b}, q_tilde_b>).
# ----------------------------------------------------------------------------


def rerank_contract(nib: np.ndarray, w: np.ndarray, qnorm, qt: np.ndarray,
                    lev32: np.ndarray, n_sub: int) -> np.ndarray:
    """float32 estimate for each row of nib [C, d] / w [C, n_sub].

    acc = 0; for b: dot = 0; for j: dot = dot + v_{b,j} * qt_{b,j};
    acc = acc + w_b * dot;  est = ||q|| * acc.
    """
    nib = np.asarray(nib)
    C, d = nib.shape
    m = d // n_sub
    v = dequantise(nib, np.asarray(lev32, dtype=F32)).reshape(C, n_sub, m)
    qt = np.asarray(qt, dtype=F32).reshape(n_sub, m)
    w = np.asarray(w, dtype=F32)
    acc = np.zeros(C, dtype=F32)
    for b in range(n_sub):
        dot = np.zeros(C, dtype=F32)
        for j in range(m):
            dot = dot + v[:, b, j] * qt[b, j]
        acc = acc + w[:, b] * dot
    return (F32(qnorm) * acc).astype(F32)


def estimator_ideal(v: np.ndarray, w: np.ndarray, qnorm: float, qt: np.ndarray) -> np.ndarray:
    """float64 ||q|| * sum_b w_b <v_b, qt_b> for v [C, n_sub, m], w [C, n_sub]."""
    C, n_sub, m = v.shape
    return qnorm * np.sum(w * np.einsum("cbj,bj->cb", v, qt.reshape(n_sub, m)), axis=1)


def topk(est: np.ndarray, cand: np.ndarray, k: int):
    """The first min(k, C) candidates by (est desc, index asc), listed in
    that order.  Returns (indices, their estimates)."""
    est = np.asarray(est)
    cand = np.asarray(cand, dtype=np.int64)
    order = np.lexsort((cand, -est.astype(np.float64)))
    keep = order[:min(k, len(cand))]
    return cand[keep], est[keep]


def exact_topk(K: np.ndarray, q: np.ndarray, k: int) -> np.ndarray:
    """float64 brute force: the k largest <k_i, q> by (value desc, index asc), ascending."""
    s = np.asarray(K, dtype=np.float64) @ np.asarray(q, dtype=np.float64)
    idx = np.arange(len(s))
    return np.sort(np.lexsort((idx, -s))[:min(k, len(s))])


def recall(found: np.ndarray, truth: np.ndarray) -> float:
    truth = np.asarray(truth)
    if len(truth) == 0:
        return 1.0
    return len(np.intersect1d(found, truth)) / len(truth)


def retrieve_contract(enc: dict, q32: np.ndarray, signs: np.ndarray, n_sub: int, rho: int,
                      cand_bp: int, k: int, lev32: np.ndarray, weighting: str = "rank",
                      table: np.ndarray = None):
    """The whole retrieval for one query over one encoded Retrieval zone.

    enc: dict(ids [N, n_sub], nib [N, d], w [N, n_sub]) from encode_contract.
    Returns dict(votes, cand, est (per candidate), top_idx, top_est, C, k_eff),
    indices relative to the zone start.
    """
    qp = query_prep_contract(q32, signs, n_sub, rho, weighting, table)
    n = enc["ids"].shape[0]
    sc = votes(enc["ids"], qp["lut"])
    c = candidate_count(n, cand_bp, k)
    cand = select_candidates(sc, c)
    est = rerank_contract(enc["nib"][cand], enc["w"][cand], qp["qnorm"], qp["qt"], lev32, n_sub)
    top_idx, top_est = topk(est, cand, k)
    return dict(votes=sc, cand=cand, est=est, top_idx=top_idx, top_est=top_est,
                C=c, k_eff=min(k, c), qp=qp)


# ----------------------------------------------------------------------------
# Sparse attention (ParisKV: attend to the Sink, Local, Update-Buffer and
# retrieved top-k tokens only; reading R9).
# ----------------------------------------------------------------------------


def attention(q: np.ndarray, Krows: np.ndarray, Vrows: np.ndarray) -> np.ndarray:
    """float64 softmax(K q / sqrt(d)) V over the given rows (each row once)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(Krows, dtype=np.float64)
    V = np.asarray(Vrows, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros(q.shape[0])
    s = K @ q / math.sqrt(q.shape[0])
    p = np.exp(s - s.max())
    return (p / p.sum()) @ V


# ----------------------------------------------------------------------------
# Zones (ParisKV, system level, "Sliding-window update mechanism": Sink,
# Local, Retrieval and Update Buffer; reading R10).
# ----------------------------------------------------------------------------


class Zones:
    """Token-position bookkeeping of one sequence.

    Sink = [0, min(S, T)), Retrieval = [S, S + N), Local = [S + N, S + N + n_local),
    Buffer = [S + N + n_local, T).  Positions only ever grow, so every zone is
    a contiguous range.
    """

    def __init__(self, sink: int, local: int, update_buf: int):
        self.S, self.L, self.U = sink, local, update_buf
        self.T = 0
        self.N = 0
        self.n_local = 0
        self.n_buf = 0

    def prefill(self, T: int):
        if self.T:
            raise RuntimeError("prefill on a non-empty cache")
        self.T = T
        rest = max(0, T - self.S)
        self.n_local = min(self.L, rest)
        self.N = rest - self.n_local
        self.n_buf = 0

    def append(self):
        """Add token T.  Returns the evicted position range (lo, hi), empty if none."""
        p = self.T
        self.T += 1
        if p < self.S:
            return (0, 0)
        self.n_buf += 1
        if self.n_buf < self.U:
            return (0, 0)
        self.n_local += self.n_buf
        self.n_buf = 0
        evict = max(0, self.n_local - self.L)
        lo = self.S + self.N
        self.N += evict
        self.n_local -= evict
        return (lo, lo + evict)

    def sink(self):
        return np.arange(0, min(self.S, self.T))

    def retrieval(self):
        return np.arange(self.S, self.S + self.N)

    def local(self):
        a = self.S + self.N
        return np.arange(a, a + self.n_local)

    def buffer(self):
        a = self.S + self.N + self.n_local
        return np.arange(a, self.T)
