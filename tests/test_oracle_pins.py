"""The oracle against its pins (closed forms, hand-worked fixtures, library
routines, brute force, Monte-Carlo).  CPU only."""
import numpy as np
import pytest

from oracle import pariskv as o
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(o)


# ---- learned-centroid baseline (ParisKV, "Problem definition": learned
# codebooks fitted on the prefill keys, compared with the analytic centroids)

def _sign_table(n_sub=16, m=8):
    return np.tile(np.stack([o.centroid(c, m) for c in range(1 << m)]).astype(np.float32)[None], (n_sub, 1, 1))


def test_table_ids_with_the_sign_pattern_table_are_the_sign_pattern_ids():
    # the nearest of the 2^m analytic centroids by inner product is the sign pattern
    z = np.random.default_rng(3).standard_normal((500, 128)).astype(np.float32)
    np.testing.assert_array_equal(o.table_ids(z, 16, _sign_table()), o.sign_pattern_ids(z, 16))


def test_table_ids_break_ties_to_the_lowest_id():
    tab = np.random.default_rng(4).standard_normal((16, 256, 8)).astype(np.float32)
    tab[:, 200] = tab[:, 7]  # centroid 200 duplicates centroid 7
    z = np.repeat(tab[:, 7].reshape(1, 128), 3, axis=0)  # each subvector equals centroid 7 of its subspace
    ids = o.table_ids(z, 16, tab)
    assert np.all(ids != 200)
    sc = o.table_scores(z, 16, tab)
    assert np.all(sc[:, np.arange(16), ids] == sc.max(axis=-1))


def test_query_prep_with_the_sign_pattern_table_picks_the_analytic_hot_centroids():
    q = np.random.default_rng(5).standard_normal(128).astype(np.float32)
    signs = np.where(np.random.default_rng(6).random(128) < 0.5, -1, 1).astype(np.int8)
    a = o.query_prep_contract(q, signs, 16, 4)
    b = o.query_prep_contract(q, signs, 16, 4, table=_sign_table())
    np.testing.assert_array_equal(a["hot_ids"], b["hot_ids"])


def test_kmeans_ends_at_a_fixed_point_and_improves_on_its_start():
    # Lloyd's algorithm on the sphere: at convergence every centroid is the
    # normalised mean of the points nearest to it, and the mean best inner
    # product never falls below that of the starting centroids
    rng = np.random.default_rng(7)
    centres = rng.standard_normal((2, 16, 3))
    centres /= np.linalg.norm(centres, axis=-1, keepdims=True)
    a = rng.integers(0, 16, size=4000)
    pts = np.stack([centres[b, a] + 0.05 * rng.standard_normal((4000, 3)) for b in range(2)], axis=1)
    tab = o.kmeans_table(pts, 16, iters=100, seed=1).astype(np.float64)
    np.testing.assert_allclose(np.linalg.norm(tab, axis=-1), 1.0, rtol=1e-6)
    u = pts / np.linalg.norm(pts, axis=-1, keepdims=True)
    start_rng = np.random.default_rng(1)
    for b in range(2):
        start = u[start_rng.choice(4000, size=16, replace=False), b]
        assign = np.argmax(u[:, b] @ tab[b].T, axis=1)
        for k in np.unique(assign):
            mu = u[assign == k, b].mean(axis=0)
            np.testing.assert_allclose(tab[b, k], mu / np.linalg.norm(mu), atol=1e-6)
        assert (u[:, b] @ tab[b].T).max(axis=1).mean() >= (u[:, b] @ start.T).max(axis=1).mean()
