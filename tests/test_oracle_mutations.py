"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check
that at least one pin catches each of them."""
import importlib.util
import inspect
import sys
import types

import pytest

from oracle import pariskv
from tests import oracle_pins as P

MUTATIONS = [
    ("fwht butterfly sign", "v[..., 1, :] = a - b", "v[..., 1, :] = b - a", P.pin_fwht_golden),
    ("fwht stage skipped", "h *= 2\n    return y", "h *= 4\n    return y", P.pin_fwht_matches_library_hadamard),
    ("srht scale", "/ math.sqrt(d)\n", "/ d\n", P.pin_srht_orthogonal),
    ("zero counted negative", "ids |= (zb[..., j] < 0)", "ids |= (zb[..., j] <= 0)", P.pin_ids_are_nearest_centroids),
    ("centroid bit order", "ids |= (zb[..., j] < 0).astype(np.int64) << j",
     "ids |= (zb[..., j] < 0).astype(np.int64) << (m - 1 - j)", P.pin_ids_are_nearest_centroids),
    ("beta prior shape", "return betainc(0.5, (m - 1) / 2.0, t * t)", "return betainc(0.5, m / 2.0, t * t)",
     P.pin_levels_quadrature),
    ("lloyd thresholds not midpoints", "edges = np.concatenate([[0.0], 0.5 * (lev[1:] + lev[:-1]), [1.0]])",
     "edges = np.concatenate([[0.0], lev[1:], [1.0]])", P.pin_levels_closed_forms),
    ("partial-mean constant", "c = beta_fn(1.0, b) / beta_fn(0.5, b)", "c = beta_fn(0.5, b) / beta_fn(1.0, b)",
     P.pin_levels_monte_carlo),
    ("w drops ||k||", "w = np.where(un > 0, knorm[:, None] * un", "w = np.where(un > 0, un", P.pin_estimator_exact_when_lossless),
    ("w not divided by <v,x>", "knorm[:, None] * un / np.where(vx != 0, vx, 1.0)", "knorm[:, None] * un",
     P.pin_estimator_level_scale_invariant),
    ("q~ transposed rotation", "return qnorm, srht_matrix(signs) @ (q / qnorm)",
     "return qnorm, srht_matrix(signs).T @ (q / qnorm)", P.pin_estimator_exact_when_lossless),
    ("contract w missing sqrt(d)", "np.divide(n, sqrtd * vx, out=w, where=live)", "np.divide(n, vx, out=w, where=live)",
     P.pin_contract_tracks_ideal),
    ("contract <v,x> uses z", "vx = vx + v[..., j] * x[..., j]", "vx = vx + v[..., j] * zb[..., j]", P.pin_contract_tracks_ideal),
    ("rerank drops w", "acc = acc + w[:, b] * dot", "acc = acc + dot", P.pin_contract_tracks_ideal),
    ("rerank wrong coordinate", "dot = dot + v[:, b, j] * qt[b, j]", "dot = dot + v[:, b, j] * qt[b, m - 1 - j]",
     P.pin_contract_tracks_ideal),
    ("q~ not normalised", "qt = (z / zn).astype(F32) if zn > 0", "qt = z.astype(F32) if zn > 0", P.pin_contract_tracks_ideal),
    ("dequantise sign", "return np.where(nib >> 3 == 1, -lv, lv)", "return np.where(nib >> 3 == 1, lv, -lv)",
     P.pin_codes_nearest_level),
    ("magnitude index off by one", "t += (thr < ax).astype(np.int64)", "t += (thr <= ax).astype(np.int64) + 0 * t",
     None),
    ("code nibble order", "return (nib[:, 0::2] | (nib[:, 1::2] << 4))", "return (nib[:, 1::2] | (nib[:, 0::2] << 4))",
     P.pin_codes_nearest_level),
    ("centroid score sign", "term = np.where(neg[None, :], -zb[:, j:j + 1], zb[:, j:j + 1])",
     "term = np.where(neg[None, :], zb[:, j:j + 1], -zb[:, j:j + 1])", P.pin_top_rho_closed_form),
    ("top-rho ties to higher id", "order = np.lexsort((ids, -scores[b]", "order = np.lexsort((-ids, -scores[b]",
     P.pin_top_rho_closed_form),
    ("vote weights reversed", "hot_w = np.broadcast_to(rho - np.arange(rho)", "hot_w = np.broadcast_to(1 + np.arange(rho)",
     P.pin_votes),
    ("candidate count floor", "c = max((cand_bp * n + 9999) // 10000", "c = max((cand_bp * n) // 10000", P.pin_candidate_counts),
    ("candidates ascending score", "order = np.lexsort((idx, -np.asarray(scores, dtype=np.int64)))",
     "order = np.lexsort((idx, np.asarray(scores, dtype=np.int64)))", P.pin_selection),
    ("top-k ties to higher index", "order = np.lexsort((cand, -est.astype(np.float64)))",
     "order = np.lexsort((-cand, -est.astype(np.float64)))", P.pin_selection),
    ("top-k listed by position", "keep = order[:min(k, len(cand))]", "keep = np.sort(order[:min(k, len(cand))])",
     P.pin_selection),
    ("top-k over positions that are not the candidates", "top_idx, top_est = topk(est, cand, k)",
     "top_idx, top_est = topk(est, np.arange(c), k)", P.pin_pipeline_tiny_full_sort),
    ("k_eff not capped by C", "C=c, k_eff=min(k, c)", "C=c, k_eff=k", P.pin_pipeline_tiny_full_sort),
    ("rerank of the wrong rows", 'est = rerank_contract(enc["nib"][cand], enc["w"][cand]',
     'est = rerank_contract(enc["nib"][:c], enc["w"][:c]', P.pin_pipeline_tiny_full_sort),
    ("pipeline candidate count ignores k", "c = candidate_count(n, cand_bp, k)",
     "c = candidate_count(n, cand_bp, 0)", P.pin_pipeline_tiny_full_sort),
    ("recall over found", "return len(np.intersect1d(found, truth)) / len(truth)",
     "return len(np.intersect1d(found, truth)) / max(1, len(found))", P.pin_recall_hand_made_sets),
    ("recall counts duplicates", "return len(np.intersect1d(found, truth)) / len(truth)",
     "return int(np.isin(found, truth).sum()) / len(truth)", P.pin_recall_hand_made_sets),
    ("attention unscaled","s = K @ q / math.sqrt(q.shape[0])", "s = K @ q", P.pin_attention_dense),
    ("zone eviction off by one", "evict = max(0, self.n_local - self.L)", "evict = max(0, self.n_local - self.L - 1)",
     P.pin_zones),
    ("sink overwritten", "if p < self.S:\n            return (0, 0)", "if p < 0:\n            return (0, 0)", P.pin_zones),
]


def _mutant(old, new):
    src = inspect.getsource(pariskv)
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    src = src.replace(old, new, 1)
    mod = types.ModuleType("oracle_mutant")
    mod.__dict__["__name__"] = "oracle_mutant"
    exec(compile(src, "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new,pin", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(name, old, new, pin):
    mod = _mutant(old, new)
    pins = [pin] if pin is not None else P.ALL_PINS
    caught = False
    for p in pins:
        try:
            p(mod)
        except Exception:
            caught = True
            break
    assert caught, f"no pin caught the planted mistake: {name}"
