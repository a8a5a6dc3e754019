"""The learned-centroid baseline (paris_set_centroids) against the oracle:
bucket ids from a table of learned centroids, the query's hot centroids by
the same table, then the unchanged votes, candidates and RSQ-IP rerank, all
bit for bit (ParisKV, "Problem definition": codebooks learned on the prefill
keys, which the analytic centroids are compared with under drift).  The
last test runs the comparison itself: recall@k of the analytic and the
k-means centroids as decode keys drift away from the prefill keys."""
import numpy as np
import pytest
import torch

from long_context_kv_gb300 import paris as P
from long_context_kv_gb300 import synth
from oracle import pariskv as o
from tests import gpu_cases as g

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_kv_gb300 import build
    build.build()
    P.load()


def kmeans_for(seed, b, hkv, T, S, dtype=torch.bfloat16, iters=8):
    """Per KV head, spherical k-means (oracle) on the rotated Retrieval-zone keys of sequence 0."""
    scale = synth.channel_scale(seed, hkv, 128)
    K = g.as_seen(synth.keys(seed, b, hkv, 0, T, 128, scale), dtype)
    signs = synth.srht_signs(seed, 128)
    tabs = []
    for h in range(hkv):
        z = o.fwht(K[0, h, S:] * signs.astype(np.float32)[None, :])
        tabs.append(o.kmeans_table(z.reshape(-1, 16, 8), 256, iters=iters, seed=seed + h))
    return np.stack(tabs)


def test_random_table_encodes_and_retrieves_like_the_oracle():
    rng = np.random.default_rng(71)
    tab = rng.standard_normal((2, 16, 256, 8)).astype(np.float32)
    tab /= np.linalg.norm(tab, axis=-1, keepdims=True)
    c = g.make_case(20000, seed=71, table=tab, batch=2, n_kv_heads=2, n_q_heads=8, sink=16, local=128,
                    update_buf=32, topk=128, cand_bp=500)
    g.check_encoding(c)
    g.check_retrieve(c, g.queries_from_zone(c))


def test_kmeans_table_after_appends_and_flushes():
    T, S = 12000, 16
    tab = kmeans_for(72, 1, 2, T, S)
    c = g.make_case(T, seed=72, table=tab, batch=1, n_kv_heads=2, n_q_heads=4, sink=S, local=128, update_buf=32,
                    topk=96, cand_bp=500)
    for step in range(70):  # two flushes: the flushed keys are encoded against the same table
        g.append(c, synth.drift_keys(c.seed, 1, 2, step, 128, c.scale, rate=0.5), synth.decode_values(c.seed, 1, 2, step, 128))
    g.check_encoding(c)
    qd, idx, k_eff = g.check_retrieve(c, g.queries_from_zone(c, step=2))
    g.check_attention(c, qd, idx, k_eff)


def test_restoring_the_analytic_centroids():
    cfg = dict(batch=1, n_kv_heads=1, n_q_heads=1, head_dim=128, n_sub=16, rho=4, sink=0, local=0, update_buf=32,
               topk=16, cand_bp=1000, max_ctx=4096, retrieval_on_host=0, vote_weighting=P.PARIS_VOTE_RANK)
    c = g.Case(cfg=cfg, seed=73, T=3000)
    c.signs = synth.srht_signs(73, 128)
    c.scale = synth.channel_scale(73, 1, 128)
    c.ctx = P.Context(P.make_config(**cfg), c.signs)
    tab = np.ones((1, 16, 256, 8), dtype=np.float32)
    c.ctx.paris_set_centroids(torch.from_numpy(tab).cuda())
    c.ctx.paris_set_centroids(None)  # back to the sign patterns before any token
    K = synth.keys(73, 1, 1, 0, 3000, 128, c.scale)
    V = synth.values(73, 1, 1, 0, 3000, 128)
    c.ctx.paris_encode_prefill(g.to_dev(K, torch.bfloat16), g.to_dev(V, torch.bfloat16), 3000)
    torch.cuda.synchronize()
    c.K, c.V = g.as_seen(K, torch.bfloat16), g.as_seen(V, torch.bfloat16)
    c.zones = o.Zones(0, 0, 32)
    c.zones.prefill(3000)
    g.check_encoding(c)
    with pytest.raises(P.ParisError):
        c.ctx.paris_set_centroids(torch.from_numpy(tab).cuda())  # not once the cache holds tokens


def test_recall_under_drift_analytic_versus_learned_centroids():
    # the pages' claim: centroids learned on the prefill keys lose recall as
    # decode keys drift; the analytic sign patterns do not depend on the data
    T, S, L, U, hkv, hq, k = 16384, 16, 256, 64, 2, 8, 256
    steps, rate = 1536, 1.0  # drift of 1.0 sigma per 256 decode steps (6 sigma at the end)
    cases = {
        "analytic": g.make_case(T, seed=74, max_ctx=T + steps + 8, batch=1, n_kv_heads=hkv, n_q_heads=hq, sink=S,
                                local=L, update_buf=U, topk=k, cand_bp=500),
        "learned": g.make_case(T, seed=74, max_ctx=T + steps + 8, table=kmeans_for(74, 1, hkv, T, S), batch=1,
                               n_kv_heads=hkv, n_q_heads=hq, sink=S, local=L, update_buf=U, topk=k, cand_bp=500),
    }
    recall = {name: {} for name in cases}
    for step in range(steps):
        kn = synth.drift_keys(74, 1, hkv, step, 128, cases["analytic"].scale, rate=rate)
        vn = synth.decode_values(74, 1, hkv, step, 128)
        for c in cases.values():
            g.append(c, kn, vn)
        if step % 512 != 511:
            continue
        # queries near the most recently flushed (drifted) keys
        z = cases["analytic"].zones
        lo = max(S, S + z.N - 512)
        pos = synth.query_positions(74, 1, hq, lo, S + z.N, step)
        for name, c in cases.items():
            picked = np.stack([c.K[0, h // (hq // hkv), pos[0, h]] for h in range(hq)])[None]
            q = synth.queries_from_keys(74, picked, 0.5, step)
            qd, idx, k_eff = g.check_retrieve(c, q, stages=False)
            idx_h = idx.cpu().numpy()
            rs = []
            for h in range(hq):
                truth = o.exact_topk(c.K[0, h // (hq // hkv), S:S + c.zones.N], g.as_seen(q, torch.bfloat16)[0, h], k_eff)
                rs.append(o.recall(idx_h[0, h, :k_eff] - S, truth))
            recall[name][step + 1] = float(np.mean(rs))
    print("recall@k vs decode step, drift 1 sigma / 256 steps:", recall)
    assert set(recall["analytic"]) == set(recall["learned"])
