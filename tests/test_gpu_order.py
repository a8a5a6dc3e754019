"""The order of the top-k lists (ParisKV, Methodology 2, "Candidate
reranking (RSQ-IP)": the k best candidates by estimate).  With
topk_order = PARIS_TOPK_BY_SCORE (the default) each list runs best first,
equal estimates by ascending position, bit for bit the oracle's list; with
PARIS_TOPK_BY_POSITION the same set in ascending position.  Covers ties
(duplicated keys give equal estimates), k_eff below k, k_eff not a power of
two, the largest sortable list (16384 entries), a NULL score array and the
limit on topk."""
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


def test_both_orders_list_the_same_set():
    kw = dict(batch=2, n_kv_heads=2, n_q_heads=8, sink=16, local=128, update_buf=32, topk=300, cand_bp=500)
    by_score = g.make_case(20000, seed=81, **kw)
    by_pos = g.make_case(20000, seed=81, topk_order=P.PARIS_TOPK_BY_POSITION, **kw)
    q = g.queries_from_zone(by_score)
    _, i_s, s_s, k_eff = g.run_retrieve(by_score, q)
    _, i_p, s_p, k_eff_p = g.run_retrieve(by_pos, q)
    assert k_eff == k_eff_p == 300
    i_s, s_s, i_p, s_p = i_s.cpu().numpy(), s_s.cpu().numpy(), i_p.cpu().numpy(), s_p.cpu().numpy()
    g.assert_score_order(i_s, s_s, k_eff)
    assert np.all(np.diff(i_p, axis=-1) > 0)
    for seq in range(2):
        for h in range(8):
            perm = np.argsort(i_s[seq, h])
            np.testing.assert_array_equal(i_s[seq, h][perm], i_p[seq, h])
            assert np.array_equal(s_s[seq, h][perm].view(np.uint32), s_p[seq, h].view(np.uint32))
    g.check_retrieve(by_score, q)


def test_equal_estimates_are_listed_by_ascending_position():
    # every key four times: each estimate occurs (at least) four times
    T = 8000
    scale = synth.channel_scale(82, 1, 128)
    base = synth.keys(82, 1, 1, 0, T // 4, 128, scale)
    K = np.repeat(base, 4, axis=2)
    c = g.make_case(T, seed=82, K=K, batch=1, n_kv_heads=1, n_q_heads=4, sink=16, local=64, update_buf=32,
                    topk=257, cand_bp=800)
    qd, idx, k_eff = g.check_retrieve(c, g.queries_from_zone(c))
    idx_h = idx.cpu().numpy()
    ties = 0
    for h in range(4):
        e = c.ctx.paris_debug_dump(P.DUMP_CAND_EST, 0, h)
        ties += int(np.sum(np.diff(np.sort(e)) == 0))
    assert ties > 0
    g.check_attention(c, qd, idx, k_eff)
    assert np.all(idx_h[..., k_eff:] == -1)


def test_short_lists_and_a_null_score_array():
    # N = 40 Retrieval keys, k = 100: k_eff = 40, the rest -1 / -inf
    c = g.make_case(16 + 40 + 64, seed=83, batch=1, n_kv_heads=2, n_q_heads=4, sink=16, local=64, update_buf=16,
                    topk=100, cand_bp=500)
    q = g.queries_from_zone(c)
    qd, idx, k_eff = g.check_retrieve(c, q)
    assert k_eff == 40
    idx2 = torch.full_like(idx, -9)
    assert c.ctx.paris_retrieve(qd, idx2, None) == k_eff
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2)


@pytest.mark.parametrize("k,T", [(5000, 30000), (16384, 20000), (8000, 12000)])
def test_long_lists(k, T):
    # every key a candidate (cand_bp = 10000): k_eff = min(k, N), sorted in one block
    # (12000 tokens: every candidate's key fits the blocks' key tables, more than
    # the counting sort takes)
    c = g.make_case(T, seed=84, batch=1, n_kv_heads=1, n_q_heads=2, sink=16, local=64, update_buf=32, topk=k,
                    cand_bp=10000)
    qd, idx, k_eff = g.check_retrieve(c, g.queries_from_zone(c), stages=False)
    assert k_eff == min(k, c.zones.N)


def test_topk_limit_of_the_score_order():
    with pytest.raises(P.ParisError):
        P.Context(P.make_config(topk=16385, max_ctx=1 << 15), synth.srht_signs(1, 128))
    ctx = P.Context(P.make_config(topk=16385, max_ctx=1 << 15, topk_order=P.PARIS_TOPK_BY_POSITION),
                    synth.srht_signs(1, 128))
    ctx.close()
    with pytest.raises(P.ParisError):
        P.Context(P.make_config(topk_order=2), synth.srht_signs(1, 128))


def test_gqa_union_of_score_ordered_lists():
    c = g.make_case(6000, seed=85, batch=1, n_kv_heads=2, n_q_heads=8, sink=16, local=128, update_buf=32,
                    topk=200, cand_bp=500)
    qd, idx, _, k_eff = g.run_retrieve(c, g.queries_from_zone(c))
    out = torch.zeros((1, 8, 128), dtype=torch.bfloat16, device="cuda")
    c.ctx.paris_sparse_attend_gqa(qd, idx, out)
    c.ctx.paris_check_device()
    out_h, q_seen, idx_h = out.float().cpu().numpy(), qd.float().cpu().numpy(), idx.cpu().numpy()
    z = c.zones
    for h in range(8):
        kvh = h // 4
        grp = idx_h[0, 4 * kvh:4 * kvh + 4, :k_eff]
        rows = np.concatenate([z.sink(), z.local(), z.buffer(), np.unique(grp)]).astype(np.int64)
        ref = o.attention(q_seen[0, h], c.K[0, kvh, rows], g.as_seen(c.V, torch.bfloat16)[0, kvh, rows])
        assert np.max(np.abs(out_h[0, h] - ref)) <= g.ATTN_ATOL


def test_a_zero_query_lists_equal_estimates_by_position():
    # every estimate is 0: one bin holds the whole list, which the sort orders by position
    c = g.make_case(12000, seed=86, batch=1, n_kv_heads=1, n_q_heads=2, sink=16, local=64, update_buf=32, topk=700,
                    cand_bp=1000)
    qd, idx, k_eff = g.check_retrieve(c, np.zeros((1, 2, 128), np.float32))
    idx_h = idx.cpu().numpy()[0, :, :k_eff]
    assert np.all(np.diff(idx_h, axis=-1) > 0)
