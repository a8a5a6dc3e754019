"""GQA-shared sparse attention (paris_sparse_attend_gqa) against the oracle:
every query head of a KV head attends over Sink, Local, the Update Buffer
and the union of the retrieved tokens of all the KV head's query heads
(each row read once per KV head), within 2e-2 of float64.  With one query
head per KV head it attends over the same rows as paris_sparse_attend."""
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


def gqa(c: g.Case, qd: torch.Tensor, idx: torch.Tensor) -> np.ndarray:
    b, hq, d = c.cfg["batch"], c.cfg["n_q_heads"], c.cfg["head_dim"]
    out = torch.full((b, hq, d), 3.0, dtype=torch.bfloat16, device="cuda")
    c.ctx.paris_sparse_attend_gqa(qd, idx, out)
    c.ctx.paris_check_device()
    return out.float().cpu().numpy()


def check_gqa(c: g.Case, qd: torch.Tensor, idx: torch.Tensor, k_eff: int, heads=None):
    out = gqa(c, qd, idx)
    q_seen = qd.float().cpu().numpy()
    idx_h = idx.cpu().numpy()
    Kb, Vb = g.as_seen(c.K, torch.bfloat16), g.as_seen(c.V, torch.bfloat16)
    z = c.zones
    heads = heads or [(s, h) for s in range(c.cfg["batch"]) for h in range(c.cfg["n_q_heads"])]
    sizes = {}
    for seq, qh in heads:
        kvh = qh // c.G
        group = idx_h[seq, kvh * c.G:(kvh + 1) * c.G, :k_eff]
        union = np.unique(group[group >= 0])
        sizes[(seq, kvh)] = len(union)
        rows = np.concatenate([z.sink(), z.local(), z.buffer(), union]).astype(np.int64)
        assert len(np.unique(rows)) == len(rows)
        ref = o.attention(q_seen[seq, qh], Kb[seq, kvh, rows], Vb[seq, kvh, rows])
        err = float(np.max(np.abs(out[seq, qh] - ref)))
        assert err <= g.ATTN_ATOL, (seq, qh, err)
    return out, sizes


@pytest.mark.parametrize("hkv,hq", [(2, 4), (2, 8), (1, 3)])
def test_gqa_attends_over_the_union_of_the_group(hkv, hq):
    c = g.make_case(6000, seed=61, batch=2, n_kv_heads=hkv, n_q_heads=hq, sink=16, local=256, update_buf=64,
                    topk=256, cand_bp=500)
    qd, idx, _, k_eff = g.run_retrieve(c, g.queries_from_zone(c))
    _, sizes = check_gqa(c, qd, idx, k_eff)
    assert all(k_eff <= n <= c.G * k_eff for n in sizes.values())


def test_one_query_head_per_kv_head_equals_sparse_attention():
    c = g.make_case(5000, seed=62, batch=1, n_kv_heads=2, n_q_heads=2, sink=16, local=128, update_buf=32,
                    topk=200, cand_bp=1000)
    qd, idx, _, k_eff = g.run_retrieve(c, g.queries_from_zone(c))
    out, _ = check_gqa(c, qd, idx, k_eff)
    sparse = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda")
    c.ctx.paris_sparse_attend(qd, idx, sparse)
    assert np.max(np.abs(out - sparse.float().cpu().numpy())) <= 2 * g.ATTN_ATOL


def test_shared_rows_after_appends_and_from_host_memory():
    c = g.make_case(3000, seed=63, batch=1, n_kv_heads=2, n_q_heads=8, sink=16, local=128, update_buf=32,
                    topk=128, cand_bp=1000, retrieval_on_host=1)
    for step in range(100):
        g.append(c, synth.decode_keys(c.seed, 1, 2, step, 128, c.scale), synth.decode_values(c.seed, 1, 2, step, 128))
    qd, idx, _, k_eff = g.run_retrieve(c, g.queries_from_zone(c, step=5))
    check_gqa(c, qd, idx, k_eff)


def test_overlapping_heads_share_their_rows():
    # every query head of a group copies the same key (different noise): their top-k sets overlap
    c = g.make_case(8000, seed=64, batch=1, n_kv_heads=2, n_q_heads=8, sink=16, local=128, update_buf=32,
                    topk=256, cand_bp=500)
    q = g.queries_from_zone(c)
    for kvh in range(2):
        q[0, 4 * kvh + 1:4 * kvh + 4] = q[0, 4 * kvh] + 0.05 * np.random.default_rng(kvh).standard_normal((3, 128))
    qd, idx, _, k_eff = g.run_retrieve(c, q)
    _, sizes = check_gqa(c, qd, idx, k_eff)
    assert all(n < 2 * k_eff for n in sizes.values()), sizes


def test_gqa_at_full_size_on_sampled_heads():
    T0 = 131072
    c = g.make_case(T0, seed=65, max_ctx=T0 + 64, batch=1, n_kv_heads=8, n_q_heads=32, sink=16, local=512,
                    update_buf=128, topk=1024, cand_bp=500)
    qd, idx, _, k_eff = g.run_retrieve(c, g.queries_from_zone(c))
    check_gqa(c, qd, idx, k_eff, heads=[(0, 0), (0, 13), (0, 31)])


@pytest.mark.parametrize("hq", [4, 16])
def test_lists_crowded_into_a_few_slices(hq):
    """Caller-made lists whose G heads cover one contiguous run of positions
    (each head its own 1024, in shuffled order): the union piles up in the
    first slices of the Retrieval zone, so those blocks hold more union rows
    than they keep in shared memory (the rest go through the context's union
    list) and stream many tiles while the others have none; with G = 16
    every row of the kernel's head tiles is a real query head."""
    S, L, U, N = 16, 64, 32, 100000
    c = g.make_case(S + N + L, seed=66, batch=1, n_kv_heads=1, n_q_heads=hq, sink=S, local=L, update_buf=U,
                    topk=1024, cand_bp=10000)
    assert c.zones.N == N
    rng = np.random.default_rng(hq)
    lists = (S + np.arange(hq * 1024)).reshape(hq, 1024)
    lists = np.stack([rng.permutation(r) for r in lists]).astype(np.int32)
    idx = torch.from_numpy(lists[None]).cuda()
    qd = g.to_dev(g.queries_from_zone(c), torch.bfloat16)
    _, sizes = check_gqa(c, qd, idx, 1024)
    assert sizes[(0, 0)] == hq * 1024


def test_gqa_and_dense_right_after_decode_steps_see_the_step_token():
    """paris_sparse_attend_gqa and paris_dense_attend enqueued on the same
    stream directly behind paris_decode_step (no host synchronisation) read
    the window as the step left it, its own token included (through a flush
    every 16 steps), and match the oracle over the window plus the union of
    the group's top-k sets, and over every cached token."""
    c = g.make_case(16 + 12000 + 64, seed=67, batch=1, n_kv_heads=2, n_q_heads=8, sink=16, local=64,
                    update_buf=16, topk=128, cand_bp=500)
    b, hq, d, k = 1, 8, 128, 128
    for t in range(36):
        kn = synth.decode_keys(67, b, 2, t, d, c.scale)
        vn = synth.decode_values(67, b, 2, t, d)
        q = g.queries_from_zone(c, step=t)
        qd = g.to_dev(q, torch.bfloat16)
        idx = torch.empty((b, hq, k), dtype=torch.int32, device="cuda")
        sc = torch.empty((b, hq, k), dtype=torch.float32, device="cuda")
        o_step = torch.empty((b, hq, d), dtype=torch.bfloat16, device="cuda")
        o_gqa = torch.full((b, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        o_dense = torch.full((b, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        k_eff = c.ctx.paris_decode_step(g.to_dev(kn, torch.bfloat16), g.to_dev(vn, torch.bfloat16), qd, idx, sc,
                                        o_step)
        c.ctx.paris_sparse_attend_gqa(qd, idx, o_gqa)
        c.ctx.paris_dense_attend(qd, o_dense)
        torch.cuda.synchronize()
        c.ctx.paris_check_device()
        g.append(c, kn, vn, device=False)
        if t % 6 == 5:
            q_seen = qd.float().cpu().numpy()
            idx_h = idx.cpu().numpy()
            got_g, got_d = o_gqa.float().cpu().numpy(), o_dense.float().cpu().numpy()
            Kb, Vb = g.as_seen(c.K, torch.bfloat16), g.as_seen(c.V, torch.bfloat16)
            z = c.zones
            for qh in range(hq):
                kvh = qh // c.G
                group = idx_h[0, kvh * c.G:(kvh + 1) * c.G, :k_eff]
                rows = np.concatenate([z.sink(), z.local(), z.buffer(), np.unique(group[group >= 0])])
                rows = rows.astype(np.int64)
                ref = o.attention(q_seen[0, qh], Kb[0, kvh, rows], Vb[0, kvh, rows])
                assert np.max(np.abs(got_g[0, qh] - ref)) <= g.ATTN_ATOL, (t, qh)
                ref = o.attention(q_seen[0, qh], Kb[0, kvh, :z.T], Vb[0, kvh, :z.T])
                assert np.max(np.abs(got_d[0, qh] - ref)) <= g.ATTN_ATOL, (t, qh)
    assert c.ctx.paris_get_state()["n_flushes"] >= 2
