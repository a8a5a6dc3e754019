"""The dense full-attention comparator (paris_dense_attend) against the oracle:
softmax attention of every query head over every cached token, Sink,
Retrieval zone, Local and Update Buffer (ParisKV, Experiments, "Efficiency":
the full-attention baseline), within 2e-2 of float64.  Covers GQA groups of
1, 2, 3 and 4 query heads per KV head, batches, ragged lengths, a wrapped
Local/Buffer ring, the Retrieval zone in pinned host memory, an empty cache,
a cache still inside the Sink, and the 131072-token Llama-shaped layer."""
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


def dense(c: g.Case, q: np.ndarray) -> np.ndarray:
    b, hq, d = c.cfg["batch"], c.cfg["n_q_heads"], c.cfg["head_dim"]
    out = torch.full((b, hq, d), 3.0, dtype=torch.bfloat16, device="cuda")
    c.ctx.paris_dense_attend(g.to_dev(q, c.dtype), out)
    c.ctx.paris_check_device()
    return out.float().cpu().numpy()


def check_dense(c: g.Case, q: np.ndarray, heads=None):
    out = dense(c, q)
    q_seen = g.as_seen(q, c.dtype)
    Kb, Vb = g.as_seen(c.K, torch.bfloat16), g.as_seen(c.V, torch.bfloat16)
    T = c.zones.T
    heads = heads or [(s, h) for s in range(c.cfg["batch"]) for h in range(c.cfg["n_q_heads"])]
    worst = 0.0
    for seq, qh in heads:
        ref = o.attention(q_seen[seq, qh], Kb[seq, qh // c.G, :T], Vb[seq, qh // c.G, :T])
        err = float(np.max(np.abs(out[seq, qh] - ref)))
        worst = max(worst, err)
        assert err <= g.ATTN_ATOL, (seq, qh, err)
    return worst


@pytest.mark.parametrize("hkv,hq", [(2, 2), (2, 4), (2, 6), (2, 8)])
def test_dense_matches_the_oracle_for_every_gqa_group(hkv, hq):
    c = g.make_case(5000, seed=51, batch=2, n_kv_heads=hkv, n_q_heads=hq, sink=16, local=256, update_buf=64,
                    topk=128, cand_bp=500)
    check_dense(c, g.queries_from_zone(c))


def test_dense_after_appends_wraps_the_window_ring_and_reads_host_memory():
    c = g.make_case(3000, seed=52, batch=1, n_kv_heads=2, n_q_heads=8, sink=16, local=128, update_buf=32,
                    topk=64, cand_bp=1000, retrieval_on_host=1)
    for step in range(150):  # several flushes: the ring wraps, the Retrieval zone grows
        kn = synth.decode_keys(c.seed, 1, 2, step, 128, c.scale)
        vn = synth.decode_values(c.seed, 1, 2, step, 128)
        g.append(c, kn, vn)
    g.check_state(c)
    check_dense(c, g.queries_from_zone(c, step=3))


def test_dense_on_an_empty_cache_and_inside_the_sink():
    c = g.make_case(0, seed=53, batch=1, n_kv_heads=1, n_q_heads=4, sink=16, local=32, update_buf=16, topk=8)
    q = np.random.default_rng(0).standard_normal((1, 4, 128)).astype(np.float32)
    assert np.all(dense(c, q) == 0.0)
    for step in range(5):
        g.append(c, synth.decode_keys(c.seed, 1, 1, step, 128, c.scale), synth.decode_values(c.seed, 1, 1, step, 128))
    assert c.zones.T == 5 and c.zones.N == 0
    check_dense(c, q)


def test_dense_equals_sparse_attention_when_everything_is_retrieved():
    # k >= N and every key a candidate: the sparse set is every token
    c = g.make_case(2048, seed=54, batch=1, n_kv_heads=1, n_q_heads=2, sink=16, local=64, update_buf=32,
                    topk=4096, cand_bp=10000)
    q = g.queries_from_zone(c)
    qd, idx, _, k_eff = g.run_retrieve(c, q)
    assert k_eff == c.zones.N
    sparse = torch.zeros((1, 2, 128), dtype=torch.bfloat16, device="cuda")
    c.ctx.paris_sparse_attend(qd, idx, sparse)
    d = dense(c, q)
    assert np.max(np.abs(d - sparse.float().cpu().numpy())) <= 2 * g.ATTN_ATOL
    check_dense(c, q)


def test_dense_at_full_size_on_sampled_heads():
    T0 = 131072
    c = g.make_case(T0, seed=55, max_ctx=T0 + 64, batch=1, n_kv_heads=8, n_q_heads=32, sink=16, local=512,
                    update_buf=128, topk=1024, cand_bp=500)
    check_dense(c, g.queries_from_zone(c), heads=[(0, 0), (0, 9), (0, 31)])
