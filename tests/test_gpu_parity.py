"""GPU parity: the CUDA path through the C ABI against the CPU oracle, stage
by stage (bucket ids, codes, w bit for bit; q~, ||q||, hot centroids, votes,
candidates, estimates and top-k bit for bit; estimates also within 1e-4
relative; attention within 2e-2 absolute of float64)."""
import numpy as np
import pytest
import torch

from long_context_kv_gb300 import paris as P
from long_context_kv_gb300 import synth
from tests import gpu_cases as g

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_kv_gb300 import build
    build.build()
    P.load()


def test_tiny_workload_32_queries():
    """1 KV head, d = 128, N = 4096 float32 keys (channel scale LogNormal(0, 0.5)),
    B = 16, rho = 4, 10% candidates, k = 64, 32 queries = key + N(0, 0.5^2)."""
    c = g.make_case(4096, seed=11, dtype=torch.float32, topk=64, cand_bp=1000, rho=4)
    g.check_encoding(c)
    for step in range(32):
        q = g.queries_from_zone(c, step=step)
        qd, idx, k_eff = g.check_retrieve(c, q)
        assert k_eff == 64
        g.check_attention(c, qd, idx, k_eff)


def test_multichunk_gqa_ragged_bf16():
    """3 index chunks with a ragged tail, GQA 4:1, sink and local zones."""
    c = g.make_case(16 + 40000 + 64, seed=12, n_kv_heads=2, n_q_heads=8, sink=16, local=64, update_buf=32,
                    topk=256, cand_bp=500, rho=4)
    assert c.zones.N == 40000
    g.check_encoding(c)
    for step in range(3):
        q = g.queries_from_zone(c, step=step)
        qd, idx, k_eff = g.check_retrieve(c, q)
        g.check_attention(c, qd, idx, k_eff)


def test_batch_sequences_are_independent():
    c = g.make_case(16 + 5000 + 32, seed=13, batch=3, n_kv_heads=2, n_q_heads=4, sink=16, local=32,
                    update_buf=8, topk=100, cand_bp=300, rho=3)
    g.check_encoding(c)
    q = g.queries_from_zone(c)
    qd, idx, k_eff = g.check_retrieve(c, q)
    g.check_attention(c, qd, idx, k_eff)


def test_appends_and_flushes_match_zone_model():
    """Decode appends with drifting keys; every flush moves Local's oldest
    tokens into the Retrieval zone and re-indexes the touched chunk."""
    c = g.make_case(16 + 16300 + 64, seed=14, batch=2, n_kv_heads=2, n_q_heads=4, sink=16, local=64,
                    update_buf=32, topk=128, cand_bp=500, rho=4)
    for t in range(200):
        k = synth.drift_keys(c.seed, 2, 2, t, 128, c.scale, rate=0.5)
        v = synth.decode_values(c.seed, 2, 2, t, 128)
        g.append(c, k, v)
        g.check_state(c)
        if t % 50 == 49:
            q = g.queries_from_zone(c, step=t)
            qd, idx, k_eff = g.check_retrieve(c, q)
            g.check_attention(c, qd, idx, k_eff)
    assert c.zones.N > 16300 + 64  # crossed into the second chunk
    g.check_encoding(c)
    # the K/V the attention reads, by position, are the appended values
    for seq in range(2):
        for h in range(2):
            kv = c.ctx.paris_debug_dump(P.DUMP_KV, seq, h)
            want_k = g.as_seen(c.K[seq, h], torch.bfloat16)
            got_k = torch.from_numpy(kv[0].astype(np.int32) << 16).view(torch.float32).numpy()
            np.testing.assert_array_equal(got_k, want_k)


def test_prefill_then_appends_encode_like_a_fresh_prefill():
    """ids/codes/w of tokens that entered by append equal those of the same
    tokens given at prefill."""
    T0, steps = 16 + 3000 + 32, 70
    a = g.make_case(T0, seed=15, sink=16, local=32, update_buf=16, topk=64)
    for t in range(steps):
        k = synth.decode_keys(a.seed, 1, 1, t, 128, a.scale)
        v = synth.decode_values(a.seed, 1, 1, t, 128)
        g.append(a, k, v)
    b = g.make_case(T0 + steps, seed=15, K=a.K.copy(), sink=16, local=32, update_buf=16, topk=64)
    n = a.zones.N
    for what in (P.DUMP_IDS, P.DUMP_CODES, P.DUMP_W):
        x = a.ctx.paris_debug_dump(what)
        y = b.ctx.paris_debug_dump(what)
        np.testing.assert_array_equal(x[:n], y[:n])


@pytest.mark.parametrize("T", [0, 5, 16, 16 + 64, 16 + 65])
def test_empty_and_tiny_retrieval_zone(T):
    c = g.make_case(max(T, 0), seed=16, sink=16, local=64, update_buf=8, topk=32, max_ctx=T + 64)
    q = np.random.default_rng(0).standard_normal((1, 1, 128)).astype(np.float32)
    qd, idx, k_eff = g.check_retrieve(c, q)
    assert k_eff == min(32, c.zones.N)
    g.check_attention(c, qd, idx, k_eff)


def test_all_candidates_and_k_above_c():
    """cand_bp = 10000 keeps every key; k larger than C returns all of C."""
    c = g.make_case(3000, seed=17, topk=5000, cand_bp=10000)
    q = g.queries_from_zone(c)
    qd, idx, k_eff = g.check_retrieve(c, q)
    assert k_eff == 3000
    g.check_attention(c, qd, idx, k_eff)


def test_flat_votes_every_centroid_uniform():
    """rho = 2^m with flat weights: every key gets B votes (ParisKV's vote
    invariant), so candidates are the lowest positions."""
    c = g.make_case(2000, seed=18, topk=50, cand_bp=1000, rho=256, vote_weighting=P.PARIS_VOTE_FLAT)
    q = g.queries_from_zone(c)
    g.check_retrieve(c, q)
    assert np.all(c.ctx.paris_debug_dump(P.DUMP_VOTES) == 16)


@pytest.mark.parametrize("rho", [1, 2, 8, 15])
def test_rho_range(rho):
    c = g.make_case(6000, seed=19, n_kv_heads=1, n_q_heads=2, topk=64, cand_bp=200, rho=rho)
    g.check_retrieve(c, g.queries_from_zone(c))


def test_ties_duplicates_and_zero_subvectors():
    """Duplicate keys tie in votes and estimates (lower position wins);
    zero keys and zero subvectors give w = 0 and bucket id 0."""
    rng = np.random.default_rng(20)
    base = rng.standard_normal((300, 128)).astype(np.float32)
    K = base[np.arange(6000) % 300].copy()
    K[::7] = 0.0
    K[1::5, 24:32] = 0.0
    K = K[None, None]
    c = g.make_case(6000, seed=20, dtype=torch.float32, K=K, topk=100, cand_bp=500)
    g.check_encoding(c)
    q = np.stack([base[3] + 0.1, np.zeros(128, np.float32)])[None, :1]
    g.check_retrieve(c, q.astype(np.float32))
    g.check_retrieve(c, np.zeros((1, 1, 128), np.float32))


def test_bad_index_is_flagged_not_faulted():
    c = g.make_case(2000, seed=21, sink=4, local=8, topk=16)
    q = g.queries_from_zone(c)
    qd, idx, k_eff = g.check_retrieve(c, q)
    idx[0, 0, 3] = 10 ** 6  # outside the Retrieval zone
    out = torch.zeros((1, 1, 128), dtype=torch.bfloat16, device="cuda")
    c.ctx.paris_sparse_attend(qd, idx, out)
    with pytest.raises(P.ParisError) as e:
        c.ctx.paris_check_device()
    assert e.value.status == P.PARIS_EDEVICE
    c.ctx.paris_check_device()  # cleared


def test_capacity_and_state_errors():
    c = g.make_case(100, seed=22, max_ctx=101, sink=4, local=8)
    k = torch.zeros((1, 1, 128), dtype=torch.bfloat16, device="cuda")
    c.ctx.paris_append_decode(k, k)
    with pytest.raises(P.ParisError) as e:
        c.ctx.paris_append_decode(k, k)
    assert e.value.status == P.PARIS_ECAPACITY
    K = torch.zeros((1, 1, 10, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(P.ParisError) as e:
        c.ctx.paris_encode_prefill(K, K, 10)
    assert e.value.status == P.PARIS_ESTATE


def test_retrieval_zone_in_host_memory_matches_hbm():
    """Retrieval K/V in mapped pinned host memory, read through UVA, give the
    same attention output as the HBM store."""
    kw = dict(seed=23, n_kv_heads=2, n_q_heads=4, sink=16, local=64, update_buf=16, topk=64, cand_bp=500)
    a = g.make_case(8000, retrieval_on_host=0, **kw)
    b = g.make_case(8000, retrieval_on_host=1, **kw)
    q = g.queries_from_zone(a)
    qa, ia, ka = g.check_retrieve(a, q)
    qb, ib, kb = g.check_retrieve(b, q)
    assert torch.equal(ia, ib)
    oa = torch.zeros((1, 4, 128), dtype=torch.bfloat16, device="cuda")
    ob = torch.zeros_like(oa)
    a.ctx.paris_sparse_attend(qa, ia, oa)
    b.ctx.paris_sparse_attend(qb, ib, ob)
    torch.cuda.synchronize()
    assert torch.equal(oa, ob)
    for t in range(20):
        k = synth.decode_keys(23, 1, 2, t, 128, a.scale)
        v = synth.decode_values(23, 1, 2, t, 128)
        g.append(b, k, v)
    qd, idx, k_eff = g.check_retrieve(b, g.queries_from_zone(b, step=5))
    g.check_attention(b, qd, idx, k_eff)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_step_equals_the_three_calls(dtype):
    """paris_decode_step (one fused kernel unless the append flushes) gives
    the top-k and estimates of append + retrieve + sparse_attend bit for bit,
    and their attention output up to float32 summation order, across
    flushes; with float32 inputs the step's own token enters the attention
    converted as the append stores it."""
    kw = dict(seed=24, batch=2, n_kv_heads=2, n_q_heads=4, sink=16, local=64, update_buf=16, topk=64,
              cand_bp=500, rho=4, dtype=dtype)
    a = g.make_case(16 + 20000 + 64, **kw)
    b = g.make_case(16 + 20000 + 64, **kw)
    shp = (2, 4, 64)
    for t in range(60):
        k = synth.drift_keys(24, 2, 2, t, 128, a.scale, rate=0.3)
        v = synth.decode_values(24, 2, 2, t, 128)
        q = g.queries_from_zone(a, step=t)
        kd, vd, qd = g.to_dev(k, dtype), g.to_dev(v, dtype), g.to_dev(q, dtype)
        ia = torch.empty(shp, dtype=torch.int32, device="cuda")
        sa = torch.empty(shp, dtype=torch.float32, device="cuda")
        oa = torch.empty((2, 4, 128), dtype=torch.bfloat16, device="cuda")
        ib, sb, ob = torch.empty_like(ia), torch.empty_like(sa), torch.empty_like(oa)
        a.ctx.paris_append_decode(kd, vd)
        ka = a.ctx.paris_retrieve(qd, ia, sa)
        a.ctx.paris_sparse_attend(qd, ia, oa)
        kb = b.ctx.paris_decode_step(kd, vd, qd, ib, sb, ob)
        torch.cuda.synchronize()
        assert ka == kb
        assert torch.equal(ia, ib) and torch.equal(sa, sb), t
        torch.testing.assert_close(ob.float(), oa.float(), rtol=0, atol=g.ATTN_ATOL)
        g.append(a, k, v, device=False)  # host-side mirror of what both contexts now hold
        if t % 20 == 19:
            g.check_state(a)
            qd2, idx, k_eff = g.check_retrieve(a, q)
            g.check_attention(a, qd2, idx, k_eff)
    assert a.ctx.paris_get_state()["n_flushes"] == b.ctx.paris_get_state()["n_flushes"] > 0


def test_sparse_attend_right_after_a_decode_step_sees_its_token():
    """paris_sparse_attend enqueued on the same stream directly behind
    paris_decode_step (no host synchronisation between them) attends over
    the step's own token as the decode step wrote it into the window: the
    same rows, so the same output up to float32 order, and the oracle's."""
    c = g.make_case(16 + 20000 + 64, seed=27, batch=1, n_kv_heads=2, n_q_heads=8, sink=16, local=64,
                    update_buf=16, topk=64, cand_bp=500, rho=4)
    shp = (1, 8, 64)
    for t in range(40):
        k = synth.decode_keys(27, 1, 2, t, 128, c.scale)
        v = synth.decode_values(27, 1, 2, t, 128)
        q = g.queries_from_zone(c, step=t)
        kd, vd, qd = g.to_dev(k, torch.bfloat16), g.to_dev(v, torch.bfloat16), g.to_dev(q, torch.bfloat16)
        idx = torch.empty(shp, dtype=torch.int32, device="cuda")
        sc = torch.empty(shp, dtype=torch.float32, device="cuda")
        o_step = torch.empty((1, 8, 128), dtype=torch.bfloat16, device="cuda")
        o_call = torch.full((1, 8, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        k_eff = c.ctx.paris_decode_step(kd, vd, qd, idx, sc, o_step)
        c.ctx.paris_sparse_attend(qd, idx, o_call)
        torch.cuda.synchronize()
        torch.testing.assert_close(o_call.float(), o_step.float(), rtol=0, atol=g.ATTN_ATOL)
        g.append(c, k, v, device=False)
        if t % 8 == 7:
            out_h = o_call.float().cpu().numpy()
            idx_h = idx.cpu().numpy()
            Kb, Vb = g.as_seen(c.K, torch.bfloat16), g.as_seen(c.V, torch.bfloat16)
            z = c.zones
            for h in range(8):
                rows = np.concatenate([z.sink(), z.local(), z.buffer(), idx_h[0, h, :k_eff]]).astype(np.int64)
                ref = g.o.attention(qd[0, h].float().cpu().numpy(), Kb[0, h // 4, rows], Vb[0, h // 4, rows])
                assert np.max(np.abs(out_h[0, h] - ref)) <= g.ATTN_ATOL, (t, h)
    c.ctx.paris_check_device()
