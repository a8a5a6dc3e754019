"""Parity on the three remaining workloads, at their full sizes, on sampled
outputs the oracle computes one by one:

* long generation under drift (Qwen3-8B-shaped: batch 8, 32 q / 8 KV heads,
  32768-token prompt, 4096 decode steps whose new keys drift by 0.02 sigma
  per 256 steps, update buffer 128 flushed Local -> Retrieval every 128
  steps), every step through paris_decode_step, checked at sampled steps;
* a 1M-token context whose Retrieval-zone K/V live in pinned host memory
  (read by the kernels through UVA), k = 2048, 5% candidates: more
  candidates than the kernels keep in shared memory;
* the sweep at 256K tokens, batch 5: candidate fraction 2-20%, rho 1-8,
  k 256-4096.

Top-k positions and estimates are compared bit for bit; the attention output
within 2e-2 of float64 (ParisKV — Methodology, Candidate reranking; System,
Sliding-window update mechanism)."""
import numpy as np
import pytest
import torch

from long_context_kv_gb300 import paris as P
from long_context_kv_gb300 import synth
from oracle import pariskv as o
from tests import gpu_cases as g

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_kv_gb300 import build
    build.build()
    P.load()


def _check_head(enc, q_seen, signs, rho, cand_bp, k, idx_h, sc_h, S):
    r = o.retrieve_contract(enc, q_seen, signs, 16, rho, cand_bp, k, g.LEV32, "rank")
    np.testing.assert_array_equal(idx_h[:r["k_eff"]], S + r["top_idx"])
    assert np.array_equal(sc_h[:r["k_eff"]].view(np.uint32), r["top_est"].view(np.uint32))
    assert np.all(idx_h[r["k_eff"]:] == -1)
    return r


def _attention_rows(z, top):
    return np.concatenate([z.sink(), z.local(), z.buffer(), top]).astype(np.int64)


def test_long_generation_under_drift_sampled_steps():
    b, hkv, hq, d, S, Lw, U, k, rho, bp = 8, 8, 32, 128, 16, 512, 128, 1024, 4, 500
    T0, STEPS, seed = 32768, 4096, 43
    G = hq // hkv
    check_at = {0, 127, 128, 1000, 2047, 4095}  # 127: a flush step; 128: the step after it
    sampled = [(0, 0), (3, 17), (7, 31)]
    scale = synth.channel_scale(seed, hkv, d)
    signs = synth.srht_signs(seed, d)
    cfg = P.make_config(batch=b, n_kv_heads=hkv, n_q_heads=hq, head_dim=d, n_sub=16, rho=rho, sink=S, local=Lw,
                        update_buf=U, topk=k, cand_bp=bp, max_ctx=T0 + STEPS + 8, retrieval_on_host=0)
    ctx = P.Context(cfg, signs)
    # host mirror of every token as the library stores it (bf16), preallocated for all steps
    Km = np.empty((b, hkv, T0 + STEPS, d), dtype=np.float32)
    Vm = np.empty_like(Km)
    Kd = torch.empty((b, hkv, T0, d), dtype=BF, device="cuda")
    Vd = torch.empty_like(Kd)
    for s in range(b):
        for h in range(hkv):
            kt = torch.from_numpy(synth.key_rows(seed, s, h, 0, T0, d, scale)).to(BF)
            vt = torch.from_numpy(synth.value_rows(seed, s, h, 0, T0, d)).to(BF)
            Kd[s, h].copy_(kt)
            Vd[s, h].copy_(vt)
            Km[s, h, :T0] = kt.float().numpy()
            Vm[s, h, :T0] = vt.float().numpy()
    ctx.paris_encode_prefill(Kd, Vd, T0)
    del Kd, Vd
    z = o.Zones(S, Lw, U)
    z.prefill(T0)
    idx = torch.empty((b, hq, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((b, hq, k), dtype=torch.float32, device="cuda")
    out = torch.empty((b, hq, d), dtype=BF, device="cuda")
    kvh_of = np.arange(hq) // G
    recall = {}
    for step in range(STEPS):
        kn = g.as_seen(synth.drift_keys(seed, b, hkv, step, d, scale), BF)
        vn = g.as_seen(synth.decode_values(seed, b, hkv, step, d), BF)
        t = z.T
        Km[:, :, t], Vm[:, :, t] = kn, vn
        z.append()
        pos = synth.query_positions(seed, b, hq, S, S + z.N, step)
        picked = Km[np.arange(b)[:, None], kvh_of[None, :], pos]
        q = g.as_seen(synth.queries_from_keys(seed, picked, 0.5, step), BF)
        k_eff = ctx.paris_decode_step(g.to_dev(kn, BF), g.to_dev(vn, BF), g.to_dev(q, BF), idx, sc, out)
        if step not in check_at:
            continue
        ctx.paris_check_device()
        st = ctx.paris_get_state()
        assert (st["T"], st["N"], st["n_local"], st["n_buf"]) == (z.T, z.N, z.n_local, z.n_buf)
        C = o.candidate_count(z.N, bp, k)
        assert k_eff == min(k, C)
        idx_h, sc_h, out_h = idx.cpu().numpy(), sc.cpu().numpy(), out.float().cpu().numpy()
        encs, rs = {}, []
        for seq, qh in sampled:
            kvh = qh // G
            if (seq, kvh) not in encs:
                encs[(seq, kvh)] = o.encode_contract(Km[seq, kvh, S:S + z.N], signs, 16, g.LEV32, g.THR32)
            r = _check_head(encs[(seq, kvh)], q[seq, qh], signs, rho, bp, k, idx_h[seq, qh], sc_h[seq, qh], S)
            rows = _attention_rows(z, S + r["top_idx"])
            ref = o.attention(q[seq, qh], Km[seq, kvh, rows], Vm[seq, kvh, rows])
            assert np.max(np.abs(out_h[seq, qh] - ref)) <= g.ATTN_ATOL, (step, seq, qh)
            truth = o.exact_topk(Km[seq, kvh, S:S + z.N], q[seq, qh], k_eff)
            rs.append(o.recall(idx_h[seq, qh, :k_eff] - S, truth))
        recall[step] = float(np.mean(rs))
        # every head: a full top-k inside the Retrieval zone, best first
        g.assert_score_order(idx_h, sc_h, k_eff)
        assert np.all((idx_h >= S) & (idx_h < S + z.N))
    print("recall@k vs decode step under drift:", recall)
    assert z.N == T0 - S - Lw + (STEPS // U) * U


def test_one_million_tokens_retrieval_zone_in_host_memory():
    b, hkv, hq, d, S, Lw, U, k, rho, bp = 1, 8, 32, 128, 16, 512, 128, 2048, 4, 500
    T, seed = 1 << 20, 44
    G = hq // hkv
    sampled = [(0, 0), (0, 22)]
    scale = synth.channel_scale(seed, hkv, d)
    signs = synth.srht_signs(seed, d)
    cfg = P.make_config(batch=b, n_kv_heads=hkv, n_q_heads=hq, head_dim=d, n_sub=16, rho=rho, sink=S, local=Lw,
                        update_buf=U, topk=k, cand_bp=bp, max_ctx=T + 16, retrieval_on_host=1)
    ctx = P.Context(cfg, signs)
    Kd = torch.empty((b, hkv, T, d), dtype=BF, device="cuda")
    Vd = torch.empty_like(Kd)
    keep = {}
    for h in range(hkv):
        kt = torch.from_numpy(synth.key_rows(seed, 0, h, 0, T, d, scale)).to(BF)
        vt = torch.from_numpy(synth.value_rows(seed, 0, h, 0, T, d)).to(BF)
        Kd[0, h].copy_(kt)
        Vd[0, h].copy_(vt)
        if h in {qh // G for _, qh in sampled}:
            keep[h] = (np.concatenate([kt.float().numpy(), np.zeros((2, d), np.float32)]),
                       np.concatenate([vt.float().numpy(), np.zeros((2, d), np.float32)]))
    ctx.paris_encode_prefill(Kd, Vd, T)
    z = o.Zones(S, Lw, U)
    z.prefill(T)
    # two steps' queries, drawn from the Retrieval zone while all keys are on the device
    kvh_of = torch.arange(hq, device="cuda") // G
    qs = []
    for step in range(2):
        pos = torch.from_numpy(synth.query_positions(seed, b, hq, S, S + z.N, step)).cuda()
        picked = Kd[0, kvh_of, pos[0]].float().cpu().numpy()[None]
        qs.append(g.as_seen(synth.queries_from_keys(seed, picked, 0.5, step), BF))
    del Kd, Vd
    torch.cuda.synchronize()
    encs = {h: o.encode_contract(keep[h][0][S:S + z.N], signs, 16, g.LEV32, g.THR32) for h in keep}
    C = o.candidate_count(z.N, bp, k)
    assert C > 4 * 4096  # more candidates than the block slices and the top-k keep in shared memory

    def check(q, idx, sc, out):
        idx_h, sc_h, out_h = idx.cpu().numpy(), sc.cpu().numpy(), out.float().cpu().numpy()
        for seq, qh in sampled:
            kvh = qh // G
            r = _check_head(encs[kvh], q[seq, qh], signs, rho, bp, k, idx_h[seq, qh], sc_h[seq, qh], S)
            rows = _attention_rows(z, S + r["top_idx"])
            ref = o.attention(q[seq, qh], keep[kvh][0][rows], keep[kvh][1][rows])
            assert np.max(np.abs(out_h[seq, qh] - ref)) <= g.ATTN_ATOL, (seq, qh)
        g.assert_score_order(idx_h[0], sc_h[0], k)
        assert np.all((idx_h[0] >= S) & (idx_h[0] < S + z.N))

    # the separate calls: paris_retrieve, then paris_sparse_attend gathering host-resident rows
    idx = torch.full((b, hq, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((b, hq, k), 7.0, dtype=torch.float32, device="cuda")
    out = torch.zeros((b, hq, d), dtype=BF, device="cuda")
    qd = g.to_dev(qs[0], BF)
    assert ctx.paris_retrieve(qd, idx, sc) == k
    ctx.paris_sparse_attend(qd, idx, out)
    ctx.paris_check_device()
    check(qs[0], idx, sc, out)
    # one fused decode step with a new token
    kn = g.as_seen(synth.decode_keys(seed, b, hkv, 0, d, scale), BF)
    vn = g.as_seen(synth.decode_values(seed, b, hkv, 0, d), BF)
    for h in keep:
        keep[h][0][z.T], keep[h][1][z.T] = kn[0, h], vn[0, h]
    z.append()
    assert ctx.paris_decode_step(g.to_dev(kn, BF), g.to_dev(vn, BF), g.to_dev(qs[1], BF), idx, sc, out) == k
    ctx.paris_check_device()
    check(qs[1], idx, sc, out)


SWEEP = [  # (candidates in basis points, rho, k): the grid's corners and interior points
    (200, 1, 256),
    (200, 8, 4096),
    (2000, 1, 256),
    (2000, 8, 4096),
    (500, 4, 1024),
    (1000, 2, 4096),
    (500, 2, 512),
    (1000, 4, 2048),
]


def test_sweep_at_256k_batch_5():
    b, hkv, hq, d, S, Lw, U = 5, 8, 32, 128, 16, 512, 128
    T, seed = 1 << 18, 45
    G = hq // hkv
    sampled = [(0, 0), (2, 13), (4, 31)]
    scale = synth.channel_scale(seed, hkv, d)
    signs = synth.srht_signs(seed, d)
    Kd = torch.empty((b, hkv, T, d), dtype=BF, device="cuda")
    Vd = torch.empty_like(Kd)
    keep = {}
    for s in range(b):
        for h in range(hkv):
            kt = torch.from_numpy(synth.key_rows(seed, s, h, 0, T, d, scale)).to(BF)
            vt = torch.from_numpy(synth.value_rows(seed, s, h, 0, T, d)).to(BF)
            Kd[s, h].copy_(kt)
            Vd[s, h].copy_(vt)
            if (s, h) in {(seq, qh // G) for seq, qh in sampled}:
                keep[(s, h)] = (kt.float().numpy(), vt.float().numpy())
    z = o.Zones(S, Lw, U)
    z.prefill(T)
    pos = torch.from_numpy(synth.query_positions(seed, b, hq, S, S + z.N, 0)).cuda()
    kvh_of = torch.arange(hq, device="cuda") // G
    picked = Kd[torch.arange(b, device="cuda")[:, None], kvh_of[None, :], pos].float().cpu().numpy()
    q = g.as_seen(synth.queries_from_keys(seed, picked, 0.5, 0), BF)
    qd = g.to_dev(q, BF)
    encs = {key: o.encode_contract(kv[0][S:S + z.N], signs, 16, g.LEV32, g.THR32) for key, kv in keep.items()}
    for bp, rho, k in SWEEP:
        cfg = P.make_config(batch=b, n_kv_heads=hkv, n_q_heads=hq, head_dim=d, n_sub=16, rho=rho, sink=S, local=Lw,
                            update_buf=U, topk=k, cand_bp=bp, max_ctx=T + 16, retrieval_on_host=0)
        ctx = P.Context(cfg, signs)
        ctx.paris_encode_prefill(Kd, Vd, T)
        idx = torch.full((b, hq, k), -7, dtype=torch.int32, device="cuda")
        sc = torch.full((b, hq, k), 7.0, dtype=torch.float32, device="cuda")
        out = torch.zeros((b, hq, d), dtype=BF, device="cuda")
        k_eff = ctx.paris_retrieve(qd, idx, sc)
        ctx.paris_sparse_attend(qd, idx, out)
        ctx.paris_check_device()
        assert k_eff == min(k, o.candidate_count(z.N, bp, k))
        idx_h, sc_h, out_h = idx.cpu().numpy(), sc.cpu().numpy(), out.float().cpu().numpy()
        for seq, qh in sampled:
            kvh = qh // G
            r = _check_head(encs[(seq, kvh)], q[seq, qh], signs, rho, bp, k, idx_h[seq, qh], sc_h[seq, qh], S)
            rows = _attention_rows(z, S + r["top_idx"])
            ref = o.attention(q[seq, qh], keep[(seq, kvh)][0][rows], keep[(seq, kvh)][1][rows])
            assert np.max(np.abs(out_h[seq, qh] - ref)) <= g.ATTN_ATOL, (bp, rho, k, seq, qh)
        g.assert_score_order(idx_h, sc_h, k_eff)
        assert np.all((idx_h >= S) & (idx_h < S + z.N))
        ctx.close()
        del ctx
