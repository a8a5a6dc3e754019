"""Analytic against learned centroids under decoding drift, on the
Qwen3-8B-shaped long-generation workload as configured: batch 8, 32 query /
8 KV heads, a 32768-token prompt, 4096 decode steps whose new keys drift by
0.02 sigma per 256 steps, the Update Buffer (128) flushed Local -> Retrieval
32 times (ParisKV, "Problem definition": centroids learned on the prefill
keys go stale as decode-time keys drift; "Drift-robust analytic centroids").

Both contexts take the same tokens and queries through paris_decode_step.
Every 256 steps recall@k against the exact float64 top-k is measured for two
query sets: queries drawn uniformly from the current Retrieval zone (the
workload's own) and queries near the 2048 newest Retrieval-zone keys (the
most drifted ones).  The curves are printed; the learned context's top-k is
checked bit for bit against the oracle on sampled heads at the end."""
import json
import os

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


def _recall(ctx, Kd, S, N, q, k):
    """Mean recall@k over every (sequence, query head) of one retrieval."""
    b, hq = q.shape[:2]
    hkv = Kd.shape[1]
    G = hq // hkv
    idx = torch.empty((b, hq, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((b, hq, k), dtype=torch.float32, device="cuda")
    qd = q.to(BF).contiguous()
    k_eff = ctx.paris_retrieve(qd, idx, sc)
    rs = []
    for s in range(b):
        for h in range(hkv):
            Kz = Kd[s, h, S:S + N].double()
            ex = torch.topk(Kz @ qd[s, h * G:(h + 1) * G].double().T, k_eff, dim=0).indices + S
            for gi in range(G):
                got = idx[s, h * G + gi, :k_eff].long()
                rs.append(torch.isin(got, ex[:, gi]).float().mean().item())
    return float(np.mean(rs))


def test_recall_under_drift_qwen3_shaped_analytic_versus_learned():
    b, hkv, hq, d, S, Lw, U, k, bp, rho = 8, 8, 32, 128, 16, 512, 128, 1024, 500, 4
    T0, steps, rate, seed = 32768, 4096, 0.02, 47
    G = hq // hkv
    scale = synth.channel_scale(seed, hkv, d)
    signs = synth.srht_signs(seed, d)
    # every token as the library stores it (bf16 values), prompt then decode steps
    Km = np.empty((b, hkv, T0 + steps, d), dtype=np.float32)
    Vm = np.empty_like(Km)
    for s in range(b):
        for h in range(hkv):
            Km[s, h, :T0] = g.as_seen(synth.key_rows(seed, s, h, 0, T0, d, scale), BF)
            Vm[s, h, :T0] = g.as_seen(synth.value_rows(seed, s, h, 0, T0, d), BF)
    for t in range(steps):
        Km[:, :, T0 + t] = g.as_seen(synth.drift_keys(seed, b, hkv, t, d, scale, rate=rate), BF)
        Vm[:, :, T0 + t] = g.as_seen(synth.decode_values(seed, b, hkv, t, d), BF)
    Kd = torch.from_numpy(Km).to(BF).cuda()
    Vd = torch.from_numpy(Vm).to(BF).cuda()
    # learned centroids: spherical k-means per KV head on a 16384-key sample
    # of sequence 0's rotated prompt keys (Retrieval zone)
    rng = np.random.default_rng(seed)
    tabs = []
    for h in range(hkv):
        sample = Km[0, h, S + rng.choice(T0 - S - Lw, 16384, replace=False)]
        z = o.fwht(sample * signs.astype(np.float32)[None, :])
        tabs.append(o.kmeans_table(z.reshape(-1, 16, 8), 256, iters=4, seed=seed + h))
    table = np.ascontiguousarray(np.stack(tabs), dtype=np.float32)
    cfg = dict(batch=b, n_kv_heads=hkv, n_q_heads=hq, head_dim=d, n_sub=16, rho=rho, sink=S, local=Lw,
               update_buf=U, topk=k, cand_bp=bp, max_ctx=T0 + steps + 8, retrieval_on_host=0)
    ctxs = {"analytic": P.Context(P.make_config(**cfg), signs), "learned": P.Context(P.make_config(**cfg), signs)}
    ctxs["learned"].paris_set_centroids(torch.from_numpy(table).cuda())
    for c in ctxs.values():
        c.paris_encode_prefill(Kd[:, :, :T0].contiguous(), Vd[:, :, :T0].contiguous(), T0)
    z = o.Zones(S, Lw, U)
    z.prefill(T0)
    kvh_of = np.arange(hq) // G
    idx = torch.empty((b, hq, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((b, hq, k), dtype=torch.float32, device="cuda")
    out = torch.empty((b, hq, d), dtype=BF, device="cuda")
    curves = {name: {"zone": {}, "newest": {}} for name in ctxs}

    def queries(lo, hi, tag):
        pos = synth.query_positions(seed, b, hq, lo, hi, tag)
        picked = np.stack([np.stack([Km[s, kvh_of[h], pos[s, h]] for h in range(hq)]) for s in range(b)])
        return torch.from_numpy(synth.queries_from_keys(seed, picked, 0.5, tag)).cuda()

    for t in range(steps):
        kn, vn = Kd[:, :, T0 + t].contiguous(), Vd[:, :, T0 + t].contiguous()
        q = queries(S, S + z.N, t).to(BF).contiguous()  # the step's queries: the Retrieval zone as it stands
        z.append()
        for c in ctxs.values():
            c.paris_decode_step(kn, vn, q, idx, sc, out)
        if t % 256 == 255 or t == 0:
            for name, c in ctxs.items():
                curves[name]["zone"][t + 1] = _recall(c, Kd, S, z.N, queries(S, S + z.N, 10**6 + t), k)
                curves[name]["newest"][t + 1] = _recall(c, Kd, S, z.N, queries(S + z.N - 2048, S + z.N, 2 * 10**6 + t),
                                                        k)
    torch.cuda.synchronize()
    for c in ctxs.values():
        c.paris_check_device()
        st = c.paris_get_state()
        assert (st["T"], st["N"], st["n_flushes"]) == (z.T, z.N, steps // U)
    print("recall@k vs decode step (drift 0.02 sigma / 256 steps):", json.dumps(curves))
    path = os.environ.get("PARIS_DRIFT_CURVES")
    if path:
        with open(path, "w") as f:
            json.dump(curves, f)
    # the learned context against the oracle on sampled heads after the last step
    q = queries(S, S + z.N, 3 * 10**6)
    qd = q.to(BF).contiguous()
    k_eff = ctxs["learned"].paris_retrieve(qd, idx, sc)
    idx_h, sc_h, q_seen = idx.cpu().numpy(), sc.cpu().numpy(), g.as_seen(q.cpu().numpy(), BF)
    for s, h in ((0, 0), (5, 23)):
        kvh = kvh_of[h]
        enc = o.encode_contract(Km[s, kvh, S:S + z.N], signs, 16, g.LEV32, g.THR32, table[kvh])
        r = o.retrieve_contract(enc, q_seen[s, h], signs, 16, rho, bp, k, g.LEV32, "rank", table[kvh])
        assert k_eff == r["k_eff"]
        np.testing.assert_array_equal(idx_h[s, h, :k_eff], S + r["top_idx"])
        assert np.array_equal(sc_h[s, h, :k_eff].view(np.uint32), r["top_est"].view(np.uint32))
    for name in ctxs:
        assert len(curves[name]["zone"]) == steps // 256 + 1
        assert all(0.0 < v <= 1.0 for v in curves[name]["zone"].values())
