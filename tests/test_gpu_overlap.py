"""How much of a layer's top-k carries over from one decode step to the next,
on the Qwen3-8B-shaped workload (batch 8, 32 query / 8 KV heads, a
32768-token prompt, rho = 4, 5% candidates, k = 1024).  A row cache in HBM
for a host-resident Retrieval zone pays only in proportion to this overlap
(ParisKV, System-level innovations, "UVA offloading": the top-k rows are
read from host memory every step).

The pages fix no model of how a decode step's query relates to the previous
one, so the overlap is measured as a function of that relation: each step's
queries are a correlated walk from the previous step's (cos about c, for c
from 0, independent queries, to 0.99).  For every c, nine consecutive
paris_decode_step calls; the overlap of ParisKV's top-k with the previous
step's, with the union of the four previous steps', and the same for the
exact float64 top-k, are printed (and written where PARIS_OVERLAP names).
The first step's top-k is checked bit for bit against the oracle on sampled
heads."""
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
CORR = (0.0, 0.5, 0.9, 0.97, 0.99)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_kv_gb300 import build
    build.build()
    P.load()


def _carried(cur: torch.Tensor, prev: list) -> float:
    """Mean over (sequence, query head) of the share of cur's rows found in
    any of the prev top-k lists (all [batch, Hq, k'])."""
    held = torch.cat(prev, dim=-1)
    b, hq, k = cur.shape
    return float(np.mean([torch.isin(cur[s, h], held[s, h]).float().mean().item()
                          for s in range(b) for h in range(hq)]))


def test_topk_overlap_between_consecutive_decode_steps_qwen3_shaped():
    b, hkv, hq, d, S, Lw, U, k, bp, rho, T0, seed = 8, 8, 32, 128, 16, 512, 128, 1024, 500, 4, 32768, 47
    c = g.make_case(T0, seed=seed, batch=b, n_kv_heads=hkv, n_q_heads=hq, sink=S, local=Lw, update_buf=U, topk=k,
                    cand_bp=bp, rho=rho, max_ctx=T0 + 64)
    G, N = hq // hkv, c.zones.N
    Kz = torch.from_numpy(np.ascontiguousarray(g.as_seen(c.K, BF)[:, :, S:S + N])).cuda().double()
    idx = torch.empty((b, hq, k), dtype=torch.int32, device="cuda")
    sc = torch.empty((b, hq, k), dtype=torch.float32, device="cuda")
    out = torch.empty((b, hq, d), dtype=BF, device="cuda")

    def exact_topk(qd):
        qq = qd.double().view(b, hkv, G, d)
        scores = torch.einsum("bhnd,bhgd->bhgn", Kz, qq)  # [b, Hkv, G, N]
        return (torch.topk(scores, k, dim=-1).indices + S).view(b, hq, k).int()

    result, step, held1, held4 = {}, 0, {}, {}
    for corr in CORR:
        q = g.queries_from_zone(c, step=int(corr * 1000))
        ours, exact, r1, r4, e1, e4 = [], [], [], [], [], []
        for t in range(9):
            if t:
                q = synth.query_walk(seed, q, corr, step)
            kn = synth.decode_keys(seed, b, hkv, step, d, c.scale)
            vn = synth.decode_values(seed, b, hkv, step, d)
            qd = g.to_dev(q, BF)
            k_eff = c.ctx.paris_decode_step(g.to_dev(kn, BF), g.to_dev(vn, BF), qd, idx, sc, out)
            assert k_eff == k
            if step == 0:  # the first step against the oracle (the new token sits in the Update Buffer)
                q_seen, idx_h, sc_h = g.as_seen(q, BF), idx.cpu().numpy(), sc.cpu().numpy()
                for s, h in ((0, 0), (7, 29)):
                    enc = g.oracle_encoding(c, s, h // G)
                    r = o.retrieve_contract(enc, q_seen[s, h], c.signs, 16, rho, bp, k, g.LEV32, "rank")
                    np.testing.assert_array_equal(idx_h[s, h], S + r["top_idx"])
                    assert np.array_equal(sc_h[s, h].view(np.uint32), r["top_est"].view(np.uint32))
            step += 1
            ours.append(idx.clone())
            exact.append(exact_topk(qd))
            if t:
                r1.append(_carried(ours[-1], ours[-2:-1]))
                e1.append(_carried(exact[-1], exact[-2:-1]))
            if t >= 4:
                r4.append(_carried(ours[-1], ours[-5:-1]))
                e4.append(_carried(exact[-1], exact[-5:-1]))
        held1[corr], held4[corr] = r1, r4
        result[str(corr)] = {"paris_prev_step": float(np.mean(r1)), "paris_prev_4_steps": float(np.mean(r4)),
                             "exact_prev_step": float(np.mean(e1)), "exact_prev_4_steps": float(np.mean(e4))}
    torch.cuda.synchronize()
    c.ctx.paris_check_device()
    st = c.ctx.paris_get_state()
    assert (st["T"], st["N"], st["n_buf"]) == (T0 + step, N, step)
    print("top-k overlap between consecutive decode steps vs query correlation:", json.dumps(result))
    path = os.environ.get("PARIS_OVERLAP")
    if path:
        with open(path, "w") as f:
            json.dump(result, f)
    for v in result.values():
        assert all(0.0 <= x <= 1.0 for x in v.values())
    for corr in CORR:  # a union of four lists holds at least what the last one does
        assert np.all(np.array(held4[corr]) >= np.array(held1[corr][3:]) - 1e-9)
    # more correlated queries share more rows
    assert result["0.99"]["paris_prev_step"] > result["0.0"]["paris_prev_step"]
