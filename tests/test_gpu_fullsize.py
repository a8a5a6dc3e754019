"""Parity at the full size the bench times: the Llama-3.1-8B-shaped decode
layer (32 query / 8 KV heads, d = 128, 131072-token bf16 context, S = 16,
L = 512, U = 128, B = 16, rho = 4, 5% candidates, k = 1024), run through
paris_decode_step (the bench's launch configuration: one fused kernel per
step).  The oracle checks sampled query heads one by one: top-k positions
and estimates bit for bit, the attention output within 2e-2 of float64."""
import numpy as np
import pytest
import torch

from long_context_kv_gb300 import paris as P
from long_context_kv_gb300 import synth
from oracle import pariskv as o
from tests import gpu_cases as g

pytestmark = pytest.mark.gpu

CFG = dict(batch=1, n_kv_heads=8, n_q_heads=32, sink=16, local=512, update_buf=128, topk=1024, cand_bp=500,
           rho=4)
T0 = 131072
SAMPLED = [(0, 0), (0, 5), (0, 10), (0, 15), (0, 16), (0, 21), (0, 26), (0, 31)]  # one per KV head


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_kv_gb300 import build
    build.build()
    P.load()


def test_decode_steps_at_full_size_match_the_oracle_on_sampled_heads():
    c = g.make_case(T0, seed=41, max_ctx=T0 + 64, **CFG)
    assert c.zones.N == T0 - 16 - 512
    b, hkv, hq, k = 1, 8, 32, CFG["topk"]
    encs = {}
    for step in range(2):
        kn = synth.decode_keys(c.seed, b, hkv, step, 128, c.scale)
        vn = synth.decode_values(c.seed, b, hkv, step, 128)
        q = g.queries_from_zone(c, step=step)
        kd, vd, qd = g.to_dev(kn, torch.bfloat16), g.to_dev(vn, torch.bfloat16), g.to_dev(q, torch.bfloat16)
        idx = torch.full((b, hq, k), -7, dtype=torch.int32, device="cuda")
        sc = torch.full((b, hq, k), 7.0, dtype=torch.float32, device="cuda")
        out = torch.zeros((b, hq, 128), dtype=torch.bfloat16, device="cuda")
        k_eff = c.ctx.paris_decode_step(kd, vd, qd, idx, sc, out)
        c.ctx.paris_check_device()
        g.append(c, kn, vn, device=False)  # the host mirror of the step's own token
        g.check_state(c)
        idx_h, sc_h, out_h = idx.cpu().numpy(), sc.cpu().numpy(), out.float().cpu().numpy()
        q_seen = g.as_seen(q, torch.bfloat16)
        S, N = CFG["sink"], c.zones.N
        Kb, Vb = g.as_seen(c.K, torch.bfloat16), g.as_seen(c.V, torch.bfloat16)
        for seq, qh in SAMPLED:
            kvh = qh // c.G
            if (seq, kvh) not in encs:
                encs[(seq, kvh)] = g.oracle_encoding(c, seq, kvh)
            r = o.retrieve_contract(encs[(seq, kvh)], q_seen[seq, qh], c.signs, 16, CFG["rho"], CFG["cand_bp"], k,
                                    g.LEV32, "rank")
            assert k_eff == r["k_eff"] == k
            np.testing.assert_array_equal(idx_h[seq, qh], S + r["top_idx"])
            assert np.array_equal(sc_h[seq, qh].view(np.uint32), r["top_est"].view(np.uint32))
            rows = np.concatenate([c.zones.sink(), c.zones.local(), c.zones.buffer(), S + r["top_idx"]]).astype(np.int64)
            ref = o.attention(q_seen[seq, qh], Kb[seq, kvh, rows], Vb[seq, kvh, rows])
            assert np.max(np.abs(out_h[seq, qh] - ref)) <= g.ATTN_ATOL, (step, seq, qh)
        # every query head: a full, in-zone top-k, best first
        g.assert_score_order(idx_h[0], sc_h[0], k)
        assert np.all((idx_h[0] >= S) & (idx_h[0] < S + N))
