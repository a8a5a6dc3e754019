"""Seeded random shapes through the whole path, every stage against the
oracle (ParisKV: the decode step of Methodology 2 and the sliding-window
update mechanism).  Each case draws batch, KV heads, query heads per KV head,
rho, the candidate fraction, k and the zone sizes, then runs decode steps
(appends that flush the Update Buffer included) and checks, on sampled query
heads, the rotated query, its hot centroids, the votes, candidates,
estimates and top-k bit for bit (against the oracle's encoding of every
key, flushed ones included) and the attention within 2e-2.  The shapes
reach the kernel's different regimes: one to five index chunks per head, one
to four blocks per head, candidate lists held in shared memory or not, the
cluster-shared k-th key search, the best-first list placed directly or
sorted, (every fourth case) learned centroids instead of the analytic ones,
and (every sixth) the Retrieval zone's K/V in mapped host memory."""
import numpy as np
import pytest
import torch

from long_context_kv_gb300 import paris as P
from long_context_kv_gb300 import synth
from tests import gpu_cases as g

pytestmark = pytest.mark.gpu

CASES = 24


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_kv_gb300 import build
    build.build()
    P.load()


def draw(i):
    rng = np.random.default_rng(1000 + i)
    N = int(rng.integers(1, 5 * 16384))
    b = int(rng.integers(1, 4))
    hkv = int(rng.integers(1, 4))
    while b * hkv * N > 240000 and b * hkv > 1:  # keep the host-side oracle quick
        b, hkv = (b - 1, hkv) if b >= hkv else (b, hkv - 1)
    G = int(rng.choice([1, 2, 4]))
    S = int(rng.choice([0, 4, 16]))
    L = int(rng.choice([0, 32, 128]))
    U = int(rng.choice([8, 16, 32]))
    cand_bp = int(rng.choice([100, 500, 2000, 10000]))
    k = int(rng.choice([1, 64, 300, 1024, 2048]))
    rho = int(rng.integers(1, 9))
    order = P.PARIS_TOPK_BY_SCORE if rng.random() < 0.8 else P.PARIS_TOPK_BY_POSITION
    table = None
    if i % 4 == 3:  # learned centroids: a random unit table per KV head
        table = rng.standard_normal((hkv, 16, 256, 8)).astype(np.float32)
        table /= np.linalg.norm(table, axis=-1, keepdims=True)
    host = 1 if i % 6 == 5 else 0  # every sixth case: Retrieval K/V in mapped host memory
    return dict(T=S + N + L, batch=b, n_kv_heads=hkv, n_q_heads=hkv * G, sink=S, local=L, update_buf=U,
                topk=k, cand_bp=cand_bp, rho=rho, topk_order=order, seed=2000 + i, table=table,
                retrieval_on_host=host)


@pytest.mark.parametrize("i", range(CASES))
def test_random_shapes_every_stage_matches_the_oracle(i):
    c_ = draw(i)
    T, seed = c_.pop("T"), c_.pop("seed")
    c = g.make_case(T, seed=seed, max_ctx=T + 3 * c_["update_buf"] + 8, **c_)
    b, hkv, hq = c.cfg["batch"], c.cfg["n_kv_heads"], c.cfg["n_q_heads"]
    rng = np.random.default_rng(3000 + i)
    heads = sorted({(int(rng.integers(0, b)), int(rng.integers(0, hq))) for _ in range(3)})
    steps = c.cfg["update_buf"] + 2  # one flush among them
    for step in range(steps):
        kn = synth.decode_keys(seed, b, hkv, step, 128, c.scale)
        vn = synth.decode_values(seed, b, hkv, step, 128)
        q = g.queries_from_zone(c, step=step)
        qd = g.to_dev(q, torch.bfloat16)
        k = c.cfg["topk"]
        idx = torch.full((b, hq, k), -7, dtype=torch.int32, device="cuda")
        sc = torch.full((b, hq, k), 7.0, dtype=torch.float32, device="cuda")
        out = torch.zeros((b, hq, 128), dtype=torch.bfloat16, device="cuda")
        c.ctx.paris_decode_step(g.to_dev(kn, torch.bfloat16), g.to_dev(vn, torch.bfloat16), qd, idx, sc, out)
        c.ctx.paris_check_device()
        g.append(c, kn, vn, device=False)
        g.check_state(c)
        if step in (0, steps - 1):  # the first step and the one after the flush: every stage
            qd2, idx2, k_eff = g.check_retrieve(c, q, heads=heads)
            assert torch.equal(idx2, idx) or c.zones.N == 0
            g.check_attention(c, qd2, idx2, k_eff, heads=heads)
            if c.cfg["topk_order"] == P.PARIS_TOPK_BY_SCORE and k_eff > 0:
                g.assert_score_order(idx2.cpu().numpy(), sc.cpu().numpy(), k_eff)
