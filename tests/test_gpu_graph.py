"""Decode steps of two layers captured in one CUDA graph (the multi-layer
step: one token through every layer's cache in one launch sequence).  The
captured kernels read the zone bookkeeping as it stood at capture; a replay
performs exactly those steps, and replaying again repeats the same work.
Sampled query heads of each layer are checked against the oracle: top-k
positions and estimates bit for bit, the attention within 2e-2 (ParisKV,
system level: the per-layer decode path of the sliding-window cache)."""
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


@pytest.mark.parametrize("on_host", [0, 1])
def test_two_layers_decode_steps_in_one_captured_graph(on_host):
    b, hkv, hq, d, k = 1, 2, 8, 128, 128
    cases = [g.make_case(16 + 20000 + 64, seed=91 + li, batch=b, n_kv_heads=hkv, n_q_heads=hq, sink=16, local=64,
                         update_buf=32, topk=k, cand_bp=500, retrieval_on_host=on_host) for li in range(2)]
    inputs = []
    for li, c in enumerate(cases):
        kn = synth.decode_keys(c.seed, b, hkv, 0, d, c.scale)
        vn = synth.decode_values(c.seed, b, hkv, 0, d)
        q = g.queries_from_zone(c, step=li)
        inputs.append(dict(kn=kn, vn=vn, q=q, kd=g.to_dev(kn, BF), vd=g.to_dev(vn, BF), qd=g.to_dev(q, BF),
                           idx=torch.full((b, hq, k), -7, dtype=torch.int32, device="cuda"),
                           sc=torch.full((b, hq, k), 7.0, dtype=torch.float32, device="cuda"),
                           out=torch.zeros((b, hq, d), dtype=BF, device="cuda")))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    keffs = []
    with torch.cuda.graph(graph, stream=stream):
        for c, x in zip(cases, inputs):
            keffs.append(c.ctx.paris_decode_step(x["kd"], x["vd"], x["qd"], x["idx"], x["sc"], x["out"]))
    for c, x in zip(cases, inputs):
        g.append(c, x["kn"], x["vn"], device=False)  # the captured step's token, on the host mirror
    results = []
    for _ in range(2):  # a second replay repeats the same work
        graph.replay()
        torch.cuda.synchronize()
        results.append([(x["idx"].clone(), x["sc"].clone(), x["out"].clone()) for x in inputs])
    for (i0, s0, o0), (i1, s1, o1) in zip(*results):
        assert torch.equal(i0, i1) and torch.equal(s0, s1) and torch.equal(o0, o1)
    for c, x, k_eff in zip(cases, inputs, keffs):
        c.ctx.paris_check_device()
        g.check_state(c)
        S, N = 16, c.zones.N
        q_seen = g.as_seen(x["q"], BF)
        idx_h, sc_h, out_h = x["idx"].cpu().numpy(), x["sc"].cpu().numpy(), x["out"].float().cpu().numpy()
        for h in (0, 5):
            kvh = h // c.G
            enc = g.oracle_encoding(c, 0, kvh)
            r = o.retrieve_contract(enc, q_seen[0, h], c.signs, 16, 4, 500, k, g.LEV32, "rank")
            assert k_eff == r["k_eff"]
            np.testing.assert_array_equal(idx_h[0, h, :k_eff], S + r["top_idx"])
            assert np.array_equal(sc_h[0, h, :k_eff].view(np.uint32), r["top_est"].view(np.uint32))
            rows = np.concatenate([c.zones.sink(), c.zones.local(), c.zones.buffer(), S + r["top_idx"]]).astype(np.int64)
            Kb, Vb = g.as_seen(c.K, BF), g.as_seen(c.V, BF)
            ref = o.attention(q_seen[0, h], Kb[0, kvh, rows], Vb[0, kvh, rows])
            assert np.max(np.abs(out_h[0, h] - ref)) <= g.ATTN_ATOL, (h, N)
