"""The k-th best estimate when a query head has far more candidates than a
block of the decode kernel holds (ParisKV, Methodology 2, "Candidate
reranking (RSQ-IP)": the k best candidates by estimate).  Past 24576
candidates the cluster shares the search: each block histograms its own
slice, the blocks exchange histograms, then the few keys of the k-th bin.
Checked bit for bit against the oracle, stage by stage, on a 60000-key zone
with every key a candidate, both with distinct estimates (the shared search
decides) and with every key repeated 200 times (the k-th bin holds more keys
than the shared search ranks, so every block falls back to searching all
keys itself); then the sparse attention over the rows it selects."""
import numpy as np
import pytest

from long_context_kv_gb300 import paris as P
from long_context_kv_gb300 import synth
from tests import gpu_cases as g

pytestmark = pytest.mark.gpu

T = 16 + 60000 + 64
KW = dict(batch=1, n_kv_heads=1, n_q_heads=4, sink=16, local=64, update_buf=32, topk=700, cand_bp=10000)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_kv_gb300 import build
    build.build()
    P.load()


@pytest.mark.parametrize("repeat", [1, 200])
def test_many_candidates_shared_search_matches_the_oracle(repeat):
    scale = synth.channel_scale(91, 1, 128)
    base = synth.keys(91, 1, 1, 0, -(-T // repeat), 128, scale)
    K = np.ascontiguousarray(np.repeat(base, repeat, axis=2)[:, :, :T])
    c = g.make_case(T, seed=91, K=K, **KW)
    assert c.zones.N == 60000  # C = N: every key is a candidate, well past 24576
    qd, idx, k_eff = g.check_retrieve(c, g.queries_from_zone(c))
    assert k_eff == 700
    idx_h = idx.cpu().numpy()
    if repeat > 1:  # ties at the k-th estimate: the lowest positions are taken first
        for h in range(4):
            e = c.ctx.paris_debug_dump(P.DUMP_CAND_EST, 0, h)
            assert np.sum(np.diff(np.sort(e)) == 0) > 0
    g.check_attention(c, qd, idx, k_eff)
    assert np.all(idx_h[..., k_eff:] == -1)
