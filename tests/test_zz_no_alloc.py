"""paris_sparse_attend_noalloc: the attention entry point for callers that
must not allocate device memory (for instance while another component owns
the device allocator, or under a fixed memory budget).  Its scratch is a fixed
area inside the library; it must give what paris_sparse_attend gives (and
the oracle's attention), call after call, and refuse shapes its area cannot
hold.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

from long_context_kv_gb300 import paris as P
from oracle import pariskv as o
from tests import gpu_cases as g

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_kv_gb300 import build
    build.build()
    P.load()


def _check_against_oracle(c, qd, idx, k_eff, got):
    """Every (sequence, query head) of the no-alloc output within 2e-2 of the
    float64 attention over Sink, Local, Update Buffer and its top-k rows."""
    q_seen = qd.float().cpu().numpy()
    idx_h = idx.cpu().numpy()
    got_h = got.float().cpu().numpy()
    Kb, Vb = g.as_seen(c.K, torch.bfloat16), g.as_seen(c.V, torch.bfloat16)
    z = c.zones
    for seq in range(c.cfg["batch"]):
        for qh in range(c.cfg["n_q_heads"]):
            kvh = qh // c.G
            rows = np.concatenate([z.sink(), z.local(), z.buffer(), idx_h[seq, qh, :k_eff]]).astype(np.int64)
            ref = o.attention(q_seen[seq, qh], Kb[seq, kvh, rows], Vb[seq, kvh, rows])
            assert np.max(np.abs(got_h[seq, qh] - ref)) <= g.ATTN_ATOL, (seq, qh)


def test_noalloc_attention_matches_the_context_scratch_version_twice():
    c = g.make_case(16 + 20000 + 64, seed=31, batch=2, n_kv_heads=2, n_q_heads=8, sink=16, local=64,
                    update_buf=16, topk=256, cand_bp=500)
    for step in range(2):  # two calls in a row through the shared fixed area
        q = g.queries_from_zone(c, step=step)
        qd, idx, _, k_eff = g.run_retrieve(c, q)
        ref = torch.zeros((2, 8, 128), dtype=torch.bfloat16, device="cuda")
        got = torch.full((2, 8, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        c.ctx.paris_sparse_attend(qd, idx, ref)
        c.ctx.paris_sparse_attend_noalloc(qd, idx, got)
        torch.cuda.synchronize()
        c.ctx.paris_check_device()
        np.testing.assert_allclose(got.float().cpu().numpy(), ref.float().cpu().numpy(), rtol=0, atol=g.ATTN_ATOL)
        assert k_eff == 256
        _check_against_oracle(c, qd, idx, k_eff, got)


def test_noalloc_attention_across_contexts_of_different_shapes():
    """Calls on two contexts of different shapes share the one area: a large
    call right at its limit (16 query heads x 64 splits = 1024 rows) before
    and after small calls of another shape.  Each must still equal
    paris_sparse_attend (no stale merge counter, no row stride carried over)."""
    big = g.make_case(16 + 5000 + 64, seed=33, n_kv_heads=4, n_q_heads=16, sink=16, local=64, update_buf=16,
                      topk=4000, cand_bp=10000)
    small = g.make_case(16 + 20000 + 64, seed=34, batch=2, n_kv_heads=2, n_q_heads=8, sink=16, local=64,
                        update_buf=16, topk=256, cand_bp=500)

    def compare(c, step):
        b, hq = c.cfg["batch"], c.cfg["n_q_heads"]
        q = g.queries_from_zone(c, step=step)
        qd, idx, _, k_eff = g.run_retrieve(c, q)
        ref = torch.zeros((b, hq, 128), dtype=torch.bfloat16, device="cuda")
        got = torch.full((b, hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        c.ctx.paris_sparse_attend(qd, idx, ref)
        c.ctx.paris_sparse_attend_noalloc(qd, idx, got)
        torch.cuda.synchronize()
        c.ctx.paris_check_device()
        np.testing.assert_allclose(got.float().cpu().numpy(), ref.float().cpu().numpy(), rtol=0, atol=g.ATTN_ATOL)
        _check_against_oracle(c, qd, idx, k_eff, got)
        return k_eff

    assert compare(big, 0) == 4000  # (16 + 64 + 4000) rows -> 64 splits per head
    assert compare(small, 0) == 256
    assert compare(small, 1) == 256
    assert compare(big, 1) == 4000


def test_noalloc_attention_rejects_shapes_beyond_its_area():
    # 64 query heads x ceil((16 + 64 + 4096) / 64) = 66 splits = 4224 rows > 1024
    c = g.make_case(16 + 5000 + 64, seed=32, n_kv_heads=8, n_q_heads=64, sink=16, local=64, update_buf=16,
                    topk=4096, cand_bp=10000)
    q = g.queries_from_zone(c)
    qd, idx, _, k_eff = g.run_retrieve(c, q)
    assert k_eff == 4096
    out = torch.zeros((1, 64, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(P.ParisError) as e:
        c.ctx.paris_sparse_attend_noalloc(qd, idx, out)
    assert e.value.status == P.PARIS_EINVAL
    assert "exceeds its fixed scratch" in str(e.value)
