"""Shared machinery of the GPU parity tests: build a context through the
C ABI from seeded synthetic inputs, and compare every stage with the oracle.

The oracle sees exactly the values the library sees: float32 inputs as they
are, bf16 inputs converted to float32 exactly, and attention K/V rounded to
bf16 (the library stores K/V as bf16)."""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from long_context_kv_gb300 import paris as P
from long_context_kv_gb300 import synth
from oracle import pariskv as o

LEV32, THR32 = o.rsq_levels_f32(8)
SCORE_RTOL = 1e-4     # rerank estimates vs the float32 contract oracle
ATTN_ATOL = 2e-2      # bf16 attention output vs the float64 oracle


def to_dev(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).cuda().contiguous()


def as_seen(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """The float32 values the library reads from an input of this dtype."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).float().numpy()


@dataclass
class Case:
    cfg: dict
    seed: int = 1
    dtype: torch.dtype = torch.bfloat16
    T: int = 0
    K: np.ndarray = None    # float32 [batch, Hkv, T, d] as the library sees it
    V: np.ndarray = None
    signs: np.ndarray = None
    ctx: P.Context = None
    zones: list = field(default_factory=list)
    appended: int = 0
    table: np.ndarray = None  # learned centroids [Hkv][16][256][8] (None: analytic)

    @property
    def G(self):
        return self.cfg["n_q_heads"] // self.cfg["n_kv_heads"]


def make_case(T: int, seed: int = 1, dtype=torch.bfloat16, K=None, table=None, **cfg_kw) -> Case:
    cfg = dict(batch=1, n_kv_heads=1, n_q_heads=1, head_dim=128, n_sub=16, rho=4, sink=0, local=0,
               update_buf=128, topk=64, cand_bp=1000, max_ctx=T + 1024, retrieval_on_host=0,
               vote_weighting=P.PARIS_VOTE_RANK)
    cfg.update(cfg_kw)
    b, h, d = cfg["batch"], cfg["n_kv_heads"], cfg["head_dim"]
    scale = synth.channel_scale(seed, h, d)
    if K is None:
        K = synth.keys(seed, b, h, 0, T, d, scale)
    V = synth.values(seed, b, h, 0, T, d)
    c = Case(cfg=cfg, seed=seed, dtype=dtype, T=T)
    c.signs = synth.srht_signs(seed, d)
    c.ctx = P.Context(P.make_config(**cfg), c.signs)
    if table is not None:
        c.table = np.ascontiguousarray(table, dtype=np.float32)
        c.ctx.paris_set_centroids(torch.from_numpy(c.table).cuda())
    Kd, Vd = to_dev(K, dtype), to_dev(V, dtype)
    c.ctx.paris_encode_prefill(Kd, Vd, T)
    torch.cuda.synchronize()
    c.K = as_seen(K, dtype)
    c.V = as_seen(V, dtype)
    c.zones = o.Zones(cfg["sink"], cfg["local"], cfg["update_buf"])
    c.zones.prefill(T)
    c.scale = scale
    return c


def append(c: Case, k: np.ndarray, v: np.ndarray, device: bool = True):
    """Append one token per (sequence, KV head): k, v float32 [batch, Hkv, d].
    device=False only updates the host-side mirror (the library already has it)."""
    if device:
        c.ctx.paris_append_decode(to_dev(k, c.dtype), to_dev(v, c.dtype))
    c.K = np.concatenate([c.K, as_seen(k, c.dtype)[:, :, None, :]], axis=2)
    c.V = np.concatenate([c.V, as_seen(v, c.dtype)[:, :, None, :]], axis=2)
    c.zones.append()
    c.appended += 1


def oracle_encoding(c: Case, seq: int, kvh: int) -> dict:
    S, N = c.cfg["sink"], c.zones.N
    return o.encode_contract(c.K[seq, kvh, S:S + N], c.signs, 16, LEV32, THR32,
                             None if c.table is None else c.table[kvh])


def check_state(c: Case):
    st = c.ctx.paris_get_state()
    z = c.zones
    assert (st["T"], st["N"], st["n_local"], st["n_buf"]) == (z.T, z.N, z.n_local, z.n_buf)


def check_encoding(c: Case, rows=None):
    """ids, codes and w of the Retrieval zone, bit for bit."""
    check_state(c)
    for seq in range(c.cfg["batch"]):
        for kvh in range(c.cfg["n_kv_heads"]):
            enc = oracle_encoding(c, seq, kvh)
            ids = c.ctx.paris_debug_dump(P.DUMP_IDS, seq, kvh)
            codes = c.ctx.paris_debug_dump(P.DUMP_CODES, seq, kvh)
            w = c.ctx.paris_debug_dump(P.DUMP_W, seq, kvh)
            sel = slice(None) if rows is None else rows
            np.testing.assert_array_equal(ids[sel], enc["ids"][sel])
            np.testing.assert_array_equal(codes[sel], o.pack_codes(enc["nib"])[sel])
            np.testing.assert_array_equal(w[sel].view(np.uint32), enc["w"][sel].view(np.uint32))


def queries_from_zone(c: Case, sigma=0.5, step=0) -> np.ndarray:
    """float32 [batch, Hq, d]: a random Retrieval-zone key of each query's KV head plus noise."""
    b, hq = c.cfg["batch"], c.cfg["n_q_heads"]
    S, N = c.cfg["sink"], c.zones.N
    lo, hi = (S, S + N) if N > 0 else (0, max(1, c.zones.T))
    pos = synth.query_positions(c.seed, b, hq, lo, hi, step)
    picked = np.stack([np.stack([c.K[s, h // c.G, pos[s, h]] for h in range(hq)]) for s in range(b)])
    return synth.queries_from_keys(c.seed, picked, sigma, step)


def run_retrieve(c: Case, q: np.ndarray):
    b, hq, k = c.cfg["batch"], c.cfg["n_q_heads"], c.cfg["topk"]
    qd = to_dev(q, c.dtype)
    idx = torch.full((b, hq, k), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((b, hq, k), 7.0, dtype=torch.float32, device="cuda")
    k_eff = c.ctx.paris_retrieve(qd, idx, sc)
    torch.cuda.synchronize()
    return qd, idx, sc, k_eff


def check_retrieve(c: Case, q: np.ndarray, heads=None, stages=True):
    """Votes, candidates, estimates and the top-k of every (or the listed)
    (sequence, query head) against the oracle.  Returns the device outputs."""
    qd, idx, sc, k_eff = run_retrieve(c, q)
    q_seen = as_seen(q, c.dtype)
    S, N = c.cfg["sink"], c.zones.N
    k = c.cfg["topk"]
    weighting = "flat" if c.cfg["vote_weighting"] == P.PARIS_VOTE_FLAT else "rank"
    idx_h, sc_h = idx.cpu().numpy(), sc.cpu().numpy()
    if N == 0:
        assert k_eff == 0
        assert np.all(idx_h == -1) and np.all(np.isneginf(sc_h))
        return qd, idx, k_eff
    encs = {}
    heads = heads if heads is not None else [(s, h) for s in range(c.cfg["batch"]) for h in range(c.cfg["n_q_heads"])]
    for seq, qh in heads:
        kvh = qh // c.G
        if (seq, kvh) not in encs:
            e = oracle_encoding(c, seq, kvh)
            encs[(seq, kvh)] = e
        r = o.retrieve_contract(encs[(seq, kvh)], q_seen[seq, qh], c.signs, 16, c.cfg["rho"], c.cfg["cand_bp"],
                                k, LEV32, weighting, None if c.table is None else c.table[kvh])
        assert k_eff == r["k_eff"]
        if stages:
            qt = c.ctx.paris_debug_dump(P.DUMP_QT, seq, qh)
            np.testing.assert_array_equal(qt.view(np.uint32), r["qp"]["qt"].view(np.uint32))
            qn = c.ctx.paris_debug_dump(P.DUMP_QNORM, seq, qh)
            assert qn[0] == r["qp"]["qnorm"]
            hot = c.ctx.paris_debug_dump(P.DUMP_HOT, seq, qh)
            np.testing.assert_array_equal(hot & 0xFFFF, r["qp"]["hot_ids"])
            np.testing.assert_array_equal(hot >> 16, r["qp"]["hot_w"])
            votes = c.ctx.paris_debug_dump(P.DUMP_VOTES, seq, qh)
            np.testing.assert_array_equal(votes.astype(np.int64), r["votes"])
            cands = c.ctx.paris_debug_dump(P.DUMP_CANDS, seq, qh)
            np.testing.assert_array_equal(cands, S + r["cand"])
            est = c.ctx.paris_debug_dump(P.DUMP_CAND_EST, seq, qh)
            np.testing.assert_allclose(est, r["est"], rtol=SCORE_RTOL, atol=1e-30)
            assert np.array_equal(est.view(np.uint32), r["est"].view(np.uint32)), "estimates not bit-identical"
        top_idx, top_est = r["top_idx"], r["top_est"]
        if c.cfg.get("topk_order") == P.PARIS_TOPK_BY_POSITION:  # the same set in ascending position
            perm = np.argsort(top_idx, kind="stable")
            top_idx, top_est = top_idx[perm], top_est[perm]
        np.testing.assert_array_equal(idx_h[seq, qh, :k_eff], S + top_idx)
        np.testing.assert_allclose(sc_h[seq, qh, :k_eff], top_est, rtol=SCORE_RTOL, atol=1e-30)
        assert np.all(idx_h[seq, qh, k_eff:] == -1)
        assert np.all(np.isneginf(sc_h[seq, qh, k_eff:]))
    return qd, idx, k_eff


def check_attention(c: Case, qd: torch.Tensor, idx: torch.Tensor, k_eff: int, heads=None):
    b, hq, d = c.cfg["batch"], c.cfg["n_q_heads"], c.cfg["head_dim"]
    out = torch.zeros((b, hq, d), dtype=torch.bfloat16, device="cuda")
    c.ctx.paris_sparse_attend(qd, idx, out)
    c.ctx.paris_check_device()
    out_h = out.float().cpu().numpy()
    q_seen = qd.float().cpu().numpy()
    idx_h = idx.cpu().numpy()
    Kb = as_seen(c.K, torch.bfloat16)
    Vb = as_seen(c.V, torch.bfloat16)
    z = c.zones
    heads = heads if heads is not None else [(s, h) for s in range(b) for h in range(hq)]
    worst = 0.0
    for seq, qh in heads:
        kvh = qh // c.G
        top = idx_h[seq, qh, :k_eff]
        rows = np.concatenate([z.sink(), z.local(), z.buffer(), top]).astype(np.int64)
        assert len(np.unique(rows)) == len(rows)
        ref = o.attention(q_seen[seq, qh], Kb[seq, kvh, rows], Vb[seq, kvh, rows])
        err = np.max(np.abs(out_h[seq, qh] - ref))
        worst = max(worst, err)
        assert err <= ATTN_ATOL, (seq, qh, err)
    return worst


def assert_score_order(idx: np.ndarray, sc: np.ndarray, k_eff: int):
    """Each top-k list (last axis) is listed by (estimate desc, position asc)
    over its first k_eff entries: the order the top-k contract fixes."""
    dk = np.diff(sc[..., :k_eff].astype(np.float64), axis=-1)
    di = np.diff(idx[..., :k_eff].astype(np.int64), axis=-1)
    assert np.all((dk < 0) | ((dk == 0) & (di > 0)))
