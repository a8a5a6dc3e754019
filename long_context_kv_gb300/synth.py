"""Seeded synthetic inputs for the ParisKV decode path.

This module is the only code shared by the oracle side and the CUDA side of
the tests and the benchmark.  It draws random numbers and nothing else: it
holds none of the method's arithmetic (no rotation, no quantisation, no
scoring).  Every array comes from a NumPy PCG64 stream keyed by
(seed, stream id), so the same call gives the same bits on x86 and on Arm.

Workload recipe (the pages evaluate on GPQA-Diamond, MATH500, AIME25,
LongBench-V2 and RULER with trained 8B models; these synthetic arrays stand in
for them):

* keys      k = g * s, g ~ N(0, 1) i.i.d., s a per-(layer, KV head, channel)
              scale drawn once from LogNormal(0, 0.5);
* values    v ~ N(0, 1);
* queries   a uniformly drawn key of the query's KV head, taken from a given
              position range (the Retrieval zone), plus N(0, 0.5^2) noise;
* drift     decode-time keys k = g * s + mu(t) with
              mu(t) = rate * (t / 256) * delta * s and delta a fixed random
              +-1 vector per KV head (ParisKV, "Problem definition":
              decoding keys drift away from the prefill distribution);
* SRHT signs  the random diagonal D of the shared rotation, +-1 per
              coordinate, drawn here and passed to both sides as an input.
"""
from __future__ import annotations

import numpy as np

# Stream ids keep the draws of one seed independent of each other.
_S_SIGNS, _S_SCALE, _S_KEYS, _S_VALUES, _S_QPOS, _S_QNOISE, _S_DELTA, _S_DRIFT, _S_QWALK = range(9)


def _rng(seed: int, stream: int, *extra: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), stream, *map(int, extra)])))


def srht_signs(seed: int, d: int) -> np.ndarray:
    """The diagonal of D: d entries in {-1, +1}, int8."""
    bits = _rng(seed, _S_SIGNS).integers(0, 2, size=d, dtype=np.int8)
    return (1 - 2 * bits).astype(np.int8)


def channel_scale(seed: int, n_kv_heads: int, d: int, sigma: float = 0.5) -> np.ndarray:
    """Per-(KV head, channel) key scale s ~ LogNormal(0, sigma), float32 [Hkv, d]."""
    g = _rng(seed, _S_SCALE).standard_normal((n_kv_heads, d), dtype=np.float64)
    return np.exp(sigma * g).astype(np.float32)


def keys(seed: int, batch: int, n_kv_heads: int, t0: int, t1: int, d: int,
         scale: np.ndarray) -> np.ndarray:
    """Keys of token positions [t0, t1): float32 [batch, Hkv, t1 - t0, d].

    Each (sequence, KV head) has its own stream, and each position block of
    4096 tokens its own sub-stream, so any position range can be regenerated
    without drawing the ones before it.
    """
    out = np.empty((batch, n_kv_heads, t1 - t0, d), dtype=np.float32)
    for b in range(batch):
        for h in range(n_kv_heads):
            out[b, h] = key_rows(seed, b, h, t0, t1, d, scale)
    return out


def values(seed: int, batch: int, n_kv_heads: int, t0: int, t1: int, d: int) -> np.ndarray:
    """Values of token positions [t0, t1): float32 [batch, Hkv, t1 - t0, d]."""
    out = np.empty((batch, n_kv_heads, t1 - t0, d), dtype=np.float32)
    for b in range(batch):
        for h in range(n_kv_heads):
            out[b, h] = value_rows(seed, b, h, t0, t1, d)
    return out


def key_rows(seed: int, b: int, h: int, t0: int, t1: int, d: int, scale: np.ndarray) -> np.ndarray:
    """keys(...)[b, h] alone, float32 [t1 - t0, d]: the same bits, without
    drawing the other (sequence, head) pairs (long contexts, one head at a time)."""
    return _blocked_normal(seed, _S_KEYS, b, h, t0, t1, d) * scale[h][None, :]


def value_rows(seed: int, b: int, h: int, t0: int, t1: int, d: int) -> np.ndarray:
    """values(...)[b, h] alone, float32 [t1 - t0, d]."""
    return _blocked_normal(seed, _S_VALUES, b, h, t0, t1, d)


_BLOCK = 4096


def _blocked_normal(seed, stream, b, h, t0, t1, d):
    rows = []
    blk0, blk1 = t0 // _BLOCK, (t1 + _BLOCK - 1) // _BLOCK
    for blk in range(blk0, blk1):
        g = _rng(seed, stream, b, h, blk).standard_normal((_BLOCK, d), dtype=np.float32)
        lo = max(t0, blk * _BLOCK) - blk * _BLOCK
        hi = min(t1, (blk + 1) * _BLOCK) - blk * _BLOCK
        rows.append(g[lo:hi])
    if not rows:
        return np.zeros((0, d), dtype=np.float32)
    return np.concatenate(rows, axis=0)


def drift_offset(seed: int, n_kv_heads: int, d: int, scale: np.ndarray, t: int,
                 rate: float = 0.02) -> np.ndarray:
    """mu(t) = rate * (t / 256) * delta * s, float32 [Hkv, d]; t counts decode steps."""
    delta = 1.0 - 2.0 * _rng(seed, _S_DELTA).integers(0, 2, size=(n_kv_heads, d))
    return (rate * (t / 256.0) * delta * scale).astype(np.float32)


def drift_keys(seed: int, batch: int, n_kv_heads: int, step: int, d: int,
               scale: np.ndarray, rate: float = 0.02) -> np.ndarray:
    """One decode step's new keys under drift: float32 [batch, Hkv, d]."""
    g = _rng(seed, _S_DRIFT, step).standard_normal((batch, n_kv_heads, d), dtype=np.float32)
    return g * scale[None] + drift_offset(seed, n_kv_heads, d, scale, step, rate)[None]


def decode_values(seed: int, batch: int, n_kv_heads: int, step: int, d: int) -> np.ndarray:
    """One decode step's new values: float32 [batch, Hkv, d]."""
    return _rng(seed, _S_VALUES + 100, step).standard_normal((batch, n_kv_heads, d), dtype=np.float32)


def decode_keys(seed: int, batch: int, n_kv_heads: int, step: int, d: int,
                scale: np.ndarray) -> np.ndarray:
    """One decode step's new keys without drift: float32 [batch, Hkv, d]."""
    return drift_keys(seed, batch, n_kv_heads, step, d, scale, rate=0.0)


def query_positions(seed: int, batch: int, n_q_heads: int, lo: int, hi: int, step: int = 0) -> np.ndarray:
    """Uniform token positions in [lo, hi), int64 [batch, Hq]: the key each query copies."""
    if hi <= lo:
        raise ValueError("empty position range for queries")
    return _rng(seed, _S_QPOS, step).integers(lo, hi, size=(batch, n_q_heads), dtype=np.int64)


def queries_from_keys(seed: int, picked: np.ndarray, sigma: float = 0.5, step: int = 0) -> np.ndarray:
    """q = picked key + N(0, sigma^2) noise.  picked: float32 [batch, Hq, d]."""
    noise = _rng(seed, _S_QNOISE, step).standard_normal(picked.shape, dtype=np.float32)
    return (picked + np.float32(sigma) * noise).astype(np.float32)


def query_walk(seed: int, q: np.ndarray, corr: float, step: int) -> np.ndarray:
    """The next decode step's queries as a correlated walk from q (float32
    [..., d]): corr * q + sqrt(1 - corr^2) * n, with n Gaussian and each row of
    n scaled to the norm of q's row, so that cos(q, q_next) is close to corr."""
    n = _rng(seed, _S_QWALK, step).standard_normal(q.shape, dtype=np.float32)
    n *= np.linalg.norm(q, axis=-1, keepdims=True) / np.linalg.norm(n, axis=-1, keepdims=True)
    return (np.float32(corr) * q + np.float32(np.sqrt(1.0 - corr * corr)) * n).astype(np.float32)
