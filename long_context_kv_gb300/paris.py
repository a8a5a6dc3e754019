"""Thin ctypes binding of the ParisKV C ABI (include/paris.h).

Argument marshalling only: tensors are passed as raw pointers
(``tensor.data_ptr()``) with the current torch CUDA stream; every step of the
retrieval path runs in the CUDA library.  There is no CPU fallback: if the
library is missing or fails to load, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libparis.so")

PARIS_OK, PARIS_EINVAL, PARIS_ENOMEM, PARIS_ECUDA, PARIS_ESTATE, PARIS_ECAPACITY, PARIS_EDEVICE = 0, -1, -2, -3, -4, -6, -7
PARIS_F32, PARIS_BF16 = 0, 1
PARIS_VOTE_RANK, PARIS_VOTE_FLAT = 0, 1
PARIS_TOPK_BY_SCORE, PARIS_TOPK_BY_POSITION = 0, 1
(DUMP_IDS, DUMP_CODES, DUMP_W, DUMP_VOTES, DUMP_CANDS, DUMP_CAND_EST, DUMP_QT, DUMP_QNORM, DUMP_HOT,
 DUMP_LEVELS, DUMP_KV, DUMP_TRACE) = range(12)

# Every function the header declares, with its ctypes signature.
_SIGNATURES = {
    "paris_create": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]),
    "paris_destroy": (None, [ctypes.c_void_p]),
    "paris_encode_prefill": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                            ctypes.c_int64, ctypes.c_void_p]),
    "paris_append_decode": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                           ctypes.c_void_p]),
    "paris_retrieve": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p]),
    "paris_sparse_attend": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_void_p]),
    "paris_get_state": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "paris_check_device": (ctypes.c_int, [ctypes.c_void_p]),
    "paris_debug_dump": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_size_t]),
    "paris_last_error": (ctypes.c_char_p, [ctypes.c_void_p]),
    "paris_rsq_levels": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "paris_sparse_attend_gqa": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p]),
    "paris_set_centroids": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "paris_dense_attend": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                          ctypes.c_void_p]),
    "paris_sparse_attend_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "paris_decode_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p]),
    "paris_launch_counts": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "paris_profile_begin": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int]),
    "paris_profile_end": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
}

KERNELS = ["place_kv", "encode", "build_index", "append", "decode", "attend", "fill", "dense", "union"]


class paris_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "batch", "n_kv_heads", "n_q_heads", "head_dim", "n_sub", "rho", "sink", "local", "update_buf",
        "topk", "cand_bp", "max_ctx", "retrieval_on_host", "vote_weighting", "topk_order")]


class paris_state(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("T", "N", "n_local", "n_buf", "C", "k_eff", "n_flushes")]


_lib = None


def load(path: str = LIB_PATH):
    """Load libparis.so (built by long_context_kv_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"ParisKV CUDA library not built: {path} is missing "
                           "(run long_context_kv_gb300.build.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class ParisError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{msg} (status {status})")
        self.status = status


def _check(st, ctx=None):
    if st != PARIS_OK:
        raise ParisError(st, load().paris_last_error(ctx).decode())


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return PARIS_F32
    if t.dtype == torch.bfloat16:
        return PARIS_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    if t.data_ptr() % 16:
        raise ValueError("tensor data must be 16-byte aligned")
    return ctypes.c_void_p(t.data_ptr())


def paris_rsq_levels(m: int):
    """The library's float64 Lloyd-Max levels (host computation, no GPU)."""
    lev = (ctypes.c_double * 8)()
    thr = (ctypes.c_double * 7)()
    _check(load().paris_rsq_levels(m, lev, thr))
    return np.array(lev[:]), np.array(thr[:])


def make_config(**kw) -> paris_config:
    cfg = paris_config()
    defaults = dict(batch=1, n_kv_heads=1, n_q_heads=1, head_dim=128, n_sub=16, rho=4, sink=0, local=0,
                    update_buf=128, topk=64, cand_bp=1000, max_ctx=4096, retrieval_on_host=0,
                    vote_weighting=PARIS_VOTE_RANK, topk_order=PARIS_TOPK_BY_SCORE)
    defaults.update(kw)
    for k, v in defaults.items():
        setattr(cfg, k, int(v))
    return cfg


class Context:
    """One layer's ParisKV cache (wraps paris_create / paris_destroy)."""

    def __init__(self, cfg: paris_config, srht_signs: np.ndarray):
        lib = load()
        self.cfg = cfg
        signs = np.ascontiguousarray(srht_signs, dtype=np.int8)
        h = ctypes.c_void_p()
        _check(lib.paris_create(ctypes.byref(cfg), signs.ctypes.data_as(ctypes.c_void_p), ctypes.byref(h)))
        self._h = h

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            load().paris_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    # -- the ABI calls, same names --------------------------------------------
    def paris_encode_prefill(self, K, V, T=None, stream=None):
        T = K.shape[2] if T is None else T
        _check(load().paris_encode_prefill(self._h, _ptr(K), _ptr(V), _dtype_code(K), T, _stream(stream)), self._h)

    def paris_append_decode(self, k, v, stream=None):
        _check(load().paris_append_decode(self._h, _ptr(k), _ptr(v), _dtype_code(k), _stream(stream)), self._h)

    def paris_retrieve(self, q, topk_idx, topk_score=None, stream=None) -> int:
        k_eff = ctypes.c_int64()
        _check(load().paris_retrieve(self._h, _ptr(q), _dtype_code(q), _ptr(topk_idx), _ptr(topk_score),
                                     ctypes.byref(k_eff), _stream(stream)), self._h)
        return k_eff.value

    def paris_sparse_attend(self, q, topk_idx, out, stream=None):
        _check(load().paris_sparse_attend(self._h, _ptr(q), _dtype_code(q), _ptr(topk_idx), _ptr(out),
                                          _stream(stream)), self._h)

    def paris_sparse_attend_gqa(self, q, topk_idx, out, stream=None):
        """Sparse attention over the window and the union of the KV head's query heads' top-k."""
        _check(load().paris_sparse_attend_gqa(self._h, _ptr(q), _dtype_code(q), _ptr(topk_idx), _ptr(out),
                                              _stream(stream)), self._h)

    def paris_set_centroids(self, centroids=None, stream=None):
        """Learned centroids, device float32 [Hkv][16][256][8] (None: the analytic sign patterns)."""
        _check(load().paris_set_centroids(self._h, _ptr(centroids) if centroids is not None else None,
                                          _stream(stream)), self._h)

    def paris_dense_attend(self, q, out, stream=None):
        """Dense attention over every cached token (the full-attention comparator)."""
        _check(load().paris_dense_attend(self._h, _ptr(q), _dtype_code(q), _ptr(out), _stream(stream)), self._h)

    def paris_sparse_attend_noalloc(self, q, topk_idx, out, stream=None):
        """paris_sparse_attend with its scratch in the library's fixed area (no allocation)."""
        _check(load().paris_sparse_attend_noalloc(self._h, _ptr(q), _dtype_code(q), _ptr(topk_idx), _ptr(out),
                                                  _stream(stream)), self._h)

    def paris_decode_step(self, k, v, q, topk_idx, topk_score, out, stream=None) -> int:
        k_eff = ctypes.c_int64()
        _check(load().paris_decode_step(self._h, _ptr(k), _ptr(v), _dtype_code(k), _ptr(q), _dtype_code(q),
                                        _ptr(topk_idx), _ptr(topk_score), _ptr(out), ctypes.byref(k_eff),
                                        _stream(stream)), self._h)
        return k_eff.value

    def paris_get_state(self) -> dict:
        st = paris_state()
        _check(load().paris_get_state(self._h, ctypes.byref(st)), self._h)
        return {n: getattr(st, n) for n, _ in paris_state._fields_}

    def paris_launch_counts(self) -> dict:
        arr = (ctypes.c_int64 * len(KERNELS))()
        _check(load().paris_launch_counts(self._h, arr), self._h)
        return dict(zip(KERNELS, arr[:]))

    def paris_profile_begin(self, max_launches: int):
        _check(load().paris_profile_begin(self._h, int(max_launches)), self._h)

    def paris_profile_end(self):
        """Returns {kernel: (total_ms, launches)} for the profiled window."""
        ms = (ctypes.c_double * len(KERNELS))()
        n = (ctypes.c_int64 * len(KERNELS))()
        _check(load().paris_profile_end(self._h, ms, n), self._h)
        return {k: (ms[i], n[i]) for i, k in enumerate(KERNELS)}

    def paris_check_device(self):
        _check(load().paris_check_device(self._h), self._h)

    def paris_debug_dump(self, what: int, seq: int = 0, head: int = 0):
        st = self.paris_get_state()
        N, C, T = st["N"], st["C"], st["T"]
        d, B, rho = self.cfg.head_dim, self.cfg.n_sub, self.cfg.rho
        shapes = {
            DUMP_IDS: ((N, B), np.uint8), DUMP_CODES: ((N, d // 2), np.uint8), DUMP_W: ((N, B), np.float32),
            DUMP_VOTES: ((N,), np.uint8), DUMP_CANDS: ((C,), np.int32), DUMP_CAND_EST: ((C,), np.float32),
            DUMP_QT: ((d,), np.float32), DUMP_QNORM: ((1,), np.float32), DUMP_HOT: ((B, rho), np.uint32),
            DUMP_LEVELS: ((15,), np.float32), DUMP_KV: ((2, T, d), np.uint16),
            DUMP_TRACE: ((64 + 8 * 4096 * 4,), np.uint64),
        }
        shape, dt = shapes[what]
        out = np.zeros(shape, dtype=dt)
        _check(load().paris_debug_dump(self._h, what, seq, head, out.ctypes.data_as(ctypes.c_void_p),
                                       out.nbytes), self._h)
        return out
