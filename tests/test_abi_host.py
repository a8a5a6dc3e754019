"""C-ABI library, host side only (no GPU): it builds for sm_103a, loads,
exports every function include/paris.h declares, computes the same RSQ-IP
levels as the oracle, and rejects bad configurations before touching CUDA."""
import ctypes
import os
import re

import numpy as np
import pytest

from long_context_kv_gb300 import build as B
from long_context_kv_gb300 import paris as P
from oracle import pariskv as o

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "paris.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return P.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(paris_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("paris_create", "paris_destroy", "paris_encode_prefill", "paris_append_decode",
                 "paris_retrieve", "paris_sparse_attend", "paris_debug_dump", "paris_last_error"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in P._SIGNATURES, f"binding lacks {name}"


def test_rsq_levels_match_oracle_bitwise(lib):
    for m in (3, 4, 8, 16):
        lev, thr = P.paris_rsq_levels(m)
        ol, ot = o.rsq_levels(m)
        np.testing.assert_allclose(lev, ol, rtol=0, atol=1e-13)
        np.testing.assert_allclose(thr, ot, rtol=0, atol=1e-13)
        np.testing.assert_array_equal(lev.astype(np.float32), ol.astype(np.float32))
        np.testing.assert_array_equal(thr.astype(np.float32), ot.astype(np.float32))


@pytest.mark.parametrize("bad", [
    dict(head_dim=64), dict(n_sub=32), dict(rho=0), dict(rho=16), dict(n_q_heads=3, n_kv_heads=2),
    dict(cand_bp=0), dict(cand_bp=10001), dict(topk=0), dict(update_buf=0), dict(vote_weighting=7),
    dict(batch=0), dict(sink=-1), dict(max_ctx=-5), dict(topk_order=2), dict(topk=16385),
])
def test_create_rejects_bad_config(lib, bad):
    cfg = P.make_config(**bad)
    signs = np.ones(128, dtype=np.int8)
    h = ctypes.c_void_p()
    st = lib.paris_create(ctypes.byref(cfg), signs.ctypes.data_as(ctypes.c_void_p), ctypes.byref(h))
    assert st == P.PARIS_EINVAL
    assert h.value is None
    assert lib.paris_last_error(None).decode()


def test_create_rejects_bad_signs(lib):
    cfg = P.make_config()
    signs = np.ones(128, dtype=np.int8)
    signs[5] = 0
    h = ctypes.c_void_p()
    assert lib.paris_create(ctypes.byref(cfg), signs.ctypes.data_as(ctypes.c_void_p), ctypes.byref(h)) == P.PARIS_EINVAL
    assert "srht_signs" in lib.paris_last_error(None).decode()


def test_null_context_calls_fail_cleanly(lib):
    k = ctypes.c_int64()
    assert lib.paris_retrieve(None, None, 0, None, None, ctypes.byref(k), None) == P.PARIS_EINVAL
    assert lib.paris_append_decode(None, None, None, 0, None) == P.PARIS_EINVAL
    lib.paris_destroy(None)


def _header_nocomments():
    return re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)


def test_binding_structs_and_enums_match_the_header():
    src = _header_nocomments()
    body = re.search(r"typedef struct \{(.*?)\} paris_config;", src, flags=re.S).group(1)
    fields = re.findall(r"\bint\s+([a-z_0-9]+);", body)
    assert fields == [n for n, _ in P.paris_config._fields_]
    enum = dict((k, int(v)) for k, v in re.findall(r"\b(PARIS_[A-Z_0-9]+)\s*=\s*(\d+)", src))
    assert (enum["PARIS_TOPK_BY_SCORE"], enum["PARIS_TOPK_BY_POSITION"]) == (P.PARIS_TOPK_BY_SCORE,
                                                                              P.PARIS_TOPK_BY_POSITION)
    assert (enum["PARIS_VOTE_RANK"], enum["PARIS_VOTE_FLAT"]) == (P.PARIS_VOTE_RANK, P.PARIS_VOTE_FLAT)
    assert enum["PARIS_KERNEL_COUNT"] == len(P.KERNELS)
    for name, i in enum.items():
        if name.startswith("PARIS_KERNEL_") and name != "PARIS_KERNEL_COUNT":
            assert P.KERNELS[i] == name[len("PARIS_KERNEL_"):].lower(), name
    assert P.make_config().topk_order == P.PARIS_TOPK_BY_SCORE  # the contract's order is the default
