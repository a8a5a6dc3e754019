"""paris_create when an allocation fails: the device's memory, or pinned host
memory for a Retrieval zone offloaded through UVA, cannot hold the cache.
The call returns PARIS_ENOMEM with *out == NULL, frees whatever it had
already allocated (the device's free memory is the same before and after),
and the library stays usable.  Nothing is faulted: the failing calls are
cudaMalloc / cudaHostAlloc asked for more than exists, which return an
error code (ParisKV, system level: the zones live in HBM, the offloaded
Retrieval zone in pinned host memory)."""
import ctypes

import numpy as np
import pytest
import torch

from long_context_kv_gb300 import paris as P
from long_context_kv_gb300 import synth

pytestmark = pytest.mark.gpu

# driver bookkeeping may move the device's free-memory figure by a page or so
FREE_SLACK = 4 << 20


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_context_kv_gb300 import build
    build.build()
    P.load()


def _create(**kw):
    lib = P.load()
    cfg = P.make_config(**kw)
    signs = np.ascontiguousarray(synth.srht_signs(1, 128), dtype=np.int8)
    out = ctypes.c_void_p(12345)  # must be overwritten with NULL on failure
    st = lib.paris_create(ctypes.byref(cfg), signs.ctypes.data_as(ctypes.c_void_p), ctypes.byref(out))
    return st, out, lib.paris_last_error(None).decode()


def _free():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def _warm():
    # one small context first, so the runtime's own first-use allocations are behind us
    st, out, _ = _create(max_ctx=4096)
    assert st == P.PARIS_OK and out.value
    P.load().paris_destroy(out)


def test_device_tables_larger_than_the_device_give_enomem_and_leave_nothing():
    _warm()
    free0 = _free()
    # 2^18 (sequence, KV head) pairs x 4M tokens: the window (64 MB) is
    # allocated, the Retrieval K store (about 280 TB) is not
    st, out, err = _create(batch=4096, n_kv_heads=64, n_q_heads=64, sink=0, local=0, update_buf=1, topk=64,
                           cand_bp=500, max_ctx=(1 << 22) - 1)
    assert st == P.PARIS_ENOMEM, err
    assert out.value is None
    assert "cudaMalloc" in err
    assert abs(_free() - free0) <= FREE_SLACK
    _warm()


def test_pinned_host_store_larger_than_the_host_gives_enomem_and_leaves_nothing():
    _warm()
    free0 = _free()
    # 2^26 pairs: the two window tables (16 GB each) are allocated on the
    # device, the pinned host store (2^57 bytes) cannot be mapped at all
    st, out, err = _create(batch=65536, n_kv_heads=1024, n_q_heads=1024, sink=0, local=0, update_buf=1, topk=64,
                           cand_bp=500, max_ctx=(1 << 22) - 1, retrieval_on_host=1)
    assert st == P.PARIS_ENOMEM, err
    assert out.value is None
    assert "cudaHostAlloc" in err
    assert abs(_free() - free0) <= FREE_SLACK
    _warm()
