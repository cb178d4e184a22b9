"""qsa_sparse_decode_noalloc against qsa_sparse_decode.

Some callers cannot allocate device memory at all: a plug-in inside a host application
that owns the whole device memory pool, a process whose device memory another allocator
has fully reserved, or a latency-critical loop that must not risk the implicit
synchronisation of an allocation. For them the library offers a decode entry point whose
scratch lives in a fixed static device array. This file checks, through the C ABI, that
it returns exactly what the workspace-taking entry point returns (both run the same
kernels with the same split on the same inputs, so out and lse must be bit-identical) on
two calls in a row, the second with different inputs and batch, so a stale partial left
in the shared array by the first call would show; and that invalid calls are refused on
the host. It sits last in collection order and needs nothing from the other test files.
"""

import ctypes as C

import pytest
import torch

from indexer_driven_sparse_gb300 import binding as qb
from indexer_driven_sparse_gb300 import inputs as I
from indexer_driven_sparse_gb300.pipeline import DecodeBatch

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2      # the attention tolerance used by every parity test (secondary here)
MEAN_ABS = 2e-3


def _decode_both(w):
    L = w.layers[0]
    q, k, v = L.q.cuda(), L.k_cache.cuda(), L.v_cache.cuda()
    b = DecodeBatch(w.n_q_heads, w.n_kv_heads, w.ctx_len)
    pooled = b.new_pooled()
    b.pool(L.raw_idx_k.cuda(), pooled)
    b.step(L.q_idx.cuda(), q, k, v, pooled)                       # existing entry point (caller workspace)
    assert b.device_status()[0] == 0
    out = torch.full_like(b.out, float("nan"))
    lse = torch.full_like(b.lse, float("nan"))
    qb.qsa_sparse_decode_noalloc(b.cfg, q, k, v, b.tok_off, b.ctx_len, b.blocks, b.count, out, lse)
    torch.cuda.synchronize()
    return b.out, b.lse, out, lse


def test_noalloc_matches_workspace_decode_twice(cuda_lib):
    first = I.decode_workload("noalloc_a", [2052, 9001, 37, 70001], 1, 16, 2, "sharp", seed=21)
    second = I.decode_workload("noalloc_b", [131072, 5, 4100], 1, 16, 2, "planted", seed=22)
    for w in (first, second):
        ref, ref_lse, got, got_lse = _decode_both(w)
        assert torch.equal(got, ref) and torch.equal(got_lse, ref_lse)
        err = (got.float() - ref.float()).abs()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS


def test_noalloc_rejects_batches_beyond_its_static_scratch(cuda_lib):
    lib = qb.load()
    cfg = qb.make_config(16, 2)
    limit = 16 << 20
    b_ok = max(b for b in range(1, 64) if qb.workspace_size(qb.OP_SPARSE_DECODE, cfg, b) <= limit)
    assert b_ok == 30
    fake = 0x10000000            # never dereferenced: the size check refuses first
    st = lib.qsa_sparse_decode_noalloc(C.byref(cfg), fake, fake, fake, 100, fake, fake, b_ok + 1, fake, fake, fake,
                                       None, None)
    assert st == qb.QSA_ERR_WORKSPACE_TOO_SMALL
    assert b"16 MiB" in lib.qsa_last_error()


def test_noalloc_rejects_bad_pointers_before_enqueueing(cuda_lib):
    lib = qb.load()
    cfg = qb.make_config(16, 2)
    fake = 0x10000000
    # a NULL tensor and a misaligned one are refused by the host checks
    st = lib.qsa_sparse_decode_noalloc(C.byref(cfg), None, fake, fake, 100, fake, fake, 1, fake, fake, fake, None,
                                       None)
    assert st == qb.QSA_ERR_INVALID_ARGUMENT
    st = lib.qsa_sparse_decode_noalloc(C.byref(cfg), fake + 2, fake, fake, 100, fake, fake, 1, fake, fake, fake,
                                       None, None)
    assert st == qb.QSA_ERR_INVALID_ARGUMENT
    # host memory the device cannot read at the same address
    host = torch.zeros(4096, dtype=torch.bfloat16)
    dev = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    i32 = torch.zeros(4, dtype=torch.int32, device="cuda")
    st = lib.qsa_sparse_decode_noalloc(C.byref(cfg), dev.data_ptr(), host.data_ptr(), dev.data_ptr(), 4,
                                       i32.data_ptr(), i32.data_ptr(), 1, i32.data_ptr(), i32.data_ptr(),
                                       dev.data_ptr(), None, None)
    assert st == qb.QSA_ERR_INVALID_ARGUMENT
    # B = 0 is a no-op
    st = lib.qsa_sparse_decode_noalloc(C.byref(cfg), None, None, None, 0, None, None, 0, None, None, None, None,
                                       None)
    assert st == qb.QSA_OK
