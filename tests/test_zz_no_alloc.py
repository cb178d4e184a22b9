"""qsa_sparse_decode_noalloc against qsa_sparse_decode.

Some callers cannot allocate device memory at all: code that runs while a stream is
being captured in global mode (cudaMalloc is illegal there), plug-in hosts that own
every byte of device memory, and latency-critical loops that must not risk the
implicit synchronisation of an allocation. For them the library offers a decode
entry point whose scratch lives in a fixed static device array. This file checks,
through the C ABI, that it returns what the workspace-taking entry point returns on
two calls in a row (the second with different inputs, so stale scratch would show),
and that a batch too large for the static array is refused before anything runs.
It sits last in collection order and needs nothing from the other test files.
"""

import ctypes as C

import pytest
import torch

from indexer_driven_sparse_gb300 import binding as qb
from indexer_driven_sparse_gb300 import inputs as I
from indexer_driven_sparse_gb300.pipeline import DecodeBatch

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2      # the attention tolerance used by every parity test
MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def _decode_both(w):
    L = w.layers[0]
    q, k, v = L.q.cuda(), L.k_cache.cuda(), L.v_cache.cuda()
    b = DecodeBatch(w.n_q_heads, w.n_kv_heads, w.ctx_len)
    pooled = b.new_pooled()
    b.pool(L.raw_idx_k.cuda(), pooled)
    b.step(L.q_idx.cuda(), q, k, v, pooled)                       # existing entry point (caller workspace)
    assert b.device_status()[0] == 0
    out = torch.empty_like(b.out)
    lse = torch.empty_like(b.lse)
    qb.qsa_sparse_decode_noalloc(b.cfg, q, k, v, b.tok_off, b.ctx_len, b.blocks, b.count, out, lse)
    torch.cuda.synchronize()
    return b.out.float(), b.lse, out.float(), lse


def _close(ref, got, ref_lse, got_lse):
    err = (got - ref).abs()
    assert torch.isfinite(got).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
    assert (got_lse - ref_lse).abs().max().item() <= LSE_ABS


def test_noalloc_matches_workspace_decode_twice(cuda_lib):
    first = I.decode_workload("noalloc_a", [2052, 9001, 37, 70001], 1, 16, 2, "sharp", seed=21)
    second = I.decode_workload("noalloc_b", [131072, 5, 4100], 1, 16, 2, "planted", seed=22)
    for w in (first, second):
        ref, ref_lse, got, got_lse = _decode_both(w)
        _close(ref, got, ref_lse, got_lse)


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
