"""The VRAM row cache in front of host-resident K/V (qsa_decode_step_rowcache).

A hit returns the bytes the host holds, so every output must equal the cache-free fused step
bit for bit, whatever the cache holds; and every filled slot must hold exactly its tagged
token's K and V rows. Cases: a cold cache (all misses), a warm one (all hits), selections that
move between steps, a cache small enough that tokens collide on slots, and a re-initialised
cache after host rows change.
"""

import numpy as np
import pytest
import torch

from indexer_driven_sparse_gb300 import binding as qb
from indexer_driven_sparse_gb300 import inputs as I
from indexer_driven_sparse_gb300.pipeline import DecodeBatch

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _setup(ctx, seed, hq=16, hkv=2):
    w = I.decode_workload("rowcache", ctx, 1, hq, hkv, "planted_sharp", seed=seed)
    L = w.layers[0]
    host = [t.pin_memory() for t in (L.raw_idx_k, L.k_cache, L.v_cache)]
    q_idx, q = L.q_idx.to(DEV), L.q.to(DEV)
    b = DecodeBatch(hq, hkv, w.ctx_len)
    pooled = b.new_pooled()
    b.pool(host[0].to(DEV), pooled)
    torch.cuda.synchronize()
    return w, b, pooled, host, q_idx, q


def _reference(b, pooled, host, q_idx, q):
    b.fused_step(host[0], pooled, q_idx, q, host[1], host[2])
    torch.cuda.synchronize()
    assert b.fused_status()[0] == 0
    return b.blocks.clone(), b.count.clone(), b.out.clone(), b.lse.clone()


def _cached(b, pooled, host, q_idx, q, cache, n_slots, epoch):
    b.out.zero_()
    b.blocks.fill_(-7)
    b.fused_step_rowcache(host[0], pooled, q_idx, q, host[1], host[2], cache, n_slots, epoch)
    torch.cuda.synchronize()
    assert b.fused_status()[0] == 0
    return b.blocks.clone(), b.count.clone(), b.out.clone(), b.lse.clone()


def _check_equal(got, want):
    for g, x in zip(got, want):
        assert torch.equal(g, x)


def _cache_view(cache, n_slots, hkv=2):
    row_bytes = 2 * hkv * 256 * 2
    raw = cache.cpu().numpy()
    rows = raw[: n_slots * row_bytes].view(np.uint16).reshape(n_slots, 2, hkv, 256)
    tag = raw[n_slots * row_bytes: n_slots * (row_bytes + 8)].view(np.int64)
    hit_off = n_slots * (row_bytes + 8)
    hit = raw[hit_off: hit_off + 4 * n_slots].view(np.uint32)
    return rows, tag, hit


def _check_consistent(cache, n_slots, host, w):
    """Every filled slot holds its tagged token's K and V rows, the token belongs to the
    sequence owning the slot and sits at the slot its index maps to, inside a complete block."""
    rows, tag, _ = _cache_view(cache, n_slots)
    k = host[1].view(torch.int16).numpy().view(np.uint16)
    v = host[2].view(torch.int16).numpy().view(np.uint16)
    off, B = w.tok_off, w.batch
    filled = np.flatnonzero(tag >= 0)
    for slot in filled:
        t = int(tag[slot])
        s = max(i for i in range(B) if off[i] <= t)
        lo, hi = s * n_slots // B, (s + 1) * n_slots // B
        assert lo <= slot < hi
        tk = t - off[s]
        assert slot == lo + tk % (hi - lo)
        assert tk < 4 * (w.ctx_len[s] // 4)                      # a complete block, never the tail
        assert np.array_equal(rows[slot, 0], k[t]) and np.array_equal(rows[slot, 1], v[t])
    return filled.size


def test_rowcache_cold_then_warm_is_bit_exact(cuda_lib):
    w, b, pooled, host, q_idx, q = _setup([70001, 2052, 9001, 3], seed=81)
    want = _reference(b, pooled, host, q_idx, q)
    n_slots = 4 * 4096
    cache = qb.rowcache_new(b.cfg, n_slots)
    _check_equal(_cached(b, pooled, host, q_idx, q, cache, n_slots, 1), want)     # all misses
    n1 = _check_consistent(cache, n_slots, host, w)
    assert n1 > 3000
    _check_equal(_cached(b, pooled, host, q_idx, q, cache, n_slots, 2), want)     # all hits
    _, tag, hit = _cache_view(cache, n_slots)
    assert (hit == 2).sum() == n1 and _check_consistent(cache, n_slots, host, w) == n1


def test_rowcache_moving_selection_and_collisions(cuda_lib):
    # the indexer query drifts between steps (the selection changes partly), and a small cache
    # makes tokens of the same step collide on slots
    w, b, pooled, host, q_idx, q = _setup([40000, 9001], seed=82)
    g = torch.Generator(device="cpu").manual_seed(5)
    for n_slots in (2 * 3001, 2 * 37):
        cache = qb.rowcache_new(b.cfg, n_slots)
        qi = q_idx.clone()
        for epoch in range(1, 7):
            want = _reference(b, pooled, host, qi, q)
            _check_equal(_cached(b, pooled, host, qi, q, cache, n_slots, epoch), want)
            _check_consistent(cache, n_slots, host, w)
            qi = (qi.float() + 0.15 * torch.randn(qi.shape, generator=g).to(DEV)).to(torch.bfloat16)


def test_rowcache_reinit_after_host_rows_change(cuda_lib):
    w, b, pooled, host, q_idx, q = _setup([20000], seed=83)
    n_slots = 8192
    cache = qb.rowcache_new(b.cfg, n_slots)
    _cached(b, pooled, host, q_idx, q, cache, n_slots, 1)
    # the host rows change (another request in the same K/V slots): empty the cache first
    host[1].mul_(-1)
    host[2].add_(1)
    qb.qsa_rowcache_init(b.cfg, cache, n_slots)
    want = _reference(b, pooled, host, q_idx, q)
    _check_equal(_cached(b, pooled, host, q_idx, q, cache, n_slots, 2), want)
    _check_consistent(cache, n_slots, host, w)


def test_rowcache_rejects_bad_arguments(cuda_lib):
    w, b, pooled, host, q_idx, q = _setup([5000, 6000], seed=84)
    cache = qb.rowcache_new(b.cfg, 64)
    for n_slots, epoch, code in ((1, 1, qb.QSA_ERR_INVALID_ARGUMENT),    # fewer slots than sequences
                                 (64, 0, qb.QSA_ERR_INVALID_ARGUMENT),   # epoch 0
                                 (65, 1, qb.QSA_ERR_WORKSPACE_TOO_SMALL)):
        with pytest.raises(qb.QsaError) as e:
            b.fused_step_rowcache(host[0], pooled, q_idx, q, host[1], host[2], cache, n_slots, epoch)
        assert e.value.status == code


def test_rowcache_batched_sequences(cuda_lib):
    # 32 ragged sequences share the cache (each its own share of the slots); two steps
    w, b, pooled, host, q_idx, q = _setup(I.batched_ctx_lens(seed=3), seed=85, hq=8)
    n_slots = 32 * 1024
    cache = qb.rowcache_new(b.cfg, n_slots)
    want = _reference(b, pooled, host, q_idx, q)
    for epoch in (1, 2):
        _check_equal(_cached(b, pooled, host, q_idx, q, cache, n_slots, epoch), want)
    # a CTA caches the rows of its last two 32-token chunks (here a CTA attends several hundred
    # tokens), and the second step hits every slot the first filled
    _, tag, hit = _cache_view(cache, n_slots)
    assert (hit == 2).sum() == (tag >= 0).sum() > 32 * 40
    _check_consistent(cache, n_slots, host, w)
