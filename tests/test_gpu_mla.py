"""Sparse MLA decode (MQA form, tensor cores) through the C ABI vs the fp64 oracle.

The kernel rounds each dequantised latent value (code x scale) and each softmax weight to
bf16 for the MMA and accumulates in fp32; the oracle uses the exact values. Graded per
query on every head: max |out - ref| <= 2e-2, mean <= 2e-3, and ||out - ref|| / ||ref||
<= 2e-2 (bf16 rounding of the operands is about 2^-9 relative); lse within 2e-2.
"""

import numpy as np
import pytest
import torch

import oracle as O
from indexer_driven_sparse_gb300 import binding as qb
from indexer_driven_sparse_gb300 import inputs as I
from parity import bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(w, n_tokens=None):
    B, H = w.q.shape[0], w.q.shape[1]
    q, kv, rows, n_rows = (t.to(DEV) for t in (w.q, w.kv, w.rows, w.n_rows))
    if n_tokens is not None:
        kv = kv[:n_tokens]
    ws = qb.sparse_mla_workspace(H, B, rows.shape[1])
    out = torch.full((B, H, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=DEV)
    qb.qsa_sparse_mla_decode(q, kv, rows, n_rows, out, lse, ws)
    return out, lse, qb.qsa_read_device_status(ws)


def _check(w, out, lse, queries=None, skip=None):
    qbits = bits(w.q)
    rows, n_rows = w.rows.cpu().numpy(), w.n_rows.cpu().numpy()
    out_h, lse_h = out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)
    worst = 0.0
    for b in (range(len(n_rows)) if queries is None else queries):
        sel = rows[b, :n_rows[b]]
        if skip is not None:
            sel = sel[sel != skip]
        # the oracle decodes only this query's rows (the cache may hold a million)
        sub = w.kv[torch.as_tensor(sel, dtype=torch.long, device=w.kv.device)].cpu().numpy()
        latent, rope = O.mla_rows_from_bytes(sub)
        ref, ref_lse = O.sparse_mla_attend(qbits[b], latent, rope, np.arange(sel.size))
        if sel.size == 0:
            assert not out_h[b].any() and np.all(np.isneginf(lse_h[b])), b
            continue
        err = np.abs(out_h[b] - ref)
        rel = np.linalg.norm(out_h[b] - ref) / np.linalg.norm(ref)
        assert np.all(np.isfinite(out_h[b])), b
        assert err.max() <= 2e-2 and err.mean() <= 2e-3, (b, err.max(), err.mean())
        assert rel <= 2e-2, (b, rel)
        assert np.max(np.abs(lse_h[b] - ref_lse)) <= 2e-2, b
        worst = max(worst, rel)
    return worst


def test_mla_ragged_batch(cuda_lib):
    # full, partial and single-row tiles, an empty query, a tile boundary +-1
    w = I.mla_workload(5000, [2048, 100, 64, 65, 1, 0, 130, 2047], 64, seed=3)
    out, lse, st = _run(w)
    assert st[0] == 0, st
    _check(w, out, lse)


@pytest.mark.parametrize("heads", [1, 16, 33, 64, 65, 128])
def test_mla_head_counts(cuda_lib, heads):
    w = I.mla_workload(3000, [300, 64, 7], heads, seed=4 + heads)
    out, lse, st = _run(w)
    assert st[0] == 0, st
    _check(w, out, lse)


def test_mla_many_short_queries(cuda_lib):
    # 300 queries of 0-200 rows at 64 heads: a CTA's run crosses many (query, half) segments
    # and query changes, with single-tile segments and empty queries among them
    g = torch.Generator().manual_seed(21)
    counts = torch.randint(0, 201, (300,), generator=g).tolist()
    counts[7] = 0
    counts[8] = 64
    counts[9] = 1
    w = I.mla_workload(20000, counts, 64, seed=21)
    out, lse, st = _run(w)
    assert st[0] == 0, st
    _check(w, out, lse)


def test_mla_invalid_row_is_skipped_and_recorded(cuda_lib):
    # the cache holds 2001 rows but the call is told 2000: id 2000 is out of range for the
    # call, yet an unchecked read of it would stay inside the buffer
    w = I.mla_workload(2001, [200, 50], 64, seed=9)
    w.rows[0, 17] = 2000
    w.rows[0, :200] = w.rows[0, :200].sort().values
    out, lse, st = _run(w, n_tokens=2000)
    assert st[0] == qb.QSA_ERR_DEVICE_BOUNDS
    _check(w, out, lse, skip=2000)


def test_mla_full_size_batch(cuda_lib):
    # 2048 selected rows per query out of a million-token FP8 cache, 64 heads
    w = I.mla_workload(1 << 20, [2048] * 8, 64, seed=11, device=DEV)
    out, lse, st = _run(w)
    assert st[0] == 0, st
    worst = _check(w, out, lse)
    assert worst < 2e-2
