"""The fused decode layer-step (qsa_decode_step) against the separate calls and the oracle.

The fused kernel scores with the same fp32 arithmetic as qsa_index_score, so its
selection must equal the separate path's exactly; its attention is graded against the
oracle on that selection.
"""

import numpy as np
import pytest
import torch

import oracle as O
from indexer_driven_sparse_gb300 import binding as qb
from indexer_driven_sparse_gb300 import inputs as I
from indexer_driven_sparse_gb300.pipeline import DecodeBatch
from parity import bits, check_attention, check_lse, check_selection

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _to(layer):
    return I.Layer(*(getattr(layer, f).to(DEV) for f in ("raw_idx_k", "q_idx", "q", "k_cache", "v_cache")))


def _host(layer):
    return I.Layer(*(getattr(layer, f).cpu() for f in ("raw_idx_k", "q_idx", "q", "k_cache", "v_cache")))


def _run_both(w, corrupt_newest=False):
    L = _to(w.layers[0])
    b = DecodeBatch(w.n_q_heads, w.n_kv_heads, w.ctx_len)
    pooled = b.new_pooled()
    b.pool(L.raw_idx_k, pooled)
    b.step(L.q_idx, L.q, L.k_cache, L.v_cache, pooled)
    assert b.device_status()[0] == 0
    sep = (b.blocks.clone(), b.count.clone(), b.out.clone(), b.lse.clone())
    want_pooled = pooled.clone()
    if corrupt_newest:
        for s, p in enumerate(w.ctx_len):
            if p >= 4:
                pooled[b.blk_off[s].item() + p // 4 - 1] = 7.0
    b.blocks.fill_(-7)
    b.out.zero_()
    b.fused_step(L.raw_idx_k, pooled, L.q_idx, L.q, L.k_cache, L.v_cache)
    st = b.fused_status()
    assert st[0] == 0, st
    assert torch.equal(pooled, want_pooled)
    return b, sep, pooled


def _check(w, b, sep, pooled, rows=None, max_fp32_swaps=0):
    """The fused step's selection equals the separate calls' bit for bit; both paths' outputs
    are graded against the oracle on that selection (absolute, relative and lse rules)."""
    blocks_sep, count_sep, out_sep, lse_sep = sep
    assert torch.equal(b.count, count_sep)
    assert torch.equal(b.blocks, blocks_sep), "fused selection differs from the separate path"
    Lh = w.layers[0]
    rb, qib, qbits = bits(Lh.raw_idx_k), bits(Lh.q_idx), bits(Lh.q)
    kb, vb = bits(Lh.k_cache), bits(Lh.v_cache)
    blocks, count, out, lse = b.blocks.cpu().numpy(), b.count.cpu().numpy(), b.out.cpu(), b.lse.cpu().numpy()
    out_s, lse_s = out_sep.cpu(), lse_sep.cpu().numpy()
    off = w.tok_off
    stats = dict(band=0, fp32=0, rel=0.0, rel_sep=0.0, lse=0.0, rows=0)
    for s in (range(w.batch) if rows is None else rows):
        p = w.ctx_len[s]
        pk = O.pool_keys(rb[off[s]:off[s + 1]])
        n_band, n_fp32 = check_selection(blocks[s], count[s], qib[s], pk, p // 4)
        stats["band"] += n_band
        stats["fp32"] += n_fp32
        ref = O.decode_query(p, qib[s], pk, qbits[s], kb[off[s]:off[s + 1]], vb[off[s]:off[s + 1]], w.n_kv_heads,
                             sel=blocks[s, :count[s]])
        stats["rel"] = max(stats["rel"], check_attention(out[s], ref["out"])[2])
        stats["rel_sep"] = max(stats["rel_sep"], check_attention(out_s[s], ref["out"])[2])
        stats["lse"] = max(stats["lse"], check_lse(lse[s], ref["lse"]), check_lse(lse_s[s], ref["lse"]))
        stats["rows"] += 1
    print(f"{w.name}: {stats}")
    assert stats["fp32"] <= max_fp32_swaps, stats
    return stats


@pytest.mark.parametrize("case", ["tiny", "tiny_sharp", "planted_ragged", "batched_short", "dense_only",
                                  "sharp16_2052", "sharp16_9001", "sharp16_131072", "sharp16_ragged"])
def test_fused_step_small(cuda_lib, case):
    if case.startswith("sharp16_") and case != "sharp16_ragged":
        # 16 query / 2 KV heads (the headline kernel instance) in the sparse regime, N(0,1) Q/K/V
        p = int(case.split("_")[1])
        w = I.decode_workload(case, [p], 1, 16, 2, "sharp", seed=40 + p % 11)
    elif case == "sharp16_ragged":
        w = I.decode_workload(case, [2052, 70001, 9001, 4, 2051, 33333], 1, 16, 2, "planted_sharp", seed=41)
    elif case == "tiny":
        w = I.tiny_decode()
    elif case == "tiny_sharp":
        w = I.tiny_decode(kind="sharp", seed=3)
    elif case == "planted_ragged":
        w = I.decode_workload("planted_ragged", [5000, 2052, 70001, 4, 12345, 0, 3], 1, 16, 2, "planted", seed=4)
    elif case == "batched_short":
        w = I.decode_workload("batched_short", I.batched_ctx_lens(short_draw=True), 1, 8, 2, "gaussian", seed=0)
    else:
        w = I.decode_workload("dense_only", [0, 1, 7, 2047, 2051], 1, 16, 2, "sharp", seed=5)
    b, sep, pooled = _run_both(w, corrupt_newest=True)
    _check(w, b, sep, pooled)


def test_fused_step_repeatable(cuda_lib):
    w = I.decode_workload("rep", [40000, 9000], 1, 16, 2, "planted", seed=7)
    b, sep, pooled = _run_both(w)
    L = _to(w.layers[0])
    outs = []
    for _ in range(3):
        b.fused_step(L.raw_idx_k, pooled, L.q_idx, L.q, L.k_cache, L.v_cache)
        outs.append((b.blocks.clone(), b.out.clone(), b.lse.clone()))
    assert b.fused_status()[0] == 0
    for o in outs[1:]:
        assert all(torch.equal(x, y) for x, y in zip(o, outs[0]))


def test_fused_step_all_equal_scores(cuda_lib):
    # every score ties (zero indexer query): the lowest 512 block ids win; 50,000 candidates
    w = I.decode_workload("ties", [200003], 1, 16, 2, "gaussian", seed=8)
    w.layers[0].q_idx.zero_()
    b, sep, pooled = _run_both(w)
    assert torch.equal(b.blocks[0].cpu(), torch.arange(512, dtype=torch.int32))
    _check(w, b, sep, pooled)


@pytest.mark.parametrize("kind", ["planted", "planted_sharp"])
def test_fused_step_long_and_million_one_layer(cuda_lib, kind):
    for w in (I.long_decode(n_layers=1, kind=kind), I.million_decode(n_layers=1, kind=kind)):
        b, sep, pooled = _run_both(w)
        w.layers = [_host(w.layers[0])]
        _check(w, b, sep, pooled)
        del b, sep, pooled
        torch.cuda.empty_cache()


@pytest.mark.parametrize("kind", ["gaussian", "sharp"])
def test_fused_step_batched_full_size_one_layer(cuda_lib, kind):
    # the batched workload (32 ragged sequences, 8 query / 2 KV heads): every row graded
    w = I.batched_decode(n_layers=1, kind=kind)
    b, sep, pooled = _run_both(w)
    w.layers = [_host(w.layers[0])]
    st = _check(w, b, sep, pooled)
    assert st["rows"] == 32


def test_fused_step_prefetch_hint_changes_nothing(cuda_lib):
    # qsa_decode_step_prefetch: the L2 prefetch of another buffer (here a second layer's
    # pooled keys, and a misaligned-length view) leaves selection, out and lse bit-identical
    w = I.decode_workload("pf", [200003, 9001, 2051], 2, 16, 2, "planted", seed=12)
    L0, L1 = _to(w.layers[0]), _to(w.layers[1])
    b = DecodeBatch(16, 2, w.ctx_len)
    p0, p1 = b.new_pooled(), b.new_pooled()
    b.pool(L0.raw_idx_k, p0)
    b.pool(L1.raw_idx_k, p1)
    b.fused_step(L0.raw_idx_k, p0, L0.q_idx, L0.q, L0.k_cache, L0.v_cache)
    assert b.fused_status()[0] == 0
    want = (b.blocks.clone(), b.count.clone(), b.out.clone(), b.lse.clone())
    for nxt in (p1, p1.view(-1)[:1001], L1.k_cache):
        b.blocks.fill_(-7)
        b.out.zero_()
        b.fused_step(L0.raw_idx_k, p0, L0.q_idx, L0.q, L0.k_cache, L0.v_cache, next_read=nxt)
        assert b.fused_status()[0] == 0
        assert all(torch.equal(x, y) for x, y in zip((b.blocks, b.count, b.out, b.lse), want))
    with pytest.raises(qb.QsaError) as e:
        b.fused_step(L0.raw_idx_k, p0, L0.q_idx, L0.q, L0.k_cache, L0.v_cache, next_read=p1.view(-1)[1:])
    assert e.value.status == qb.QSA_ERR_INVALID_ARGUMENT


def test_fused_step_alternating_paths_share_barrier_state(cuda_lib):
    # Rows keep barrier counters across launches. Tied scores overflow the published
    # top-K and take the fallback (four row barriers); spread scores take the common
    # path (two). Alternating them on one workspace must keep every launch exact.
    w = I.decode_workload("alt", [200003], 1, 16, 2, "planted", seed=10)
    L = _to(w.layers[0])
    b = DecodeBatch(16, 2, w.ctx_len)
    pooled = b.new_pooled()
    b.pool(L.raw_idx_k, pooled)
    zero_q = torch.zeros_like(L.q_idx)
    want = {}
    for name, qi in (("spread", L.q_idx), ("tied", zero_q)):
        b.step(qi, L.q, L.k_cache, L.v_cache, pooled)
        want[name] = (b.blocks.clone(), b.out.clone())
    assert torch.equal(want["tied"][0][0].cpu(), torch.arange(512, dtype=torch.int32))
    for name in ("tied", "spread", "spread", "tied", "spread", "tied", "tied", "spread"):
        qi = zero_q if name == "tied" else L.q_idx
        b.fused_step(L.raw_idx_k, pooled, qi, L.q, L.k_cache, L.v_cache)
        assert b.fused_status()[0] == 0, name
        assert torch.equal(b.blocks, want[name][0]), name
        assert (b.out.float() - want[name][1].float()).abs().max().item() <= 2 ** -6, name


def test_fused_step_device_timeout_is_reported(cuda_lib):
    # The header's test knob makes the first row barrier wait for an arrival that never
    # comes; every CTA gives up after its bounded wait and the status says so.
    w = I.decode_workload("stall", [9000], 1, 16, 2, "gaussian", seed=9)
    L = _to(w.layers[0])
    b = DecodeBatch(16, 2, w.ctx_len)
    pooled = b.new_pooled()
    b.pool(L.raw_idx_k, pooled)
    b.step_ws.view(torch.int32)[3] = 0x5741171
    b.fused_step(L.raw_idx_k, pooled, L.q_idx, L.q, L.k_cache, L.v_cache)
    st, det = b.fused_status()
    assert st == qb.QSA_ERR_DEVICE_TIMEOUT and det == 0
    qb.qsa_workspace_init(b.step_ws)
    b.fused_step(L.raw_idx_k, pooled, L.q_idx, L.q, L.k_cache, L.v_cache)
    assert b.fused_status()[0] == 0


def test_fused_step_rejects_unsupported(cuda_lib):
    cfg = qb.make_config(16, 4)
    lib = qb.load()
    import ctypes as C
    fake = 0x10000000
    st = lib.qsa_decode_step(C.byref(cfg), fake, fake, 10, fake, fake, fake, fake, fake, 100, fake, fake, 1, 10,
                             fake, fake, fake, None, fake, 1 << 30, None)
    assert st == qb.QSA_ERR_UNSUPPORTED


def test_cache_in_pinned_host_memory(cuda_lib):
    """K/V (and the raw indexer keys) in pinned host memory, gathered over the host link: the
    fused step and the separate decode give the same selection and bit-identical outputs as
    with the cache in device memory. Unregistered host memory is refused on the host."""
    w = I.decode_workload("host_kv", [70001, 5000, 2051], 1, 16, 2, "planted", seed=9)
    L = _to(w.layers[0])
    b = DecodeBatch(w.n_q_heads, w.n_kv_heads, w.ctx_len)
    pooled = b.new_pooled()
    b.pool(L.raw_idx_k, pooled)
    b.fused_step(L.raw_idx_k, pooled, L.q_idx, L.q, L.k_cache, L.v_cache)
    assert b.fused_status()[0] == 0
    want = (b.blocks.clone(), b.count.clone(), b.out.clone(), b.lse.clone())
    hk, hv, hr = (t.cpu().pin_memory() for t in (L.k_cache, L.v_cache, L.raw_idx_k))
    b.blocks.fill_(-7)
    b.out.zero_()
    b.fused_step(hr, pooled, L.q_idx, L.q, hk, hv)
    assert b.fused_status()[0] == 0
    got = (b.blocks, b.count, b.out, b.lse)
    assert all(torch.equal(x, y) for x, y in zip(got, want))
    # the separate attention call on the same selection
    b.attend(L.q, L.k_cache, L.v_cache, want[0], want[1])
    dev_out = b.out.clone()
    b.out.zero_()
    b.attend(L.q, hk, hv, want[0], want[1])
    assert b.device_status()[0] == 0
    assert torch.equal(b.out, dev_out)
    with pytest.raises(qb.QsaError) as e:
        b.fused_step(hr, pooled, L.q_idx, L.q, L.k_cache.cpu(), hv)   # pageable host memory
    assert e.value.status == qb.QSA_ERR_INVALID_ARGUMENT
