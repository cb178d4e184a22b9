"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Small cases cover several tiles and ragged tails; the full-size workloads (long and
million-token decode, the prefill chunk) are checked on sampled rows that the oracle
computes one by one.
"""

import math

import numpy as np
import pytest
import torch

import oracle as O
from indexer_driven_sparse_gb300 import binding as qb
from indexer_driven_sparse_gb300 import inputs as I
from indexer_driven_sparse_gb300.pipeline import DecodeBatch, PrefillChunk
from parity import bits, check_attention, check_lse, check_selection

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _to(layer, device=DEV):
    return I.Layer(*(getattr(layer, f).to(device) for f in ("raw_idx_k", "q_idx", "q", "k_cache", "v_cache")))


def _assert_status_ok(obj):
    st, det = obj.device_status()
    assert st == 0, f"device status {st} detail {det}"


# ----------------------------------------------------------------------------- pooling

def test_pool_keys_bit_exact(cuda_lib):
    g = torch.Generator().manual_seed(0)
    lens = [0, 1, 3, 4, 7, 8, 1023, 4097, 64]
    T = sum(lens)
    raw = (torch.randn(T, 128, generator=g) / math.sqrt(128)).to(torch.bfloat16)
    t0 = sum(lens[:8])
    # last sequence: planted rounding cases (ties, spread exponents, subnormals)
    one, up = 1.0, 1.0 + 2 ** -7
    raw[t0:t0 + 4, :] = torch.tensor([one, up, one, up]).repeat_interleave(1).view(4, 1).to(torch.bfloat16)
    raw[t0 + 4:t0 + 8, :] = torch.tensor([1e-3, 1e3, -1e3, 7.0]).view(4, 1).to(torch.bfloat16)
    raw[t0 + 8:t0 + 12, :] = torch.tensor([2 ** -130, 2 ** -131, 0.0, -2 ** -133]).view(4, 1).to(torch.bfloat16)
    raw[t0 + 12:t0 + 16, :] = torch.tensor([3e38, 3e38, 3e38, 3.3e38]).view(4, 1).to(torch.bfloat16)
    nblk = [n // 4 for n in lens]
    tok_off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    blk_off = np.concatenate([[0], np.cumsum(nblk)]).astype(np.int32)
    cfg = qb.make_config(8, 2)
    ws = qb.make_workspace(qb.OP_POOL_KEYS, cfg, len(lens), max(nblk))
    pooled = torch.full((blk_off[-1], 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    dev = lambda a: torch.tensor(a, dtype=torch.int32, device=DEV)
    qb.qsa_pool_keys(cfg, raw.to(DEV), dev(tok_off), dev(blk_off), dev([0] * len(lens)), dev(nblk), max(nblk),
                     pooled, ws)
    assert qb.qsa_read_device_status(ws)[0] == 0
    got = bits(pooled)
    rb = bits(raw)
    for s in range(len(lens)):
        want = O.pool_keys(rb[tok_off[s]:tok_off[s + 1]])
        assert np.array_equal(got[blk_off[s]:blk_off[s + 1]], want), s
    # incremental: only the last block of each sequence, into a fresh buffer
    pooled2 = torch.zeros_like(pooled)
    begin = [max(0, n - 1) for n in nblk]
    qb.qsa_pool_keys(cfg, raw.to(DEV), dev(tok_off), dev(blk_off), dev(begin), dev(nblk), 1, pooled2, ws)
    got2 = bits(pooled2)
    for s in range(len(lens)):
        if nblk[s]:
            r = blk_off[s] + nblk[s] - 1
            assert np.array_equal(got2[r], got[r])
            assert not np.any(got2[blk_off[s]:r])


# ----------------------------------------------------------------------------- scoring

def test_index_score_within_fp32_bound(cuda_lib):
    ctx = [0, 3, 4, 5, 2051, 2052, 4096, 10001]
    w = I.decode_workload("t", ctx, 1, 8, 2, "gaussian", seed=1)
    L = _to(w.layers[0])
    b = DecodeBatch(8, 2, ctx)
    pooled = b.new_pooled()
    b.pool(L.raw_idx_k, pooled)
    b.score(L.q_idx, pooled)
    _assert_status_ok(b)
    sc = b.scores.cpu().numpy().astype(np.float64)
    rb, qb_ = bits(w.layers[0].raw_idx_k), bits(w.layers[0].q_idx)
    off = w.tok_off
    for s, p in enumerate(ctx):
        pk = O.pool_keys(rb[off[s]:off[s + 1]])
        nb = p // 4
        want = O.score_blocks(qb_[s], pk[:nb])
        bound = O.score_error_bound(qb_[s], pk[:nb])
        assert np.all(np.abs(sc[s, :nb] - want) <= bound + 1e-30), s


@pytest.mark.parametrize("p0,nc,seq_off", [(20000, 300, 0), (9000, 131, 77), (1000, 128, 5)])
def test_index_score_gemm_one_sequence(cuda_lib, p0, nc, seq_off):
    # The queries of a prefill chunk share one history, so their scores run as a
    # tensor-core GEMM (no per-query sequence ids). Tiles are ragged in both directions,
    # the sequence starts at an offset inside the pooled array, and entries b >= nb(p)
    # must stay untouched. The per-query kernel is checked on the same rows.
    from indexer_driven_sparse_gb300.pipeline import _workspace
    w = I.prefill_workload("gemm", p0, nc, 16, 2, "planted", seed=13)
    L = _to(w.layers[0])
    cfg = qb.make_config(16, 2)
    n_tok, i32 = p0 + nc, dict(dtype=torch.int32, device=DEV)
    nbk = n_tok // 4
    pooled = (torch.randn(seq_off + nbk + 3, 128, generator=torch.Generator().manual_seed(3)) / 8).to(
        torch.bfloat16).to(DEV)                                    # other sequences' blocks around it
    tok_off = torch.tensor([0, n_tok], **i32)
    blk_off = torch.tensor([seq_off, seq_off + nbk], **i32)
    ld = (n_tok - 1) // 4 + 3
    ws = _workspace(max(qb.workspace_size(qb.OP_POOL_KEYS, cfg, 1, nbk),
                        qb.workspace_size(qb.OP_INDEX_SCORE, cfg, nc, ld)), DEV)
    qb.qsa_pool_keys(cfg, L.raw_idx_k, tok_off, blk_off, torch.tensor([0], **i32), torch.tensor([nbk], **i32), nbk,
                     pooled, ws)
    q_pos = torch.arange(p0, p0 + nc, **i32)
    out = {}
    for name, q_seq in (("gemm", None), ("rows", torch.zeros(nc, **i32))):
        sc = torch.full((nc, ld), float("nan"), dtype=torch.float32, device=DEV)
        qb.qsa_index_score(cfg, L.q_idx, q_seq, q_pos, pooled, blk_off, sc, ws)
        st, det = qb.qsa_read_device_status(ws)
        assert st == 0, (name, st, det)
        out[name] = sc.cpu().numpy().astype(np.float64)
    pk = O.pool_keys(bits(w.layers[0].raw_idx_k))
    qib = bits(w.layers[0].q_idx)
    for i in range(nc):
        nb = (p0 + i) // 4
        want = O.score_blocks(qib[i], pk[:nb])
        bound = O.score_error_bound(qib[i], pk[:nb])
        for name, sc in out.items():
            assert np.all(np.abs(sc[i, :nb] - want) <= bound + 1e-30), (name, i)
            assert np.all(np.isnan(sc[i, nb:])), (name, i)


# ----------------------------------------------------------------------------- top-k

def _topk_case_rows():
    rng = np.random.default_rng(5)
    rows = []
    for nb in [0, 1, 511, 512, 513, 1024]:
        rows.append(rng.standard_normal(nb).astype(np.float32))
    rows.append(rng.integers(-3, 4, 5000).astype(np.float32))                   # heavy ties
    rows.append(np.full(5000, 0.25, np.float32))                                # all equal
    x = rng.standard_normal(4096).astype(np.float32)
    x[rng.choice(4096, 40, replace=False)] = np.nan
    x[rng.choice(4096, 40, replace=False)] = -0.0
    x[rng.choice(4096, 40, replace=False)] = 0.0
    x[rng.choice(4096, 7, replace=False)] = np.inf
    x[rng.choice(4096, 7, replace=False)] = -np.inf
    rows.append(x)
    y = (rng.standard_normal(3000) * 1e-30).astype(np.float32)                  # tiny and subnormal scores
    y[:600] = -y[:600]
    rows.append(y)
    rows.append(rng.standard_normal(262080).astype(np.float32))                 # million-token row
    z = (1.0 + 1e-3 * rng.standard_normal(20000)).astype(np.float32)            # one outlier squeezes
    z[123] = 1e30                                                               # the rest into one bin
    rows.append(z)
    t = np.concatenate([np.full(300, 5.0), np.full(4000, 1.0), rng.standard_normal(1000) * 0.1 - 3.0])
    rows.append(rng.permutation(t).astype(np.float32))                          # 4000 ties at the cut
    t = np.concatenate([np.full(100, 2.0), np.full(10000, 1.0), rng.standard_normal(500)])
    rows.append(rng.permutation(t).astype(np.float32))                          # 10000 ties at the cut
    rows.append((rng.standard_normal(66559) * 2.8).astype(np.float32))          # a prefill row
    return rows


def test_topk_exact_on_given_scores(cuda_lib):
    rows = _topk_case_rows()
    ld = max(len(r) for r in rows) + 1                # odd: most rows start off 16-byte alignment
    sc = np.zeros((len(rows), ld), np.float32)
    for i, r in enumerate(rows):
        sc[i, :len(r)] = r
    q_pos = [4 * len(r) + (i % 4) for i, r in enumerate(rows)]
    cfg = qb.make_config(16, 2)
    ws = qb.make_workspace(qb.OP_TOPK_BLOCKS, cfg, len(rows), ld)
    blocks = torch.empty(len(rows), 512, dtype=torch.int32, device=DEV)
    count = torch.empty(len(rows), dtype=torch.int32, device=DEV)
    qb.qsa_topk_blocks(cfg, torch.tensor(sc, device=DEV), torch.tensor(q_pos, dtype=torch.int32, device=DEV),
                       blocks, count, ws)
    assert qb.qsa_read_device_status(ws)[0] == 0
    bl, ct = blocks.cpu().numpy(), count.cpu().numpy()
    for i, r in enumerate(rows):
        want = O.select_blocks(r.astype(np.float64))       # same fp32 values, decided exactly
        assert ct[i] == len(want), i
        assert np.array_equal(bl[i, :ct[i]], want), i
        assert np.all(bl[i, ct[i]:] == -1)


# ----------------------------------------------------------------------------- decode

def _run_decode(w, layer=0):
    L = _to(w.layers[layer])
    b = DecodeBatch(w.n_q_heads, w.n_kv_heads, w.ctx_len)
    pooled = b.new_pooled()
    b.pool(L.raw_idx_k, pooled)
    b.step(L.q_idx, L.q, L.k_cache, L.v_cache, pooled)
    _assert_status_ok(b)
    return b, pooled


def _check_decode(w, b, pooled, layer=0, rows=None, max_fp32_swaps=0):
    """Every (or the listed) row: pooled keys bit-exact, selection by the band rule, and
    out / lse against the oracle on the GPU's own selection. Returns the worst errors and
    the swap counts; fp32-bound swaps beyond ``max_fp32_swaps`` fail."""
    Lh = w.layers[layer]
    rb, qib, qbits = bits(Lh.raw_idx_k), bits(Lh.q_idx), bits(Lh.q)
    kb, vb = bits(Lh.k_cache), bits(Lh.v_cache)
    pooled_gpu = bits(pooled)
    blocks, count = b.blocks.cpu().numpy(), b.count.cpu().numpy()
    out, lse = b.out.cpu(), b.lse.cpu().numpy()
    off = w.tok_off
    stats = dict(band=0, fp32=0, max_abs=0.0, rel=0.0, lse=0.0, rows=0)
    for s in (range(w.batch) if rows is None else rows):
        p = w.ctx_len[s]
        pk = O.pool_keys(rb[off[s]:off[s + 1]])
        assert np.array_equal(pooled_gpu[b.blk_off[s].item():b.blk_off[s + 1].item()], pk)
        nb = p // 4
        n_band, n_fp32 = check_selection(blocks[s], count[s], qib[s], pk, nb)
        stats["band"] += n_band
        stats["fp32"] += n_fp32
        ref = O.decode_query(p, qib[s], pk, qbits[s], kb[off[s]:off[s + 1]], vb[off[s]:off[s + 1]], w.n_kv_heads,
                             sel=blocks[s, :count[s]])
        mx, _, rel = check_attention(out[s], ref["out"])
        stats["lse"] = max(stats["lse"], check_lse(lse[s], ref["lse"]))
        stats["max_abs"] = max(stats["max_abs"], mx)
        stats["rel"] = max(stats["rel"], rel)
        stats["rows"] += 1
    print(f"{w.name}: {stats}")
    assert stats["fp32"] <= max_fp32_swaps, stats
    return stats


def test_decode_tiny(cuda_lib):
    w = I.tiny_decode()
    b, pooled = _run_decode(w)
    _check_decode(w, b, pooled)


def test_decode_tiny_sharp(cuda_lib):
    w = I.tiny_decode(kind="sharp", seed=3)
    b, pooled = _run_decode(w)
    st = _check_decode(w, b, pooled)
    assert st["rel"] < 1e-2


@pytest.mark.parametrize("p", [2052, 9001, 131072])
def test_decode_sharp_headline_heads(cuda_lib, p):
    # 16 query / 2 KV heads (8 per KV head) in the sparse regime, Q/K/V ~ N(0,1): outputs of
    # order 0.1, graded by relative error as well as the absolute rule
    w = I.decode_workload(f"sharp16_{p}", [p], 1, 16, 2, "sharp", seed=30 + p % 7)
    b, pooled = _run_decode(w)
    st = _check_decode(w, b, pooled)
    assert st["rel"] < 8e-3


def test_decode_planted_ragged(cuda_lib):
    ctx = [5000, 2052, 70001, 4, 12345]
    w = I.decode_workload("planted_ragged", ctx, 1, 16, 2, "planted", seed=4)
    b, pooled = _run_decode(w)
    _check_decode(w, b, pooled)


def test_decode_batched_short_contexts(cuda_lib):
    lens = I.batched_ctx_lens(short_draw=True)
    assert {0, 1, 3, 4, 2050, 2051, 2052, 2055} <= set(lens)
    w = I.decode_workload("batched_short", lens, 1, 8, 2, "gaussian", seed=0)
    b, pooled = _run_decode(w)
    _check_decode(w, b, pooled)


def test_decode_given_selection_any_order(cuda_lib):
    # The attention must not depend on the order of the block list.
    w = I.decode_workload("perm", [9001], 1, 16, 2, "sharp", seed=9)
    b, pooled = _run_decode(w)
    ref_out = b.out.clone()
    blocks = b.blocks.clone()
    blocks[0] = blocks[0][torch.randperm(512, device=DEV)]
    L = _to(w.layers[0])
    b.attend(L.q, L.k_cache, L.v_cache, blocks=blocks)
    torch.cuda.synchronize()
    d = (b.out.float() - ref_out.float()).abs().max().item()
    assert d <= 2 ** -7


def test_device_bounds_error_is_recorded(cuda_lib):
    # Block id == nb is invalid; the kernel must flag it and skip the access. The id is
    # chosen so that even an unchecked read would stay inside the K/V buffers.
    w = I.decode_workload("bad", [9000, 9000], 1, 8, 2, "gaussian", seed=2)
    b, pooled = _run_decode(w)
    blocks = b.blocks.clone()
    blocks[0, 5] = 9000 // 4
    L = _to(w.layers[0])
    b.attend(L.q, L.k_cache, L.v_cache, blocks=blocks)
    st, det = b.device_status()
    assert st == qb.QSA_ERR_DEVICE_BOUNDS and det == 0
    qb.qsa_workspace_init(b.ws)
    assert b.device_status()[0] == 0


# ----------------------------------------------------------------------------- prefill

def _run_prefill(w, interval=8192):
    L = _to(w.layers[0])
    c = PrefillChunk(w.n_q_heads, w.n_kv_heads, w.ctx_len[0], w.n_chunk, interval)
    pooled = c.new_pooled()
    c.pool(L.raw_idx_k, pooled)
    c.run(L.q_idx, L.q, L.k_cache, L.v_cache, pooled)
    _assert_status_ok(c)
    return c, pooled


def _check_prefill(w, c, rows, max_fp32_swaps=0):
    Lh = w.layers[0]
    rb, qib, qbits = bits(Lh.raw_idx_k), bits(Lh.q_idx), bits(Lh.q)
    kb, vb = bits(Lh.k_cache), bits(Lh.v_cache)
    pk = O.pool_keys(rb)
    blocks, count = c.blocks.cpu().numpy(), c.count.cpu().numpy()
    out, lse = c.out.cpu(), c.lse.cpu().numpy()
    stats = dict(band=0, fp32=0, max_abs=0.0, rel=0.0, lse=0.0, rows=0)
    for i in rows:
        p = c.p0 + i
        n_band, n_fp32 = check_selection(blocks[i], count[i], qib[i], pk, p // 4)
        stats["band"] += n_band
        stats["fp32"] += n_fp32
        ref = O.decode_query(p, qib[i], pk, qbits[i], kb, vb, w.n_kv_heads, sel=blocks[i, :count[i]])
        mx, _, rel = check_attention(out[i], ref["out"])
        stats["lse"] = max(stats["lse"], check_lse(lse[i], ref["lse"]))
        stats["max_abs"] = max(stats["max_abs"], mx)
        stats["rel"] = max(stats["rel"], rel)
        stats["rows"] += 1
    print(f"{w.name}: {stats}")
    assert stats["fp32"] <= max_fp32_swaps, stats
    return stats


def test_prefill_small_ragged(cuda_lib):
    w = I.prefill_workload("prefill_small", 8197, 300, 16, 2, "planted", seed=6)
    c, _ = _run_prefill(w)
    _check_prefill(w, c, range(300))


def test_prefill_sharp_multi_tile_all_rows(cuda_lib):
    # 19 query tiles of 16 (the last ragged) at p0 = 20,000: every row graded, sharp Q/K/V
    w = I.prefill_workload("prefill_sharp_20k", 20000, 300, 16, 2, "planted_sharp", seed=31)
    c, _ = _run_prefill(w)
    st = _check_prefill(w, c, range(300))
    assert st["rel"] < 8e-3


def test_prefill_interval_invariance(cuda_lib):
    w = I.prefill_workload("prefill_iv", 20000, 64, 16, 2, "sharp", seed=8)
    outs = []
    for iv in (1024, 8192, 16384):
        c, _ = _run_prefill(w, iv)
        outs.append(c.out.float().clone())
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 2 ** -7


@pytest.mark.parametrize("hq,hkv,p0,nc", [
    (16, 1, 0, 298),       # 16 heads per KV head; p < 4 .. dense; the last own block runs past the cache
    (16, 2, 2000, 77),     # 8 per KV head across the dense/sparse threshold, ragged last tile
    (32, 2, 9000, 40),     # 16 per KV head, sparse, fewer queries than one tile
    (8, 2, 2040, 50),      # 4 per KV head: the CUDA-core path
])
def test_prefill_head_ratios_and_edges(cuda_lib, hq, hkv, p0, nc):
    w = I.prefill_workload(f"prefill_{hq}_{hkv}", p0, nc, hq, hkv, "planted", seed=11)
    c, _ = _run_prefill(w, 1024)
    _check_prefill(w, c, range(nc))


def test_prefill_out_of_order_list_is_flagged(cuda_lib):
    # The tensor-core tiles walk each list interval by interval and need it ascending;
    # a reversed row is recorded as a bounds error instead of being dropped silently.
    w = I.prefill_workload("prefill_rev", 20000, 32, 16, 2, "gaussian", seed=12)
    c, _ = _run_prefill(w, 1024)
    L = _to(w.layers[0])
    blocks = c.blocks.clone()
    blocks[5] = blocks[5].flip(0)
    c.attend(L.q, L.k_cache, L.v_cache, blocks=blocks)
    st, det = c.device_status()
    assert st == qb.QSA_ERR_DEVICE_BOUNDS and det == 5
    qb.qsa_workspace_init(c.ws)
    c.attend(L.q, L.k_cache, L.v_cache)
    _assert_status_ok(c)


@pytest.mark.parametrize("case", ["chunk_full", "short_history", "all_equal", "sharp"])
def test_prefill_select_equals_score_then_topk(cuda_lib, case):
    # the fused selection (no score matrix) returns exactly the blocks of qsa_index_score +
    # qsa_topk_blocks: the same fp32 scores, the same keys; the equal-score and short-history
    # rows overflow their candidate slots and take the exact path
    if case == "chunk_full":
        w = I.prefill_chunk(device="cuda")
    elif case == "short_history":
        w = I.prefill_workload("sel_short", 3000, 300, 16, 2, "planted", seed=21)
    elif case == "all_equal":
        w = I.prefill_workload("sel_ties", 150000, 256, 16, 2, "gaussian", seed=22)
        w.layers[0].q_idx.zero_()
    else:
        w = I.prefill_workload("sel_sharp", 140000, 640, 16, 2, "sharp", seed=23)
    L = _to(w.layers[0])
    c = PrefillChunk(w.n_q_heads, w.n_kv_heads, w.ctx_len[0], w.n_chunk, 8192)
    assert c.fused_select
    pooled = c.new_pooled()
    c.pool(L.raw_idx_k, pooled)
    c.score(L.q_idx, pooled)
    c.topk()
    _assert_status_ok(c)
    want_b, want_c = c.blocks.clone(), c.count.clone()
    c.blocks.fill_(-9)
    c.count.fill_(-9)
    c.scores.fill_(float("nan"))
    c.select(L.q_idx, pooled)
    _assert_status_ok(c)
    assert torch.equal(c.count, want_c)
    assert torch.equal(c.blocks, want_b)


def test_prefill_cache_in_pinned_host_memory(cuda_lib):
    # K/V gathered from pinned host memory over the host link: the same outputs, bit for bit,
    # on the tensor-core path (16 q / 2 KV heads) and the CUDA-core path (8 q / 2 KV heads)
    for hq in (16, 8):
        w = I.prefill_workload(f"prefill_host_{hq}", 9000, 40, hq, 2, "planted", seed=13)
        c, _ = _run_prefill(w, 1024)
        L = _to(w.layers[0])
        dev_out, dev_lse = c.out.clone(), c.lse.clone()
        hk, hv = L.k_cache.cpu().pin_memory(), L.v_cache.cpu().pin_memory()
        c.out.zero_()
        c.attend(L.q, hk, hv)
        _assert_status_ok(c)
        assert torch.equal(c.out, dev_out) and torch.equal(c.lse, dev_lse)
        # staged: the rows copied into a device arena first (one pass over the link), then the
        # same kernel; a stage one byte short is refused
        need = 2 * hk.numel() * 2
        stage = torch.empty(need + 64, dtype=torch.uint8, device="cuda")
        c.out.zero_()
        c.attend_staged(L.q, hk, hv, stage)
        _assert_status_ok(c)
        assert torch.equal(c.out, dev_out) and torch.equal(c.lse, dev_lse)
        with pytest.raises(qb.QsaError) as e:
            c.attend_staged(L.q, hk, hv, stage[: need - 1])
        assert e.value.status == qb.QSA_ERR_WORKSPACE_TOO_SMALL


# ----------------------------------------------------------------------------- full-size workloads, sampled

def _host_layers(w):
    w.layers = [I.Layer(*(getattr(w.layers[0], f).cpu() for f in ("raw_idx_k", "q_idx", "q", "k_cache", "v_cache")))]


@pytest.mark.parametrize("kind", ["planted", "planted_sharp"])
def test_long_decode_full_size_one_layer(cuda_lib, kind):
    w = I.long_decode(n_layers=1, kind=kind)
    b, pooled = _run_decode(w)
    _host_layers(w)
    _check_decode(w, b, pooled)


@pytest.mark.parametrize("kind", ["planted", "planted_sharp"])
def test_million_decode_full_size_one_layer(cuda_lib, kind):
    w = I.million_decode(n_layers=1, kind=kind)
    b, pooled = _run_decode(w)
    _host_layers(w)
    _check_decode(w, b, pooled)


def test_prefill_chunk_full_size_sampled(cuda_lib):
    # the headline chunk (planted, correlated queries) on its stated distribution: the
    # first and last query of every 16-query tile
    w = I.prefill_chunk()
    c, _ = _run_prefill(w)
    _host_layers(w)
    rows = sorted({r for t in range(0, 4096, 16) for r in (t, t + 15)})
    _check_prefill(w, c, rows)


def test_prefill_chunk_full_size_sharp(cuda_lib):
    # the same chunk geometry and selection structure with Q/K/V ~ N(0,1): the first and the
    # last query of every 16-query tile (512 rows), graded by relative error too
    w = I.prefill_chunk(kind="planted_sharp")
    c, _ = _run_prefill(w)
    _host_layers(w)
    rows = sorted({r for t in range(0, 4096, 16) for r in (t, t + 15)})
    st = _check_prefill(w, c, rows)
    assert st["rows"] == 512 and st["rel"] < 8e-3
