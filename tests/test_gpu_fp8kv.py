"""FP8 K/V rows (E4M3 codes per 128-dim group with an fp32 scale): the GPU quantiser and
dequantiser against the oracle's bit for bit, the fused decode step over FP8 K/V
(qsa_decode_step_fp8kv) against the oracle's attention on the dequantised rows, with bf16 and
with FP8 indexer keys, and the prefill chunk over FP8 K/V (qsa_sparse_prefill_chunk_fp8kv).
"""

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


def _quantize_gpu(x):
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scales = torch.empty(x.shape[:-1] + (2,), dtype=torch.float32, device=x.device)
    qb.qsa_quantize_kv_fp8(x, codes, scales)
    return codes, scales


def _special_rows(n, seed):
    """bf16 rows [n, 2, 256] with the quantiser's edge cases: zero rows and groups, one
    non-zero element, the bf16 extremes, subnormal bf16 values, exact E4M3 multiples."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((n, 2, 256), generator=g)
    x[0] = 0.0
    x[1, 0, 128:] = 0.0
    x[2, 1] = 0.0
    x[2, 1, 77] = -3.0
    x[3, 0] = 3.3895e38                            # largest finite bf16
    x[3, 0, 5] = -3.3895e38
    x[4, 1, :128] = torch.randn(128, generator=g) * 1e-39     # bf16 subnormals
    x[5, 0] = torch.arange(256) % 15 - 7           # small integers: exact codes
    x[6] *= 1e-30
    x[7] *= 1e30
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("n", [8, 9, 1000, 4097])
def test_quantize_kv_fp8_bit_exact(cuda_lib, n):
    x = _special_rows(n, seed=n)
    codes, scales = _quantize_gpu(x.to(DEV))
    want_c, want_s = O.quantize_kv_fp8(bits(x))
    assert np.array_equal(codes.cpu().numpy(), want_c)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), want_s.view(np.uint32))


def _kv8(L):
    kc, ks = _quantize_gpu(L.k_cache)
    vc, vs = _quantize_gpu(L.v_cache)
    return kc, ks, vc, vs


def _grade(w, b, blocks_ref, kv8, fp8_keys=None, max_fp32_swaps=0):
    """Selection: equal to the bf16-K/V step's on the same keys, and graded against the oracle
    by the band rule. Attention: the oracle on the oracle's FP8 rows of the attended tokens."""
    assert torch.equal(b.blocks, blocks_ref), "FP8-K/V step selected other blocks than the bf16-K/V step"
    Lh = w.layers[0]
    rb, qib, qbits = bits(Lh.raw_idx_k), bits(Lh.q_idx), bits(Lh.q)
    kb, vb = bits(Lh.k_cache), bits(Lh.v_cache)
    blocks, count, out, lse = b.blocks.cpu().numpy(), b.count.cpu().numpy(), b.out.cpu(), b.lse.cpu().numpy()
    off = w.tok_off
    stats = dict(band=0, fp32=0, rel=0.0, lse=0.0, rows=0)
    for s in range(w.batch):
        p = w.ctx_len[s]
        nb = p // 4
        pk = O.pool_keys(rb[off[s]:off[s + 1]])
        if fp8_keys is None:
            n_band, n_fp32 = check_selection(blocks[s], count[s], qib[s], pk, nb)
        else:
            vals, scl = O.quantize_pooled_fp8(pk)
            n_band, n_fp32 = check_selection(blocks[s], count[s], qib[s], None, nb,
                                             scores=O.score_blocks_fp8(qib[s], vals[:nb], scl[:nb]),
                                             bound=O.score_error_bound_fp8(qib[s], vals[:nb], scl[:nb]))
        stats["band"] += n_band
        stats["fp32"] += n_fp32
        tokens = O.attended_tokens(p, blocks[s, :count[s]])
        kd = O.dequantize_kv_fp8(*O.quantize_kv_fp8(kb[off[s] + tokens]))
        vd = O.dequantize_kv_fp8(*O.quantize_kv_fp8(vb[off[s] + tokens]))
        ref_out, ref_lse = O.attend(O.bf16_bits_to_f64(qbits[s]), kd, vd, np.arange(tokens.size), w.n_kv_heads,
                                    1.0 / 16.0)
        stats["rel"] = max(stats["rel"], check_attention(out[s], ref_out)[2])
        stats["lse"] = max(stats["lse"], check_lse(lse[s], ref_lse))
        stats["rows"] += 1
    print(f"{w.name} fp8 kv: {stats}")
    assert stats["fp32"] <= max_fp32_swaps, stats
    return stats


def _run(w, fp8_keys=False):
    L = w.layers[0]
    L = I.Layer(*(getattr(L, f).to(DEV) for f in ("raw_idx_k", "q_idx", "q", "k_cache", "v_cache")))
    b = DecodeBatch(w.n_q_heads, w.n_kv_heads, w.ctx_len)
    if fp8_keys:
        keys = b.new_fp8_keys()
        b.pool_fp8(L.raw_idx_k, *keys)
        b.fused_step_fp8(L.raw_idx_k, *keys, L.q_idx, L.q, L.k_cache, L.v_cache)
    else:
        keys = b.new_pooled()
        b.pool(L.raw_idx_k, keys)
        b.fused_step(L.raw_idx_k, keys, L.q_idx, L.q, L.k_cache, L.v_cache)
    assert b.fused_status()[0] == 0
    blocks_ref = b.blocks.clone()
    kv8 = _kv8(L)
    want = O.quantize_kv_fp8(bits(w.layers[0].k_cache))
    assert np.array_equal(kv8[0].cpu().numpy(), want[0])
    b.blocks.fill_(-7)
    b.out.zero_()
    b.fused_step_fp8kv(L.raw_idx_k, keys, L.q_idx, L.q, kv8)
    st = b.fused_status()
    assert st[0] == 0, st
    return b, blocks_ref, kv8, (keys if fp8_keys else None)


@pytest.mark.parametrize("case", ["sharp16_2052", "sharp16_9001", "sharp16_131072", "sharp_ragged", "dense",
                                  "tiny_sharp", "g1", "one_kv_head", "fp8_keys_ragged"])
def test_fused_step_fp8kv(cuda_lib, case):
    fp8_keys = False
    if case.startswith("sharp16_"):
        p = int(case.split("_")[1])
        w = I.decode_workload(case, [p], 1, 16, 2, "sharp", seed=70 + p % 13)
    elif case == "sharp_ragged":
        w = I.decode_workload(case, [2052, 70001, 9001, 4, 2051, 33333], 1, 16, 2, "planted_sharp", seed=71)
    elif case == "dense":
        w = I.decode_workload(case, [0, 1, 7, 2047, 2051], 1, 16, 2, "sharp", seed=72)
    elif case == "tiny_sharp":
        w = I.tiny_decode(kind="sharp", seed=73)
    elif case == "g1":                              # one query head per KV head
        w = I.decode_workload(case, [5000, 3001], 1, 2, 2, "sharp", seed=74)
    elif case == "one_kv_head":                     # Hkv = 1: 8-byte scale pairs per token
        w = I.decode_workload(case, [9000, 2051, 40000], 1, 8, 1, "planted_sharp", seed=75)
    else:
        fp8_keys = True
        w = I.decode_workload(case, [5000, 2052, 70001, 4, 12345, 0, 3, 2051], 1, 16, 2, "planted_sharp", seed=76)
    b, blocks_ref, kv8, keys = _run(w, fp8_keys)
    _grade(w, b, blocks_ref, kv8, keys)


@pytest.mark.parametrize("fp8_keys", [False, True])
def test_fused_step_fp8kv_million_full_size(cuda_lib, fp8_keys):
    # the headline geometry (16 / 2 heads, 1,048,320 tokens) with N(0,1) Q/K/V
    w = I.million_decode(n_layers=1, kind="planted_sharp")
    b, blocks_ref, kv8, keys = _run(w, fp8_keys)
    w.layers = [I.Layer(*(getattr(w.layers[0], f).cpu() for f in ("raw_idx_k", "q_idx", "q", "k_cache", "v_cache")))]
    _grade(w, b, blocks_ref, kv8, keys)


@pytest.mark.parametrize("kind", ["gaussian", "sharp"])
def test_fused_step_fp8kv_batched_full_size(cuda_lib, kind):
    # the batched workload (32 ragged sequences, 8 query / 2 KV heads): every row graded
    w = I.batched_decode(n_layers=1, kind=kind)
    b, blocks_ref, kv8, keys = _run(w)
    w.layers = [I.Layer(*(getattr(w.layers[0], f).cpu() for f in ("raw_idx_k", "q_idx", "q", "k_cache", "v_cache")))]
    _grade(w, b, blocks_ref, kv8, keys)


def test_fused_step_fp8kv_host_memory_rows_match(cuda_lib):
    # FP8 K/V (codes and scales) in mapped pinned host memory: the same results bit for bit
    w = I.decode_workload("fp8kv_host", [70001, 2052], 1, 16, 2, "planted_sharp", seed=77)
    b, blocks_ref, kv8, _ = _run(w)
    want = (b.blocks.clone(), b.out.clone(), b.lse.clone())
    host = [t.cpu().pin_memory() for t in kv8]
    L = w.layers[0]
    L = I.Layer(*(getattr(L, f).to(DEV) for f in ("raw_idx_k", "q_idx", "q", "k_cache", "v_cache")))
    pooled = b.new_pooled()
    b.pool(L.raw_idx_k, pooled)
    b.out.zero_()
    b.fused_step_fp8kv(L.raw_idx_k, pooled, L.q_idx, L.q, host)
    torch.cuda.synchronize()
    assert b.fused_status()[0] == 0
    assert torch.equal(b.blocks, want[0]) and torch.equal(b.out, want[1]) and torch.equal(b.lse, want[2])


# ----------------------------------------------------------------------------- dequantiser

def _tie_pairs(n_want, seed):
    """(E4M3 code, fp32 scale) pairs whose fp32 product lies exactly halfway between two bf16
    values while the exact product does not: rounding the fp32 product would pick the wrong
    neighbour half of the time, so the dequantiser must decide these by the exact product."""
    rng = np.random.default_rng(seed)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    got_c, got_s = [], []
    while len(got_c) < n_want:
        c = finite[rng.integers(0, finite.size, 1 << 20)]
        sc = (rng.uniform(1.0, 2.0, 1 << 20) * 2.0 ** rng.integers(-60, 60, 1 << 20)).astype(np.float32)
        v = O.e4m3_value(c)
        p32 = v.astype(np.float32) * sc                          # IEEE fp32 product
        u = p32.view(np.uint32)
        hit = ((u & 0xFFFF) == 0x8000) & (np.abs(p32) >= np.float32(2.0 ** -126)) & \
              (v * sc.astype(np.float64) != p32.astype(np.float64))
        got_c.extend(c[hit].tolist())
        got_s.extend(sc[hit].tolist())
    return np.array(got_c[:n_want], dtype=np.uint8), np.array(got_s[:n_want], dtype=np.float32)


def test_dequantize_kv_fp8_bit_exact(cuda_lib):
    # every code (NaN codes included) against scales from fp32 subnormals to overflow, plus
    # rows whose fp32 products are bf16 rounding ties, exact or not: each element code x scale
    # rounded once
    rng = np.random.default_rng(5)
    n = 3000
    codes = rng.integers(0, 256, (n, 256), dtype=np.uint8)
    codes[0] = np.arange(256, dtype=np.uint8)
    scales = (2.0 ** rng.uniform(-148, 120, (n, 2))).astype(np.float32)
    scales[1] = 0.0
    scales[2] = 1.0
    scales[3] = np.float32(3.4028235e38)                   # products overflow to infinity
    scales[4] = np.float32(2.0 ** -149)                     # the smallest fp32 subnormal
    scales[5] = np.float32(1.0 + 2.0 ** -23)
    # scales as the quantiser makes them (a bf16 group maximum / 448): many products are exact
    # and sit on bf16 midpoints, which must round to even
    amax = O.bf16_bits_to_f64(O.f64_to_bf16_bits(np.abs(rng.standard_normal((1000, 2))) * 3 + 0.01))
    scales[1000:2000] = (amax.astype(np.float32) / np.float32(448.0)).astype(np.float32)
    tc, ts = _tie_pairs(200, seed=6)
    for i in range(tc.size):                                # one tie pair per 128-dim group
        r, g = 10 + i // 2, i % 2
        codes[r, 128 * g:128 * (g + 1)] = tc[i]
        scales[r, g] = ts[i]
    want = O.f64_to_bf16_bits(O.dequantize_kv_fp8(codes, scales))
    x = torch.empty((n, 256), dtype=torch.bfloat16, device=DEV)
    qb.qsa_dequantize_kv_fp8(torch.from_numpy(codes).to(DEV), torch.from_numpy(scales).to(DEV), x)
    got = bits(x)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{bad.shape[0]} elements differ, first {bad[:4].tolist()}"
    # the tie rows really are ties of the fp32 product: rounding it would differ somewhere
    p32 = (O.e4m3_value(tc).astype(np.float32) * ts).astype(np.float32)
    naive = (p32.view(np.uint32) >> 16).astype(np.uint16) + ((p32.view(np.uint32) >> 16) & 1).astype(np.uint16)
    assert np.any(naive != want[10:10 + tc.size // 2].reshape(-1, 128)[:, 0])


# ----------------------------------------------------------------------------- prefill over FP8 K/V

def _prefill_fp8kv(w, interval=8192, host_rows=False):
    """The chunk's selection and bf16 attention, then the attention over FP8 K/V (the GPU
    quantiser's rows, checked equal to the oracle's); returns the chunk, the rows and the stage."""
    L = w.layers[0]
    L = I.Layer(*(getattr(L, f).to(DEV) for f in ("raw_idx_k", "q_idx", "q", "k_cache", "v_cache")))
    c = PrefillChunk(w.n_q_heads, w.n_kv_heads, w.ctx_len[0], w.n_chunk, interval)
    pooled = c.new_pooled()
    c.pool(L.raw_idx_k, pooled)
    c.run(L.q_idx, L.q, L.k_cache, L.v_cache, pooled)
    assert c.device_status()[0] == 0
    kv8 = _kv8(L)
    n_chk = min(L.v_cache.shape[0], 8192)            # the quantiser against the oracle's on these rows
    want = O.quantize_kv_fp8(bits(L.v_cache[-n_chk:]))
    assert np.array_equal(kv8[2][-n_chk:].cpu().numpy(), want[0])
    assert np.array_equal(kv8[3][-n_chk:].cpu().numpy().view(np.uint32), want[1].view(np.uint32))
    stage = torch.empty(2 * L.k_cache.numel() * 2, dtype=torch.uint8, device=DEV)
    c.out.zero_()
    c.attend_fp8kv(L.q, [t.cpu().pin_memory() for t in kv8] if host_rows else kv8, stage)
    st = c.device_status()
    assert st[0] == 0, st
    return c, kv8, stage, L


def _grade_prefill_fp8kv(w, c, rows):
    """Each row against the oracle on the rows the contract computes on (code x scale rounded
    once to bf16) with every attention rule, and against the exact FP8 values (code x scale in
    float64) by the output rules, which the rounding must still meet."""
    Lh = w.layers[0]
    qbits = bits(Lh.q)
    kb, vb = bits(Lh.k_cache), bits(Lh.v_cache)
    blocks, count = c.blocks.cpu().numpy(), c.count.cpu().numpy()
    out, lse = c.out.cpu(), c.lse.cpu().numpy()
    qf = O.bf16_bits_to_f64(qbits)
    # the oracle's FP8 rows of every token the graded rows attend, quantised once
    toks = {i: O.attended_tokens(c.p0 + i, blocks[i, :count[i]]) for i in rows}
    union = np.unique(np.concatenate([toks[i] for i in rows])) if toks else np.zeros(0, np.int64)
    kd_u = O.dequantize_kv_fp8(*O.quantize_kv_fp8(kb[union]))
    vd_u = O.dequantize_kv_fp8(*O.quantize_kv_fp8(vb[union]))
    stats = dict(rel=0.0, rel_exact=0.0, lse=0.0, rows=0)
    for i in rows:
        tokens = toks[i]
        at = np.searchsorted(union, tokens)
        kd, vd = kd_u[at], vd_u[at]
        kr, vr = O.bf16_bits_to_f64(O.f64_to_bf16_bits(kd)), O.bf16_bits_to_f64(O.f64_to_bf16_bits(vd))
        ref_out, ref_lse = O.attend(qf[i], kr, vr, np.arange(tokens.size), w.n_kv_heads, 1.0 / 16.0)
        stats["rel"] = max(stats["rel"], check_attention(out[i], ref_out)[2])
        stats["lse"] = max(stats["lse"], check_lse(lse[i], ref_lse))
        ex_out, _ = O.attend(qf[i], kd, vd, np.arange(tokens.size), w.n_kv_heads, 1.0 / 16.0)
        stats["rel_exact"] = max(stats["rel_exact"], check_attention(out[i], ex_out)[2])
        stats["rows"] += 1
    print(f"{w.name} fp8 kv prefill: {stats}")
    return stats


def test_prefill_fp8kv_sharp_multi_tile_all_rows(cuda_lib):
    # 19 query tiles of 16 (the last ragged) at p0 = 20,000 on the tensor cores, every row
    w = I.prefill_workload("prefill_fp8kv_20k", 20000, 300, 16, 2, "planted_sharp", seed=81)
    c, _, _, _ = _prefill_fp8kv(w)
    st = _grade_prefill_fp8kv(w, c, range(300))
    assert st["rows"] == 300 and st["rel"] < 8e-3


def test_prefill_fp8kv_full_size_sampled(cuda_lib):
    # the bench's chunk (4096 queries at p0 = 262,144, 16 / 2 heads) over FP8 K/V with Q/K/V ~
    # N(0,1): the first and the last query of every 16-query tile (512 rows)
    w = I.prefill_chunk(kind="planted_sharp")
    c, _, _, _ = _prefill_fp8kv(w)
    w.layers = [I.Layer(*(getattr(w.layers[0], f).cpu() for f in ("raw_idx_k", "q_idx", "q", "k_cache", "v_cache")))]
    rows = sorted({r for t in range(0, 4096, 16) for r in (t, t + 15)})
    st = _grade_prefill_fp8kv(w, c, rows)
    assert st["rows"] == 512 and st["rel"] < 8e-3


@pytest.mark.parametrize("hq,hkv,p0,nc", [
    (16, 1, 0, 298),       # dense start, one KV head (the scale pairs of one head per token)
    (8, 2, 2040, 50),      # 4 query heads per KV head: the CUDA-core path
])
def test_prefill_fp8kv_head_ratios_and_edges(cuda_lib, hq, hkv, p0, nc):
    w = I.prefill_workload(f"prefill_fp8kv_{hq}_{hkv}", p0, nc, hq, hkv, "sharp", seed=82)
    c, _, _, _ = _prefill_fp8kv(w, 1024)
    _grade_prefill_fp8kv(w, c, range(nc))


def test_prefill_fp8kv_equals_bf16_prefill_on_the_dequantised_rows(cuda_lib):
    # the stage holds qsa_dequantize_kv_fp8's rows, and the chunk equals the bf16 prefill on
    # them bit for bit; FP8 rows in mapped pinned host memory give the same bits again
    w = I.prefill_workload("prefill_fp8kv_eq", 9000, 40, 16, 2, "planted_sharp", seed=83)
    c, kv8, stage, L = _prefill_fp8kv(w, 1024)
    got = (c.out.clone(), c.lse.clone())
    kx, vx = torch.empty_like(L.k_cache), torch.empty_like(L.v_cache)
    qb.qsa_dequantize_kv_fp8(kv8[0], kv8[1], kx)
    qb.qsa_dequantize_kv_fp8(kv8[2], kv8[3], vx)
    n = L.k_cache.numel() * 2
    assert torch.equal(stage[:n], kx.view(-1).view(torch.uint8)) and torch.equal(stage[n:], vx.view(-1).view(torch.uint8))
    c.out.zero_()
    c.attend(L.q, kx, vx)
    assert c.device_status()[0] == 0
    assert torch.equal(c.out, got[0]) and torch.equal(c.lse, got[1])
    c2, _, _, _ = _prefill_fp8kv(w, 1024, host_rows=True)
    assert torch.equal(c2.out, got[0]) and torch.equal(c2.lse, got[1])
    with pytest.raises(qb.QsaError) as e:
        c.attend_fp8kv(L.q, kv8, stage[: 2 * n - 1])
    assert e.value.status == qb.QSA_ERR_WORKSPACE_TOO_SMALL
