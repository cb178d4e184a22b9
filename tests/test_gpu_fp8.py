"""FP8 (E4M3) indexer keys on the GPU vs the fp64 oracle, through the C ABI.

Pooling into codes and scales must match the oracle exactly (the same fp32 divisions, the
same round-to-nearest-even onto the E4M3 grid). Scores must lie within the fp32 bound of
the oracle's; selections follow the band rule of the bf16 path on the FP8 scores; the
attention over the GPU's selection within the usual tolerance.
"""

import math

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


def _e4m3_values() -> np.ndarray:
    """Value of each of the 256 E4M3 byte codes, from the format's bit layout
    (sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 subnormal; 0x7F/0xFF NaN)."""
    out = np.empty(256)
    for b in range(256):
        s, e, m = b >> 7, (b >> 3) & 15, b & 7
        v = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        out[b] = np.nan if (e == 15 and m == 7) else (-v if s else v)
    return out


E4M3 = _e4m3_values()


def _to(layer, device=DEV):
    return I.Layer(*(getattr(layer, f).to(device) for f in ("raw_idx_k", "q_idx", "q", "k_cache", "v_cache")))


def _check_keys(codes, scales, pooled_bits):
    """GPU codes/scales of some blocks == the oracle's quantisation of their pooled keys."""
    vals, scl = O.quantize_pooled_fp8(pooled_bits)
    got_s = scales.cpu().numpy()
    assert np.array_equal(got_s.view(np.uint32), scl.view(np.uint32))
    got_v = E4M3[codes.cpu().numpy()]
    assert not np.isnan(got_v).any()
    assert np.array_equal(got_v, vals)
    return vals, scl


def test_pool_keys_fp8_exact(cuda_lib):
    g = torch.Generator().manual_seed(5)
    lens = [0, 3, 4, 9, 1024, 4097, 40]
    T = sum(lens)
    raw = (torch.randn(T, 128, generator=g) / math.sqrt(128)).to(torch.bfloat16)
    t0 = sum(lens[:6])
    # last sequence (10 blocks): planted cases
    raw[t0:t0 + 4] = 0.0                                                        # all-zero key: scale 0
    raw[t0 + 4:t0 + 8, :64] = 2 ** -130                                         # subnormal bf16 key
    raw[t0 + 4:t0 + 8, 64:] = -(2 ** -128)
    top = torch.linspace(-1.0, 1.0, 128, dtype=torch.float64) * 3e38                # near the bf16 top
    raw[t0 + 8:t0 + 12] = top.to(torch.bfloat16)
    ramp = torch.tensor([2.0 ** (k / 4.0 - 20) for k in range(128)])           # codes from subnormal E4M3 to 448
    raw[t0 + 12:t0 + 16] = ramp.to(torch.bfloat16)
    raw[t0 + 16:t0 + 20] = torch.where(torch.arange(128) % 2 == 0, 1.0, -1.0).to(torch.bfloat16)
    raw[t0 + 20:t0 + 24] = 0.0
    raw[t0 + 20:t0 + 24, 7] = 5.0                                               # one non-zero dim
    nblk = [n // 4 for n in lens]
    tok_off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    blk_off = np.concatenate([[0], np.cumsum(nblk)]).astype(np.int32)
    cfg = qb.make_config(8, 2)
    ws = qb.make_workspace(qb.OP_POOL_KEYS, cfg, len(lens), max(nblk))
    nb_tot = int(blk_off[-1])
    codes = torch.full((nb_tot, 128), 0x7F, dtype=torch.uint8, device=DEV)
    scales = torch.full((nb_tot,), float("nan"), dtype=torch.float32, device=DEV)
    dev = lambda a: torch.tensor(a, dtype=torch.int32, device=DEV)
    qb.qsa_pool_keys_fp8(cfg, raw.to(DEV), dev(tok_off), dev(blk_off), dev([0] * len(lens)), dev(nblk), max(nblk),
                         codes, scales, ws)
    assert qb.qsa_read_device_status(ws)[0] == 0
    rb = bits(raw)
    pooled = np.concatenate([O.pool_keys(rb[tok_off[s]:tok_off[s + 1]]) for s in range(len(lens))])
    vals, scl = _check_keys(codes, scales, pooled)
    last = slice(blk_off[6], blk_off[7])
    assert scl[last][0] == 0 and scl[last][1] > 0                               # zero key, subnormal key
    assert np.isfinite(O.bf16_bits_to_f64(pooled)).all()
    assert np.abs(vals[last][1:]).max(axis=1).min() == O.E4M3_MAX
    used = np.unique(np.abs(vals[last][3]))
    assert np.any((used > 0) & (used < 2.0 ** -6)) and used.max() == 448.0     # subnormal and top codes hit
    # incremental: the newest block of each sequence only
    codes2 = torch.zeros_like(codes)
    scales2 = torch.zeros_like(scales)
    begin = [max(0, n - 1) for n in nblk]
    qb.qsa_pool_keys_fp8(cfg, raw.to(DEV), dev(tok_off), dev(blk_off), dev(begin), dev(nblk), 1, codes2, scales2, ws)
    assert qb.qsa_read_device_status(ws)[0] == 0
    c1, c2, s2 = codes.cpu(), codes2.cpu(), scales2.cpu()
    for s in range(len(lens)):
        if nblk[s]:
            r = blk_off[s] + nblk[s] - 1
            assert torch.equal(c2[r], c1[r]) and s2[r].item() == scales[r].item()
            assert not c2[blk_off[s]:r].any()


def _pooled_oracle(w, s, layer=0):
    L = w.layers[layer]
    off = w.tok_off
    pk = O.pool_keys(bits(L.raw_idx_k[off[s]:off[s + 1]]))
    return pk


def check_selection_fp8(gpu_blocks, gpu_count, q_idx_bits, vals, scl, nb, k=O.BLOCK_TOPK):
    """The band rule on FP8 scores: the GPU's set equals the oracle's except for blocks whose
    fp64 score lies within 1e-4 relative of the k-th, or (counted apart) within the fp32 bound."""
    scores = O.score_blocks_fp8(q_idx_bits, vals[:nb], scl[:nb])
    bound = O.score_error_bound_fp8(q_idx_bits, vals[:nb], scl[:nb])
    return check_selection(gpu_blocks, gpu_count, q_idx_bits, None, nb, k, scores=scores, bound=bound)


def _run_fp8_decode(w):
    L = _to(w.layers[0])
    b = DecodeBatch(w.n_q_heads, w.n_kv_heads, w.ctx_len)
    codes, scales = b.new_fp8_keys()
    b.pool_fp8(L.raw_idx_k, codes, scales)
    b.step_fp8(L.q_idx, L.q, L.k_cache, L.v_cache, codes, scales)
    st, det = b.device_status()
    assert st == 0, (st, det)
    return b, codes, scales


def _check_fp8_decode(w, b, codes, scales, rows=None, check_scores=True):
    Lh = w.layers[0]
    qib, qbits, kb, vb = bits(Lh.q_idx), bits(Lh.q), bits(Lh.k_cache), bits(Lh.v_cache)
    blocks, count = b.blocks.cpu().numpy(), b.count.cpu().numpy()
    sc = b.scores.cpu().numpy().astype(np.float64)
    out, lse = b.out.cpu(), b.lse.cpu().numpy()
    off = w.tok_off
    stats = dict(band=0, fp32=0)
    for s in (range(w.batch) if rows is None else rows):
        p = w.ctx_len[s]
        nb = p // 4
        pk = _pooled_oracle(w, s)
        lo, hi = b.blk_off[s].item(), b.blk_off[s + 1].item()
        vals, scl = _check_keys(codes[lo:hi], scales[lo:hi], pk)
        want = O.score_blocks_fp8(qib[s], vals[:nb], scl[:nb])
        bound = O.score_error_bound_fp8(qib[s], vals[:nb], scl[:nb])
        if check_scores:
            assert np.all(np.abs(sc[s, :nb] - want) <= bound + 1e-30), s
        n_band, n_fp32 = check_selection_fp8(blocks[s], count[s], qib[s], vals, scl, nb)
        stats["band"] += n_band
        stats["fp32"] += n_fp32
        ref = O.decode_query(p, qib[s], pk, qbits[s], kb[off[s]:off[s + 1]], vb[off[s]:off[s + 1]], w.n_kv_heads,
                             sel=blocks[s, :count[s]])
        check_attention(out[s], ref["out"])
        check_lse(lse[s], ref["lse"])
    print(f"{w.name}: {stats}")
    assert stats["fp32"] == 0, stats
    return stats


def test_decode_fp8_planted_ragged(cuda_lib):
    ctx = [5000, 2052, 70001, 4, 0, 2051, 12345]
    w = I.decode_workload("fp8_ragged", ctx, 1, 16, 2, "planted", seed=21)
    b, codes, scales = _run_fp8_decode(w)
    _check_fp8_decode(w, b, codes, scales)


def test_decode_fp8_gaussian_tiny(cuda_lib):
    w = I.tiny_decode(seed=2)
    b, codes, scales = _run_fp8_decode(w)
    _check_fp8_decode(w, b, codes, scales)


def test_decode_fp8_selection_overlaps_bf16(cuda_lib):
    # On the planted workload the FP8 keys change the selection only near the k-th score: the
    # oracle keeps 98.8% of the bf16 selection on this input (98.6-99.2% over seeds 22-24).
    ctx = [131072]
    w = I.decode_workload("fp8_vs_bf16", ctx, 1, 16, 2, "planted", seed=22)
    b8, _, _ = _run_fp8_decode(w)
    L = _to(w.layers[0])
    b = DecodeBatch(16, 2, ctx)
    pooled = b.new_pooled()
    b.pool(L.raw_idx_k, pooled)
    b.step(L.q_idx, L.q, L.k_cache, L.v_cache, pooled)
    s8 = set(b8.blocks[0, :512].cpu().tolist())
    s16 = set(b.blocks[0, :512].cpu().tolist())
    assert len(s8 & s16) >= 0.95 * 512


def test_million_decode_fp8_full_size_one_layer(cuda_lib):
    w = I.million_decode(n_layers=1)
    b, codes, scales = _run_fp8_decode(w)
    w.layers = [I.Layer(*(getattr(w.layers[0], f).cpu() for f in ("raw_idx_k", "q_idx", "q", "k_cache", "v_cache")))]
    _check_fp8_decode(w, b, codes, scales)


# ----------------------------------------------------------------------------- fused step, FP8 keys

def _run_fused_fp8(w, corrupt_newest=True):
    """Separate FP8 calls, then qsa_decode_step_fp8 on keys whose newest block was corrupted:
    the step must re-pool it, reproduce the separate path's selection exactly and attend."""
    L = _to(w.layers[0])
    b = DecodeBatch(w.n_q_heads, w.n_kv_heads, w.ctx_len)
    codes, scales = b.new_fp8_keys()
    b.pool_fp8(L.raw_idx_k, codes, scales)
    b.step_fp8(L.q_idx, L.q, L.k_cache, L.v_cache, codes, scales)
    assert b.device_status()[0] == 0
    sep = (b.blocks.clone(), b.count.clone(), b.out.clone())
    want_codes, want_scales = codes.clone(), scales.clone()
    if corrupt_newest:
        for s, p in enumerate(w.ctx_len):
            if p >= 4:
                r = b.blk_off[s].item() + p // 4 - 1
                codes[r] = 0x38       # 1.0
                scales[r] = 3.0
    b.blocks.fill_(-7)
    b.out.zero_()
    b.fused_step_fp8(L.raw_idx_k, codes, scales, L.q_idx, L.q, L.k_cache, L.v_cache)
    st = b.fused_status()
    assert st[0] == 0, st
    assert torch.equal(codes, want_codes)
    assert torch.equal(scales.view(torch.int32), want_scales.view(torch.int32))
    assert torch.equal(b.count, sep[1])
    assert torch.equal(b.blocks, sep[0]), "fused FP8 selection differs from the separate FP8 calls"
    assert (b.out.float() - sep[2].float()).abs().max().item() <= 2 ** -6
    return b, codes, scales


@pytest.mark.parametrize("case", ["planted_ragged", "tiny_sharp", "batched_short", "sharp16"])
def test_fused_step_fp8_small(cuda_lib, case):
    if case == "sharp16":
        # 16 query / 2 KV heads, sparse rows, N(0,1) Q/K/V
        w = I.decode_workload("fp8_fused_sharp16", [2052, 9001, 131072], 1, 16, 2, "planted_sharp", seed=34)
    elif case == "planted_ragged":
        w = I.decode_workload("fp8_fused_ragged", [5000, 2052, 70001, 4, 12345, 0, 3, 2051], 1, 16, 2, "planted",
                              seed=31)
    elif case == "tiny_sharp":
        w = I.tiny_decode(kind="sharp", seed=32)
    else:
        w = I.decode_workload("fp8_fused_short", I.batched_ctx_lens(short_draw=True), 1, 8, 2, "gaussian", seed=33)
    b, codes, scales = _run_fused_fp8(w)
    _check_fp8_decode(w, b, codes, scales)


def test_fused_step_fp8_million_full_size(cuda_lib):
    w = I.million_decode(n_layers=1)
    b, codes, scales = _run_fused_fp8(w)
    w.layers = [I.Layer(*(getattr(w.layers[0], f).cpu() for f in ("raw_idx_k", "q_idx", "q", "k_cache", "v_cache")))]
    _check_fp8_decode(w, b, codes, scales)


def test_fused_step_fp8_rejects_unpadded_keys(cuda_lib):
    w = I.tiny_decode(seed=4)
    L = _to(w.layers[0])
    b = DecodeBatch(8, 2, w.ctx_len)
    codes, scales = b.new_fp8_keys()
    with pytest.raises(qb.QsaError) as e:
        b.fused_step_fp8(L.raw_idx_k, codes[:-1], scales[:-1], L.q_idx, L.q, L.k_cache, L.v_cache)
    assert e.value.status == qb.QSA_ERR_INVALID_ARGUMENT
