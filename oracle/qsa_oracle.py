"""fp64 CPU oracle of indexer-driven sparse attention (QSA-style).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs, never by the library. It shares no
code with the CUDA path and is written from the pages' statement of the method:

* "3090x3で 314 万コンテキスト; KVキャッシュをホストRAMに置けるアーキテクチャの偉大さ"
  (minamism.com, QSA KV offload), sections "なぜ" (indexer_budget 2048,
  indexer_compress_ratio 4, dense up to 4*block_topk+3 = 2051 tokens, exactly
  2048 tokens read per generated token), "カーネルを書き換えずに済む" (K/V
  addressing ``(tok*n_kv_heads + kv_head)*head_dim + d``), "VRAM に残す必要があるもの"
  (pooled key = keys grouped per 4-token block, 128 x bf16) and "ちなみにこの欠点"
  (prefill walks the history interval by interval with a softmax merge).
* "GLM-5.3 最適化 第2部：16基のH200上でのPCP、DCP、およびHybrid HiSparse" (vLLM blog),
  section "DCP: KVキャッシュもシャーディングする": partial attention results over
  disjoint key shards are combined by log-sum-exp.
* "125B MoE を 3090 3 枚で運用する vLLM 最適化編", section 3.3: top-k ties go to the
  lower id.

Everything is computed in float64 from the bf16 bit patterns. Library primitives
(numpy matmul, lexsort, exp, log) serve as steps; nothing is blocked, fused or
reordered beyond the definitions below. Readings of points the pages leave open
(pooling = mean with one round-to-nearest-even to bf16, visibility of the query's
own partial block, GQA head grouping, softmax scale 1/sqrt(head_dim), ascending
selection order) are stated beside the function that takes them.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, brute force, library routines, the pages' own byte figures).
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "COMPRESS_RATIO", "INDEXER_BUDGET", "BLOCK_TOPK", "DENSE_LIMIT",
    "bf16_bits_to_f64", "f64_to_bf16_bits", "pool_keys", "visible_blocks",
    "score_blocks", "kth_score", "select_blocks", "attended_tokens",
    "attend_partial", "lse_merge", "attend", "decode_query",
    "interval_walk_query", "score_error_bound",
    "E4M3_MAX", "e4m3_round", "quantize_pooled_fp8", "score_blocks_fp8",
    "score_error_bound_fp8", "MLA_LATENT", "MLA_ROPE", "MLA_GROUP", "quantize_mla_rows_fp8",
    "sparse_mla_attend", "MLA_ROW_BYTES", "e4m3_value", "mla_rows_from_bytes",
    "KV_GROUP", "e4m3_code", "quantize_kv_fp8", "dequantize_kv_fp8",
]

# indexer_compress_ratio and indexer_budget from the model's text_config
# (page "3090x3で 314 万コンテキスト", section "なぜ").
COMPRESS_RATIO = 4
INDEXER_BUDGET = 2048
BLOCK_TOPK = INDEXER_BUDGET // COMPRESS_RATIO        # 512 blocks
DENSE_LIMIT = 4 * BLOCK_TOPK + 3                     # 2051 tokens


# --------------------------------------------------------------------------- bf16

def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values (bf16 is the top half of fp32)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 to bf16 with round-to-nearest, ties-to-even, in one step.

    bf16 keeps 8 significant bits and fp32's exponent range: on [2^e, 2^(e+1))
    the spacing is 2^(e-7), and below 2^-126 (subnormals) it is 2^-133.
    ``x / spacing`` is exact (a power-of-two scaling), ``np.rint`` rounds half to
    even, and the rounded value is exactly representable in fp32 and bf16.
    Magnitudes that round to 2^128 or above become infinity; NaN becomes 0x7FC0.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint16)
    nan = np.isnan(x)
    inf = np.isinf(x)
    fin = ~(nan | inf)
    xf = np.where(fin, x, 0.0)
    _, exp = np.frexp(xf)                        # |x| in [2^(exp-1), 2^exp)
    e = np.maximum(exp - 1, -126)
    spacing = np.ldexp(1.0, e - 7)
    r = np.rint(xf / spacing) * spacing
    overflow = fin & (np.abs(r) >= 2.0 ** 128)
    r = np.where(overflow, 0.0, r)
    f32 = r.astype(np.float32)                   # exact: r has <= 8 significant bits
    bits = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    sign = np.signbit(x)
    bits = np.where(overflow | inf, np.where(sign, 0xFF80, 0x7F80), bits).astype(np.uint16)
    bits = np.where(nan, 0x7FC0, bits).astype(np.uint16)
    return bits


# --------------------------------------------------------------------------- pooling

def pool_keys(raw_bits: np.ndarray) -> np.ndarray:
    """Pooled indexer keys of every complete 4-token block.

    raw_bits: [T, idx_dim] bf16 bits -> [T // 4, idx_dim] bf16 bits.
    Page "3090x3で 314 万コンテキスト", "VRAM に残す必要があるもの": the pooled key
    groups the keys of one block (ratio 4) and is stored as 128 x bf16.
    Reading: the grouping is the mean of the block's four raw keys, computed in
    float64 as ((k0 + k1) + k2) + k3 times 1/4, then rounded once to bf16 (RNE).
    A trailing partial block is not pooled.
    """
    raw = bf16_bits_to_f64(raw_bits)
    nb = raw.shape[0] // COMPRESS_RATIO
    r = raw[: nb * COMPRESS_RATIO].reshape(nb, COMPRESS_RATIO, raw.shape[1])
    s = ((r[:, 0] + r[:, 1]) + r[:, 2]) + r[:, 3]
    return f64_to_bf16_bits(s * 0.25)


def visible_blocks(p: int) -> int:
    """Number of pooled blocks a query with ``p`` history tokens scores.

    Reading of "dense until 4*block_topk+3 = 2051" (section "なぜ"): the query
    sits at token index p; only blocks that end strictly before its own block
    are pooled and scored (nb = floor(p/4)); the tokens of its own block up to
    and including itself (4*nb .. p) are always attended. Then the history is
    read in full exactly while nb <= 512, i.e. p <= 2051.
    """
    if p < 0:
        raise ValueError("p must be >= 0")
    return p // COMPRESS_RATIO


# --------------------------------------------------------------------------- FP8 indexer keys

# FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; the all-ones exponent with
# mantissa 7 is NaN, so the largest finite value is 1.75 * 2^8): the "128 FP8 + 4 B scale"
# indexer key of the page "GLM-5.3 最適化 第2部" (footnote on the indexer cache).
E4M3_MAX = 448.0


def e4m3_round(x) -> np.ndarray:
    """Nearest E4M3 value of each input (ties to the even mantissa), saturating at +-448.

    In the binade [2^k, 2^(k+1)) the E4M3 values are 2^(k-3) apart (3 mantissa bits); below
    the smallest normal 2^-6 the subnormals are 2^-9 apart. The quotient by the spacing is
    exact in float64, so rint (half to even) gives the round-to-nearest-even value.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(np.where(a > 0, a, 1.0))           # a = m 2^e, m in [0.5, 1): binade k = e - 1
    k = np.maximum(e - 1, -6)
    q = np.ldexp(1.0, k - 3)
    r = np.minimum(np.rint(a / q) * q, E4M3_MAX)
    return np.copysign(r, x)


def quantize_pooled_fp8(pooled_bits):
    """Per pooled block: scale = max |key| / 448 and codes = E4M3(key / scale).

    Reading (the pages give the format, not the arithmetic): the scale and the quotient are
    single float32 operations (an IEEE division rounded to nearest), the code is the
    nearest E4M3 value of the float32 quotient; an all-zero key has scale 0 and zero codes.
    Returns (values [nb, idx_dim] float64 of the codes, scales [nb] float32).
    """
    pk = bf16_bits_to_f64(pooled_bits)
    if pk.ndim == 1:
        pk = pk[None, :]
    amax = np.abs(pk).max(axis=1) if pk.shape[0] else np.zeros(0)
    scale = (amax.astype(np.float32) / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    quot = (pk.astype(np.float32) / safe[:, None]).astype(np.float32)
    vals = e4m3_round(quot)
    vals[scale == 0] = 0.0
    return vals, scale


def score_blocks_fp8(q_idx_bits: np.ndarray, vals: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Indexer score against FP8 keys: s_b = scale_b * (q_idx . codes_b), in float64."""
    q = bf16_bits_to_f64(q_idx_bits)
    if vals.shape[0] == 0:
        return np.zeros(0, dtype=np.float64)
    return (vals @ q) * scales.astype(np.float64)


def score_error_bound_fp8(q_idx_bits: np.ndarray, vals: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Worst-case error of an FP8-key score computed as fl(scale * fl(sum_d q_d c_d)) in fp32.

    A bf16 value times an E4M3 value is exact in fp32 (8 + 4 significant bits), so the sum
    errs by at most gamma_n * sum_d |q_d c_d| (Higham ch. 3), and the final product by one
    rounding of the result, u |scale * s~|. Used only to grade GPU scores and label swaps.
    """
    q = np.abs(bf16_bits_to_f64(q_idx_bits))
    if vals.shape[0] == 0:
        return np.zeros(0, dtype=np.float64)
    n = q.shape[0]
    u = 2.0 ** -24
    gamma = n * u / (1.0 - n * u)
    a = np.abs(vals) @ q
    d = np.abs(vals @ bf16_bits_to_f64(q_idx_bits))
    sc = scales.astype(np.float64)
    return sc * (gamma * a + u * (d + gamma * a))


# --------------------------------------------------------------------------- scoring

def score_blocks(q_idx_bits: np.ndarray, pooled_bits: np.ndarray) -> np.ndarray:
    """Indexer score of every pooled block: s_b = q_idx . pooled_b, in float64.

    q_idx_bits: [idx_dim]; pooled_bits: [nb, idx_dim]. Reading: one indexer query
    of width idx_dim per query token and a plain dot product; the pages do not
    give the indexer's weights or activation, and any positive scale leaves the
    ranking unchanged.
    """
    q = bf16_bits_to_f64(q_idx_bits)
    pk = bf16_bits_to_f64(pooled_bits)
    if pk.shape[0] == 0:
        return np.zeros(0, dtype=np.float64)
    return pk @ q


def score_error_bound(q_idx_bits: np.ndarray, pooled_bits: np.ndarray) -> np.ndarray:
    """Worst-case error of an fp32-accumulated dot product of bf16 operands.

    Products of two bf16 values are exact in fp32, so the only error is the
    n-1 additions: |fl(s) - s| <= gamma_n * sum_d |q_d p_d|, gamma_n = n u/(1-n u),
    u = 2^-24 (standard forward bound for recursive summation, Higham ch. 3).
    Used only to label selection swaps as "within fp32 bound".
    """
    q = np.abs(bf16_bits_to_f64(q_idx_bits))
    pk = np.abs(bf16_bits_to_f64(pooled_bits))
    n = q.shape[0]
    u = 2.0 ** -24
    gamma = n * u / (1.0 - n * u)
    return gamma * (pk @ q)


# --------------------------------------------------------------------------- top-k

def _rank_order(scores: np.ndarray) -> np.ndarray:
    """Block ids sorted best first: score descending, then lower id first.

    NaN scores rank below every number (reading: inputs should be finite).
    """
    s = np.asarray(scores, dtype=np.float64)
    isnan = np.isnan(s)
    key = np.where(isnan, 0.0, -s)
    ids = np.arange(s.shape[0])
    # np.lexsort sorts by the last key first.
    return np.lexsort((ids, key, isnan))


def select_blocks(scores: np.ndarray, k: int = BLOCK_TOPK) -> np.ndarray:
    """Fixed-budget block selection: the min(k, nb) best blocks, ids ascending.

    Section "なぜ": beyond 2051 tokens the indexer keeps exactly 2048 tokens
    (k = 512 blocks); below that every block is kept. Ties go to the lower
    block id (page "125B MoE ...", section 3.3: the lower id wins equal keys).
    Reading: the output is sorted by block id (a canonical set).
    """
    n = len(scores)
    kk = min(k, n)
    return np.sort(_rank_order(scores)[:kk]).astype(np.int64)


def kth_score(scores: np.ndarray, k: int = BLOCK_TOPK) -> float:
    """Score of the last block the selection keeps (nan if nothing is kept)."""
    n = len(scores)
    kk = min(k, n)
    if kk == 0:
        return float("nan")
    return float(np.asarray(scores, dtype=np.float64)[_rank_order(scores)[kk - 1]])


def attended_tokens(p: int, sel: np.ndarray) -> np.ndarray:
    """Token set J a query at position p attends: the selected blocks' tokens
    plus its own block from 4*nb up to and including p. Sorted ascending.
    """
    nb = visible_blocks(p)
    sel = np.asarray(sel, dtype=np.int64)
    if sel.size and (sel.min() < 0 or sel.max() >= nb):
        raise ValueError("selected block outside the visible history")
    from_blocks = (sel[:, None] * COMPRESS_RATIO + np.arange(COMPRESS_RATIO)[None, :]).reshape(-1)
    tail = np.arange(COMPRESS_RATIO * nb, p + 1, dtype=np.int64)
    return np.sort(np.concatenate([from_blocks, tail]))


# --------------------------------------------------------------------------- attention

def attend_partial(q: np.ndarray, k: np.ndarray, v: np.ndarray, tokens: np.ndarray,
                   n_kv_heads: int, scale: float):
    """Unnormalised softmax partial of every query head over a token subset.

    q: [Hq, D] float64; k, v: [T, Hkv, D] float64 (token-major, as the gather
    kernel addresses ``(tok*n_kv_heads + kv_head)*head_dim + d``, section
    "カーネルを書き換えずに済む"). Query head h reads KV head h // (Hq/Hkv)
    (reading: contiguous GQA groups). Returns (m [Hq], l [Hq], acc [Hq, D]) with
    m = max logit, l = sum exp(logit - m), acc = sum exp(logit - m) v. An empty
    subset gives m = -inf, l = 0, acc = 0.
    """
    hq, d = q.shape
    g = hq // n_kv_heads
    m = np.full(hq, -np.inf)
    l = np.zeros(hq)
    acc = np.zeros((hq, d))
    tokens = np.asarray(tokens, dtype=np.int64)
    if tokens.size == 0:
        return m, l, acc
    for h in range(hq):
        kv = h // g
        kt = k[tokens, kv, :]
        vt = v[tokens, kv, :]
        logits = (kt @ q[h]) * scale
        m[h] = logits.max()
        w = np.exp(logits - m[h])
        l[h] = w.sum()
        acc[h] = w @ vt
    return m, l, acc


def lse_merge(parts):
    """Combine partials over disjoint token subsets by log-sum-exp.

    Page "GLM-5.3 最適化 第2部", section "DCP": each shard attends its own keys and
    the partial results are merged by log-sum-exp. With parts (m_i, l_i, acc_i):
    m = max m_i, l = sum l_i e^(m_i - m), out = sum acc_i e^(m_i - m) / l,
    lse = m + ln l.
    """
    ms = np.stack([p[0] for p in parts])          # [S, Hq]
    ls = np.stack([p[1] for p in parts])
    accs = np.stack([p[2] for p in parts])        # [S, Hq, D]
    m = ms.max(axis=0)
    safe_m = np.where(np.isfinite(m), m, 0.0)
    w = np.where(np.isfinite(ms), np.exp(ms - safe_m[None, :]), 0.0)
    l = (ls * w).sum(axis=0)
    acc = (accs * w[:, :, None]).sum(axis=0)
    with np.errstate(invalid="ignore", divide="ignore"):
        out = acc / l[:, None]
        lse = safe_m + np.log(l)
    return out, lse


def attend(q, k, v, tokens, n_kv_heads: int, scale: float):
    """Normalised softmax attention over ``tokens``: returns (out [Hq, D], lse [Hq])."""
    return lse_merge([attend_partial(q, k, v, tokens, n_kv_heads, scale)])


# --------------------------------------------------------------------------- one query

def decode_query(p: int, q_idx_bits, pooled_bits, q_bits, k_bits, v_bits, n_kv_heads: int,
                 scale: float | None = None, k_blocks: int = BLOCK_TOPK, sel=None):
    """The whole path for one query token at position p of its sequence.

    pooled_bits: the sequence's pooled keys (at least floor(p/4) rows); q_bits:
    [Hq, D]; k_bits / v_bits: the sequence's K/V [>= p+1, Hkv, D] (bf16 bits or
    already-float64 arrays). Steps: score the visible blocks, keep the top
    min(512, nb), attend the selected tokens plus the query's own block.
    ``sel`` overrides the selection (to grade attention on another selection).
    Returns dict(scores, sel, tokens, out, lse).
    """
    nb = visible_blocks(p)
    scores = score_blocks(q_idx_bits, np.asarray(pooled_bits)[:nb])
    if sel is None:
        sel = select_blocks(scores, k_blocks)
    tokens = attended_tokens(p, sel)
    q = _as_f64(q_bits)
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kk = _rows_f64(k_bits, tokens)
    vv = _rows_f64(v_bits, tokens)
    # attend over the compacted rows (row j of kk is token tokens[j])
    out, lse = attend(q, kk, vv, np.arange(tokens.size), n_kv_heads, scale)
    return dict(scores=scores, sel=np.asarray(sel, dtype=np.int64), tokens=tokens, out=out, lse=lse)


# --------------------------------------------------------------------------- sparse MLA (MQA form)

# "GLM-5.3 最適化 第2部" (footnote 1): a sparse-MLA query reads 2,048 selected rows of an FP8
# KV cache; QK runs over 576 dims and PV over 512, and one row serves all 64 heads. Readings
# (the page gives sizes only): the row is a 512-wide latent that is also the value, plus 64
# rotary dims that only enter the key; the latent is stored as E4M3 codes in 4 groups of 128
# with one fp32 scale each (512 + 16 bytes) and the rotary part as bf16 (128 bytes): 656 B.
MLA_LATENT = 512
MLA_ROPE = 64
MLA_GROUP = 128


def quantize_mla_rows_fp8(latent_bits, rope_bits):
    """FP8 rows of the sparse-MLA cache: each 128-dim group of the bf16 latent quantised as an
    FP8 indexer key is (scale = group max|x| / 448, codes = E4M3(x / scale), fp32 divisions);
    the rotary dims kept in bf16. Returns (latent [n, 512] float64 as the codes and scales
    represent it, rope [n, 64] float64, scales [n, 4] float32)."""
    lat = np.asarray(latent_bits)
    n = lat.shape[0]
    vals, scl = quantize_pooled_fp8(lat.reshape(n * (MLA_LATENT // MLA_GROUP), MLA_GROUP))
    deq = vals * scl.astype(np.float64)[:, None]
    return (deq.reshape(n, MLA_LATENT), bf16_bits_to_f64(np.asarray(rope_bits)).reshape(n, MLA_ROPE),
            scl.reshape(n, MLA_LATENT // MLA_GROUP))


MLA_ROW_BYTES = MLA_LATENT + 4 * (MLA_LATENT // MLA_GROUP) + 2 * MLA_ROPE   # 656


def e4m3_value(code) -> np.ndarray:
    """Value of E4M3 byte codes from the bit layout: sign, 4 exponent bits (bias 7), 3
    mantissa bits; exponent 0 is subnormal (m/8 * 2^-6); 0x7F and 0xFF are NaN."""
    c = np.asarray(code, dtype=np.int64)
    s, e, m = c >> 7, (c >> 3) & 15, c & 7
    v = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return np.where(s == 1, -v, v)


def mla_rows_from_bytes(row_bytes) -> tuple:
    """Decode FP8 MLA rows as stored (reading of the 656-byte row): bytes 0..511 the latent's
    E4M3 codes, 512..527 four little-endian fp32 scales (one per 128 latent dims), 528..655
    the 64 rotary dims as bf16. Returns (latent [n, 512], rope [n, 64]) in float64, the
    latent exactly code x scale."""
    r = np.ascontiguousarray(np.asarray(row_bytes, dtype=np.uint8)).reshape(-1, MLA_ROW_BYTES)
    n = r.shape[0]
    codes = e4m3_value(r[:, :MLA_LATENT])
    scales = r[:, MLA_LATENT:MLA_LATENT + 16].copy().view("<f4").astype(np.float64)
    latent = (codes.reshape(n, 4, MLA_GROUP) * scales[:, :, None]).reshape(n, MLA_LATENT)
    rope = bf16_bits_to_f64(r[:, MLA_LATENT + 16:].copy().view("<u2"))
    return latent, rope


# --------------------------------------------------------------------------- FP8 K/V rows

# "GLM-5.3 最適化 第2部" (footnote 1) stores the attended KV rows as FP8: E4M3 codes in groups
# of 128 dims, one fp32 scale per group (the 656-byte MLA row above; the indexer key of
# footnote 3 is the same 128 codes + 4 B scale). Reading for the GQA cache of the QSA path
# (the pages give no separate format for it): each token's K row and V row of each KV head
# (head_dim 256) is quantised the same way, two groups of 128 dims, and stored as a plane of
# codes [T, Hkv, 256] (uint8) beside a plane of scales [T, Hkv, 2] (fp32). Attention then
# reads the value code x scale of every element in place of the bf16 value.
KV_GROUP = 128


def e4m3_code(values) -> np.ndarray:
    """Byte code of E4M3 values (each exactly representable, |v| <= 448): bit 7 the sign,
    bits 6..3 the exponent field (bias 7; 0 for zero and subnormals), bits 2..0 the mantissa.
    A normal value v = (1 + m/8) 2^(e-7); a subnormal v = (m/8) 2^-6. Negative zero is 0x80.
    Raises ValueError for a value the format cannot hold exactly."""
    v = np.asarray(values, dtype=np.float64)
    a = np.abs(v)
    if np.any(~np.isfinite(a)) or np.any(a > E4M3_MAX):
        raise ValueError("value outside the E4M3 range")
    _, e = np.frexp(np.where(a > 0, a, 1.0))           # a = f 2^e, f in [0.5, 1): a in [2^(e-1), 2^e)
    normal = a >= 2.0 ** -6
    field = np.where(normal, e - 1 + 7, 0)
    mant = np.where(normal, (a / np.ldexp(1.0, e - 1) - 1.0) * 8.0, a / 2.0 ** -9)
    if np.any(mant != np.rint(mant)) or np.any(mant > 7):
        raise ValueError("value not exactly representable in E4M3")
    code = (np.signbit(v).astype(np.int64) << 7) | (field.astype(np.int64) << 3) | mant.astype(np.int64)
    return code.astype(np.uint8)


def quantize_kv_fp8(kv_bits):
    """FP8 K (or V) cache rows from bf16 rows [..., D] (D a multiple of 128): every 128-dim
    group quantised as an FP8 indexer key is (scale = group max|x| / 448 and codes =
    E4M3(x / scale), fp32 divisions, nearest-even codes; an all-zero group has scale 0 and
    zero codes). Returns (codes uint8 [..., D] as stored, scales float32 [..., D / 128])."""
    x = np.asarray(kv_bits)
    d = x.shape[-1]
    if d % KV_GROUP:
        raise ValueError("row length must be a multiple of 128")
    groups = x.reshape(-1, KV_GROUP)
    vals, scl = quantize_pooled_fp8(groups) if groups.shape[0] else (np.zeros((0, KV_GROUP)), np.zeros(0, np.float32))
    return e4m3_code(vals).reshape(x.shape), scl.reshape(x.shape[:-1] + (d // KV_GROUP,))


def dequantize_kv_fp8(codes, scales) -> np.ndarray:
    """Values of FP8 K/V rows: element d of a row is e4m3_value(code_d) x scale[d // 128],
    exact in float64. codes [..., D] uint8, scales [..., D / 128]; returns float64 [..., D]."""
    c = np.asarray(codes, dtype=np.uint8)
    s = np.asarray(scales, dtype=np.float64)
    d = c.shape[-1]
    v = e4m3_value(c).reshape(c.shape[:-1] + (d // KV_GROUP, KV_GROUP))
    return (v * s[..., None]).reshape(c.shape)


def sparse_mla_attend(q_bits, latent: np.ndarray, rope: np.ndarray, rows, scale: float | None = None):
    """One decode query of sparse MLA in its MQA form: head h attends the selected rows j with
    logit scale * (q_h[:512] . latent_j + q_h[512:] . rope_j) and output sum_j softmax_j latent_j.
    q_bits [H, 576] (bf16 bits or float); latent [n, 512], rope [n, 64] float64. The scale
    defaults to 1/sqrt(576) (the pages do not give it). Returns (out [H, 512], lse [H]);
    no rows give zeros and -inf."""
    q = _as_f64(q_bits)
    rows = np.asarray(rows, dtype=np.int64)
    if scale is None:
        scale = 1.0 / np.sqrt(MLA_LATENT + MLA_ROPE)
    if rows.size == 0:
        return np.zeros((q.shape[0], MLA_LATENT)), np.full(q.shape[0], -np.inf)
    k = np.concatenate([latent[rows], rope[rows]], axis=1)
    v = latent[rows]
    logits = (q @ k.T) * scale
    m = logits.max(axis=1)
    w = np.exp(logits - m[:, None])
    l = w.sum(axis=1)
    return (w @ v) / l[:, None], m + np.log(l)


def interval_walk_query(p: int, sel, q_bits, k_bits, v_bits, n_kv_heads: int,
                        interval_tokens: int, scale: float | None = None):
    """Prefill evaluation order for one query: walk the history in fixed
    intervals and merge the softmax partial of each interval into a running
    result (page "3090x3で 314 万コンテキスト", section "ちなみにこの欠点"). The
    result must equal :func:`decode_query` on the same selection; the oracle
    keeps this only to pin that equivalence.
    """
    tokens = attended_tokens(p, sel)
    q = _as_f64(q_bits)
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    hq = q.shape[0]
    running = (np.full(hq, -np.inf), np.zeros(hq), np.zeros((hq, d)))
    for start in range(0, p + 1, interval_tokens):
        inside = tokens[(tokens >= start) & (tokens < start + interval_tokens)]
        if inside.size == 0:
            continue
        part = attend_partial(q, _rows_f64(k_bits, inside), _rows_f64(v_bits, inside),
                              np.arange(inside.size), n_kv_heads, scale)
        out, lse = lse_merge([running, part])
        # re-express the merged pair as an unnormalised partial with m = lse, l = 1
        running = (lse, np.ones(hq), out)
    return lse_merge([running])


def _as_f64(a):
    a = np.asarray(a)
    return bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def _rows_f64(a, rows):
    a = np.asarray(a)
    sub = a[np.asarray(rows, dtype=np.int64)]
    return bf16_bits_to_f64(sub) if a.dtype == np.uint16 else sub.astype(np.float64)
