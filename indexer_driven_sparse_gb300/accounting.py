"""Algorithmic bytes and FLOPs of the hot path (host bookkeeping for rooflines).

These are the bytes the method must move at least once and the FLOPs it must
execute, independent of how a kernel tiles them. They are checked against the
figures printed in "3090x3で 314 万コンテキスト; KVキャッシュをホストRAMに置ける
アーキテクチャの偉大さ": section "なぜ" (4 MiB of K/V per layer per generated
token at K_pad ~ 2048, 48 MiB per 12-layer step), section "VRAM に残す必要があるもの"
(250,000 blocks x 128 x 2 B = 64 MB per layer, 732 MiB per 12-layer step; 0.75
KiB/token in VRAM, 27.00 KiB/token in RAM) and section "ちなみにこの欠点" (204 GiB
per naive 4096-token prefill chunk). The FP8 indexer key and the sparse-MLA row sizes are
checked against the footnotes of "GLM-5.3 最適化 第2部：16基のH200上でのPCP、DCP、および
Hybrid HiSparse" (132-byte indexer keys; 656-byte FP8 MLA rows with a 4-byte index; per-head
query/output bytes and FLOPs per row).
"""

from __future__ import annotations

BF16 = 2
RATIO = 4
BLOCK_TOPK = 512
FP8_KEY_SCALE_BYTES = 4          # one fp32 scale per FP8 indexer key
MLA_LATENT = 512                 # sparse MLA: latent (value) width shared by all heads
MLA_ROPE = 64                    # rotary part of the key; QK runs over 512 + 64 = 576 dims
MLA_ROW_BYTES = MLA_LATENT + 4 * 4 + MLA_ROPE * BF16   # FP8 latent, 4 fp32 scales, bf16 rope = 656
MLA_INDEX_BYTES = 4              # int32 id of a selected row


def visible_blocks(p: int) -> int:
    """Blocks scored by a query with p history tokens (complete blocks before its own)."""
    return p // RATIO


def attended(p: int, k_blocks: int = BLOCK_TOPK) -> int:
    """Tokens a query at position p attends: 4*min(k, nb) + its own block up to itself."""
    nb = visible_blocks(p)
    return RATIO * min(k_blocks, nb) + (p - RATIO * nb + 1)


def kv_read_bytes(n_tokens: int, n_kv_heads: int = 2, head_dim: int = 256) -> int:
    """K and V bytes of n_tokens tokens over all KV heads (bf16)."""
    return n_tokens * head_dim * BF16 * 2 * n_kv_heads


def pooled_scan_bytes(n_blocks: int, idx_dim: int = 128) -> int:
    """Bytes of pooled keys read by one query's indexer scan."""
    return n_blocks * idx_dim * BF16


def decode_layer_step_bytes(ctx_lens, n_q_heads: int, n_kv_heads: int = 2, head_dim: int = 256,
                            idx_dim: int = 128) -> int:
    """Algorithmic HBM bytes of one decode layer-step for a batch of queries:
    the pooled-key scan, the gathered K/V (selected blocks + own block), the
    query, the indexer query and the output. Scores and selections are not
    counted (they are produced and consumed on chip in the ideal design)."""
    total = 0
    for p in ctx_lens:
        total += pooled_scan_bytes(visible_blocks(p), idx_dim)
        total += kv_read_bytes(attended(p), n_kv_heads, head_dim)
        total += 2 * n_q_heads * head_dim * BF16 + idx_dim * BF16
    return total


def score_scan_bytes(ctx_lens, idx_dim: int = 128) -> int:
    """Bytes the scoring scan must read (pooled keys + indexer queries)."""
    return sum(pooled_scan_bytes(visible_blocks(p), idx_dim) + idx_dim * BF16 for p in ctx_lens)


def fp8_key_bytes(idx_dim: int = 128) -> int:
    """Bytes of one FP8 indexer key: idx_dim one-byte codes and an fp32 scale."""
    return idx_dim + FP8_KEY_SCALE_BYTES


def score_scan_bytes_fp8(ctx_lens, idx_dim: int = 128) -> int:
    """Bytes the scan over FP8 indexer keys must read: per visible block 128 one-byte codes
    and a 4-byte scale (the "128 FP8 + 4 B scale" key of "GLM-5.3 最適化 第2部", footnote on
    the indexer cache), plus the bf16 indexer query."""
    return sum(visible_blocks(p) * fp8_key_bytes(idx_dim) + idx_dim * BF16 for p in ctx_lens)


def decode_layer_step_bytes_fp8(ctx_lens, n_q_heads: int, n_kv_heads: int = 2, head_dim: int = 256,
                                idx_dim: int = 128) -> int:
    """decode_layer_step_bytes with the scan over FP8 indexer keys (idx_dim + 4 bytes per block)."""
    total = 0
    for p in ctx_lens:
        total += visible_blocks(p) * fp8_key_bytes(idx_dim)
        total += kv_read_bytes(attended(p), n_kv_heads, head_dim)
        total += 2 * n_q_heads * head_dim * BF16 + idx_dim * BF16
    return total


def kv_read_bytes_fp8(n_tokens: int, n_kv_heads: int = 2, head_dim: int = 256, group: int = 128) -> int:
    """K and V bytes of n_tokens tokens over all KV heads as FP8 rows: one code byte per dim and
    one fp32 scale per 128-dim group (the KV-row format of "GLM-5.3 最適化 第2部", footnote 1)."""
    return n_tokens * (head_dim + 4 * (head_dim // group)) * 2 * n_kv_heads


def decode_layer_step_bytes_fp8kv(ctx_lens, n_q_heads: int, fp8_keys: bool, n_kv_heads: int = 2,
                                  head_dim: int = 256, idx_dim: int = 128) -> int:
    """decode_layer_step_bytes with FP8 K/V rows, over bf16 or FP8 indexer keys."""
    total = 0
    for p in ctx_lens:
        nb = visible_blocks(p)
        total += nb * fp8_key_bytes(idx_dim) if fp8_keys else pooled_scan_bytes(nb, idx_dim)
        total += kv_read_bytes_fp8(attended(p), n_kv_heads, head_dim)
        total += 2 * n_q_heads * head_dim * BF16 + idx_dim * BF16
    return total


def kv_dequant_bytes_fp8(n_tokens: int, n_kv_heads: int = 2, head_dim: int = 256) -> int:
    """HBM bytes of dequantising n_tokens tokens of FP8 K and V rows into bf16 rows: the FP8
    rows read once (kv_read_bytes_fp8) and the bf16 rows written once."""
    return kv_read_bytes_fp8(n_tokens, n_kv_heads, head_dim) + n_tokens * n_kv_heads * 2 * head_dim * BF16


def prefill_attention_flops(p0: int, n_chunk: int, n_q_heads: int = 16, head_dim: int = 256) -> int:
    """QK^T + PV FLOPs over each chunk query's own selection (2 per multiply-add)."""
    return sum(attended(p0 + i) for i in range(n_chunk)) * n_q_heads * head_dim * 2 * 2


def prefill_score_flops(p0: int, n_chunk: int, idx_dim: int = 128) -> int:
    """Indexer FLOPs of a prefill chunk: every query scores all its visible blocks."""
    return sum(visible_blocks(p0 + i) for i in range(n_chunk)) * idx_dim * 2


def prefill_kv_bytes(p0: int, n_chunk: int, n_kv_heads: int = 2, head_dim: int = 256) -> int:
    """K/V bytes when the history is read once (interval walk)."""
    return kv_read_bytes(p0 + n_chunk, n_kv_heads, head_dim)


def naive_prefill_kv_bytes(n_chunk: int, k_pad: int, n_layers: int, n_kv_heads: int = 2,
                           head_dim: int = 256) -> int:
    """K/V bytes when every chunk query gathers its own padded selection."""
    return n_chunk * kv_read_bytes(k_pad, n_kv_heads, head_dim) * n_layers


def per_token_memory(n_layers: int, n_kv_heads: int = 2, head_dim: int = 256, idx_dim: int = 128):
    """(pooled-key bytes, K/V + raw indexer-key bytes) per token over all layers."""
    pooled = n_layers * idx_dim * BF16 // RATIO
    host = n_layers * (kv_read_bytes(1, n_kv_heads, head_dim) + idx_dim * BF16)
    return pooled, host


def sparse_mla_query_bytes(n_heads: int, rows: int = 2048) -> int:
    """Bytes one sparse-MLA decode query moves: its selected FP8 rows with their int32 ids,
    plus each head's bf16 query (576 dims) and output (512 dims)."""
    return rows * (MLA_ROW_BYTES + MLA_INDEX_BYTES) + n_heads * (MLA_LATENT + MLA_ROPE + MLA_LATENT) * BF16


def sparse_mla_query_flops(n_heads: int, rows: int = 2048) -> int:
    """FLOPs of one sparse-MLA decode query: QK over 576 dims and PV over 512 dims per row and head."""
    return rows * n_heads * 2 * ((MLA_LATENT + MLA_ROPE) + MLA_LATENT)
