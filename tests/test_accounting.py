"""Host accounting of algorithmic bytes/FLOPs pinned to the figures the pages print."""

import os

import pytest

from indexer_driven_sparse_gb300 import accounting as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.txt")
GOLDEN_GLM = os.path.join(os.path.dirname(__file__), "golden", "glm_page_figures.txt")
MiB = 1 << 20
GiB = 1 << 30
KiB = 1 << 10


def figs(path=GOLDEN):
    vals = {}
    with open(path, encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                vals[k] = float(v)
    return vals


def test_page_byte_figures():
    f = figs()
    assert A.kv_read_bytes(2048) == f["kv_bytes_per_layer"] == 4 * MiB
    assert 12 * A.kv_read_bytes(2048) == f["kv_bytes_per_step_12_layers"] == 48 * MiB
    assert A.pooled_scan_bytes(250_000) == f["pooled_bytes_per_layer_250000"]
    assert round(12 * A.pooled_scan_bytes(250_000) / MiB) == f["pooled_mib_per_step_12_layers"]
    vram, ram = A.per_token_memory(12)
    assert vram / KiB == f["vram_kib_per_token"]
    assert ram / KiB == f["ram_kib_per_token"]
    assert (vram + ram) / KiB == f["all_vram_kib_per_token"]
    # 204 GiB per naive 4096-token chunk: the padded selection is 2176 = 17 x 128 tokens
    assert round(A.naive_prefill_kv_bytes(4096, 2176, 12) / GiB) == f["naive_prefill_gib_per_chunk"]
    assert round(A.naive_prefill_kv_bytes(4096, 2048, 12) / GiB) != f["naive_prefill_gib_per_chunk"]


def test_attended_and_threshold():
    f = figs()
    assert max(p for p in range(5000) if A.visible_blocks(p) <= 512) == f["dense_limit_tokens"]
    for p in [2052, 2053, 2054, 2055, 1048320, 262144 + 17]:
        assert A.attended(p) == f["selected_tokens"] + p % 4 + 1
    for p in [0, 1, 3, 4, 2051]:
        assert A.attended(p) == p + 1


def test_workload_totals():
    # tiny decode: p = 4096, 8 query heads
    assert A.decode_layer_step_bytes([4096], 8) == 4_466_944
    # long decode: p = 131072, 16 query heads
    assert A.decode_layer_step_bytes([131072], 16) == 12_601_600
    # million-token decode
    assert A.decode_layer_step_bytes([1048320], 16) == 71_305_472
    assert A.pooled_scan_bytes(A.visible_blocks(1048320)) == 67_092_480
    # prefill chunk: 4096 queries at 262144 + i
    assert A.prefill_attention_flops(262144, 4096) == 8_398_848 * 16 * 1024
    assert A.prefill_score_flops(262144, 4096) == 256 * 270_530_560
    assert A.prefill_attention_flops(262144, 4096) / 1e9 == pytest.approx(137.6, abs=0.05)
    assert A.prefill_score_flops(262144, 4096) / 1e9 == pytest.approx(69.26, abs=0.01)


def test_fp8_scan_bytes():
    # 128 one-byte codes + a 4-byte scale per block: 132 of the bf16 key's 256 bytes
    assert A.score_scan_bytes_fp8([1048320]) == 262080 * 132 + 256
    assert A.score_scan_bytes_fp8([3]) == 256
    bf16 = A.score_scan_bytes([1048320]) - 256
    assert (A.score_scan_bytes_fp8([1048320]) - 256) / bf16 == 132 / 256


def test_fp8_layer_step_bytes():
    # the million-token step: the scan shrinks from 256 to 132 bytes per block, the rest is unchanged
    bf16 = A.decode_layer_step_bytes([1048320], 16)
    fp8 = A.decode_layer_step_bytes_fp8([1048320], 16)
    assert bf16 == 71_305_472
    assert bf16 - fp8 == 262080 * (256 - 132)


def test_fp8_kv_bytes():
    # an FP8 K or V row of one head: 256 code bytes + two fp32 scales = 264 of the bf16 row's 512
    assert A.kv_read_bytes_fp8(1, 1) == 2 * 264
    assert A.kv_read_bytes_fp8(2048) == 2048 * 2 * 2 * 264
    assert A.kv_read_bytes_fp8(2048) / A.kv_read_bytes(2048) == 264 / 512
    # the million-token step with FP8 K/V: only the gathered rows shrink
    bf16 = A.decode_layer_step_bytes([1048320], 16)
    assert bf16 - A.decode_layer_step_bytes_fp8kv([1048320], 16, False) == 2049 * 2 * 2 * (512 - 264)   # 2048 + own token
    assert A.decode_layer_step_bytes_fp8kv([1048320], 16, True) == \
        A.decode_layer_step_bytes_fp8([1048320], 16) - 2049 * 2 * 2 * (512 - 264)
    # a dense row (p = 10) attends p + 1 tokens
    assert A.decode_layer_step_bytes_fp8kv([10], 8, False) == 2 * 256 + 11 * 2 * 2 * 264 + 2 * 8 * 512 + 256


def test_fp8_kv_dequant_bytes():
    # one token of one head: K and V rows of 264 B read, of 512 B written
    assert A.kv_dequant_bytes_fp8(1, 1) == 2 * (264 + 512)
    # the prefill chunk's history and chunk (266,240 tokens, 2 KV heads)
    assert A.kv_dequant_bytes_fp8(262144 + 4096) == 266240 * 2 * 2 * 776


def test_glm_page_byte_figures():
    # the FP8 indexer key and the sparse-MLA row sizes against the footnotes that print them
    g = figs(GOLDEN_GLM)
    assert A.fp8_key_bytes() == g["indexer_key_bytes"]
    assert A.MLA_ROW_BYTES == g["mla_row_bytes"] and A.MLA_INDEX_BYTES == g["mla_row_index_bytes"]
    rows = int(g["mla_rows_per_query"])
    assert round(rows * (A.MLA_ROW_BYTES + A.MLA_INDEX_BYTES) / 1e6, 2) == g["mla_rows_mb"]
    assert A.sparse_mla_query_bytes(1, rows) - A.sparse_mla_query_bytes(0, rows) == g["mla_head_bytes"]
    assert A.sparse_mla_query_flops(1, 1) == g["mla_flops_per_row_head"]
    for h in (8, 64):
        b, f = A.sparse_mla_query_bytes(h, rows), A.sparse_mla_query_flops(h, rows)
        assert round(b / 1e6, 2) == g[f"mla_{h}_heads_mb"]
        assert round(f / 1e6, 1 if h == 8 else 0) == g[f"mla_{h}_heads_mflops"]
        assert round(f / b) == g[f"mla_{h}_heads_intensity"]
    per_token = 78 * A.MLA_ROW_BYTES + 21 * A.fp8_key_bytes() + 788
    assert per_token == g["token_bytes_total"]
    assert round(per_token * (1 << 20) / (1 << 30), 1) == g["million_token_gib"]
    assert round(989e12 / 4.8e12) == g["h200_ridge_flops_per_byte"]
