"""The C-ABI library loads, exports every declared symbol and validates arguments on
the host (no kernel is launched and no GPU is needed)."""

import ctypes as C
import os
import re

import pytest

from indexer_driven_sparse_gb300 import binding as qb
from indexer_driven_sparse_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qb.load()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()
            names |= set(re.findall(r"QSA_API\s+[\w\s\*]+?\b(qsa_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 11
    for n in ["qsa_pool_keys", "qsa_index_score", "qsa_topk_blocks", "qsa_sparse_decode",
              "qsa_sparse_prefill_chunk"]:
        assert n in names
    for n in names:
        assert hasattr(lib, n), n


def test_only_declared_symbols_are_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", qbuild.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and l.split()[-1].startswith("qsa_")}
    assert exported == set(declared_symbols())


def test_version_and_status_strings(lib):
    assert "sm_103a" in qb.version()
    for s in range(7):
        assert lib.qsa_status_string(s)
    assert lib.qsa_status_string(99) == b"unknown status"


def cfg(**kw):
    base = dict(n_q_heads=16, n_kv_heads=2)
    base.update(kw)
    return qb.make_config(**base)


def test_workspace_size(lib):
    c = cfg()
    assert lib.qsa_workspace_size(qb.OP_POOL_KEYS, C.byref(c), 1, 10) == 256
    dec = lib.qsa_workspace_size(qb.OP_SPARSE_DECODE, C.byref(c), 32, 0)
    assert dec >= 256 + 32 * 2 * 8 * 4
    assert lib.qsa_workspace_size(qb.OP_SPARSE_DECODE, C.byref(cfg(head_dim=128)), 32, 0) == 0
    assert lib.qsa_workspace_size(99, C.byref(c), 1, 1) == 0
    assert lib.qsa_workspace_size(qb.OP_TOPK_BLOCKS, C.byref(c), -1, 1) == 0


FAKE = 0x10000000  # never dereferenced: validation fails or returns before any launch


@pytest.mark.parametrize("bad,code", [
    (dict(head_dim=128), qb.QSA_ERR_UNSUPPORTED),
    (dict(idx_dim=64), qb.QSA_ERR_UNSUPPORTED),
    (dict(ratio=8), qb.QSA_ERR_UNSUPPORTED),
    (dict(budget=1024), qb.QSA_ERR_UNSUPPORTED),
    (dict(n_q_heads=12, n_kv_heads=8), qb.QSA_ERR_UNSUPPORTED),
    (dict(n_q_heads=96, n_kv_heads=2), qb.QSA_ERR_UNSUPPORTED),
    (dict(n_kv_heads=0), qb.QSA_ERR_INVALID_ARGUMENT),
])
def test_bad_config_rejected(lib, bad, code):
    c = cfg(**bad)
    st = lib.qsa_sparse_decode(C.byref(c), FAKE, FAKE, FAKE, 100, FAKE, FAKE, 1, FAKE, FAKE, FAKE, 0, FAKE, 1 << 20, 0)
    assert st == code
    assert lib.qsa_last_error()


def test_argument_validation(lib):
    c = cfg()
    # NULL config
    assert lib.qsa_topk_blocks(None, FAKE, 10, FAKE, 1, FAKE, FAKE, FAKE, 1 << 20, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    # NULL / misaligned / too-small workspace
    assert lib.qsa_topk_blocks(C.byref(c), FAKE, 10, FAKE, 1, FAKE, FAKE, 0, 1 << 20, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_topk_blocks(C.byref(c), FAKE, 10, FAKE, 1, FAKE, FAKE, FAKE + 8, 1 << 20, 0) == \
        qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_sparse_decode(C.byref(c), FAKE, FAKE, FAKE, 100, FAKE, FAKE, 4, FAKE, FAKE, FAKE, 0, FAKE, 256,
                                 0) == qb.QSA_ERR_WORKSPACE_TOO_SMALL
    # NULL tensors
    assert lib.qsa_sparse_decode(C.byref(c), 0, FAKE, FAKE, 100, FAKE, FAKE, 1, FAKE, FAKE, FAKE, 0, FAKE, 1 << 20,
                                 0) == qb.QSA_ERR_INVALID_ARGUMENT
    # misaligned K
    assert lib.qsa_sparse_decode(C.byref(c), FAKE, FAKE + 2, FAKE, 100, FAKE, FAKE, 1, FAKE, FAKE, FAKE, 0, FAKE,
                                 1 << 20, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    # negative / out-of-range sizes
    assert lib.qsa_index_score(C.byref(c), FAKE, FAKE, FAKE, -1, FAKE, 10, FAKE, FAKE, 10, FAKE, 256, 0) == \
        qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_pool_keys(C.byref(c), FAKE, 100, FAKE, FAKE, FAKE, FAKE, 70000, 4, FAKE, 25, FAKE, 256, 0) == \
        qb.QSA_ERR_INVALID_ARGUMENT
    # prefill interval must be a positive multiple of 128
    for iv in (0, -128, 100):
        assert lib.qsa_sparse_prefill_chunk(C.byref(c), FAKE, 0, 16, FAKE, FAKE, FAKE, FAKE, iv, FAKE, 0, FAKE,
                                            1 << 20, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert b"interval" in lib.qsa_last_error()


def test_prefill_workspace_and_alignment_checks(lib):
    # The tensor-core prefill keeps its chunk plan in the workspace; a header-only
    # workspace is refused before anything launches, and so is a misaligned block list.
    c = cfg()
    need = lib.qsa_workspace_size(qb.OP_SPARSE_PREFILL_CHUNK, C.byref(c), 4096, 0)
    assert need > 4096 // 16 * 150_000
    assert lib.qsa_sparse_prefill_chunk(C.byref(c), FAKE, 0, 4096, FAKE, FAKE, FAKE, FAKE, 8192, FAKE, 0, FAKE,
                                        256, 0) == qb.QSA_ERR_WORKSPACE_TOO_SMALL
    assert lib.qsa_sparse_prefill_chunk(C.byref(c), FAKE, 0, 16, FAKE, FAKE, FAKE + 4, FAKE, 8192, FAKE, 0, FAKE,
                                        need, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert b"aligned" in lib.qsa_last_error()


def test_empty_batches_are_no_ops(lib):
    c = cfg()
    ws = FAKE
    assert lib.qsa_pool_keys(C.byref(c), 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, ws, 256, 0) == qb.QSA_OK
    assert lib.qsa_index_score(C.byref(c), 0, 0, 0, 0, 0, 0, 0, 0, 0, ws, 256, 0) == qb.QSA_OK
    assert lib.qsa_topk_blocks(C.byref(c), 0, 0, 0, 0, 0, 0, ws, 256, 0) == qb.QSA_OK
    assert lib.qsa_sparse_decode(C.byref(c), 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, ws, 256, 0) == qb.QSA_OK
    assert lib.qsa_sparse_prefill_chunk(C.byref(c), 0, 0, 0, 0, 0, 0, 0, 8192, 0, 0, ws, 256, 0) == qb.QSA_OK


def test_copy_rows_argument_checks(lib):
    """Host-side validation of the strided row copy; an empty copy is a no-op."""
    buf = (C.c_uint8 * 64)()
    p = C.addressof(buf)
    assert lib.qsa_copy_rows(p, 16, p, 16, 16, 0, None) == qb.QSA_OK
    assert lib.qsa_copy_rows(None, 16, p, 16, 16, 1, None) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_copy_rows(p, 8, p, 16, 16, 1, None) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_copy_rows(p, 16, p, 8, 16, 1, None) == qb.QSA_ERR_INVALID_ARGUMENT


@pytest.mark.gpu
def test_copy_rows_strided_host_to_device_and_back(lib):
    """Rows land at the destination pitch, untouched bytes between them stay as they were."""
    import torch
    rows, row_bytes, pitch = 5, 48, 80
    src = torch.arange(rows * row_bytes, dtype=torch.uint8).pin_memory()
    dst = torch.full((rows * pitch,), 255, dtype=torch.uint8, device="cuda")
    qb.qsa_copy_rows(dst, pitch, src, row_bytes, row_bytes, rows)
    back = torch.empty(rows * row_bytes, dtype=torch.uint8).pin_memory()
    qb.qsa_copy_rows(back, row_bytes, dst, pitch, row_bytes, rows)
    torch.cuda.synchronize()
    d = dst.cpu().view(rows, pitch)
    assert torch.equal(d[:, :row_bytes].reshape(-1), src)
    assert bool((d[:, row_bytes:] == 255).all())
    assert torch.equal(back, src)


def test_prefill_select_host_checks(lib):
    # the fused selection: workspace sized for the chunk, refused when too small, too few
    # queries for a tensor-core tile, or NULL tensors; nothing launches on a refusal
    c = cfg()
    need = lib.qsa_workspace_size(qb.OP_PREFILL_SELECT, C.byref(c), 4096, 66560)
    assert need > 4096 * 260 * 2 * 16 * 8          # the candidate slots dominate
    assert lib.qsa_prefill_select(C.byref(c), FAKE, FAKE, 4096, FAKE, 66560, FAKE, FAKE, 66560, FAKE, FAKE, FAKE,
                                  256, 0) == qb.QSA_ERR_WORKSPACE_TOO_SMALL
    need_small = lib.qsa_workspace_size(qb.OP_PREFILL_SELECT, C.byref(c), 64, 66560)
    assert lib.qsa_prefill_select(C.byref(c), FAKE, FAKE, 64, FAKE, 66560, FAKE, FAKE, 66560, FAKE, FAKE, FAKE,
                                  need_small, 0) == qb.QSA_ERR_UNSUPPORTED
    assert lib.qsa_prefill_select(C.byref(c), FAKE, FAKE, 4096, FAKE, 66560, FAKE, 0, 66560, FAKE, FAKE, FAKE,
                                  need, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    need0 = lib.qsa_workspace_size(qb.OP_PREFILL_SELECT, C.byref(c), 0, 66560)
    assert lib.qsa_prefill_select(C.byref(c), FAKE, FAKE, 0, FAKE, 66560, FAKE, FAKE, 66560, FAKE, FAKE, FAKE,
                                  need0, 0) == qb.QSA_OK


def test_fp8_key_calls_host_checks(lib):
    # FP8 indexer keys: same validation as the bf16 calls, plus the code and scale buffers
    c = cfg()
    ws = FAKE
    assert lib.qsa_pool_keys_fp8(C.byref(c), 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, ws, 256, 0) == qb.QSA_OK
    assert lib.qsa_index_score_fp8(C.byref(c), 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, ws, 256, 0) == qb.QSA_OK
    # NULL scales, misaligned codes, misaligned scales
    assert lib.qsa_pool_keys_fp8(C.byref(c), FAKE, 100, FAKE, FAKE, FAKE, FAKE, 1, 4, FAKE, 0, 25, ws, 256,
                                 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_pool_keys_fp8(C.byref(c), FAKE, 100, FAKE, FAKE, FAKE, FAKE, 1, 4, FAKE + 8, FAKE, 25, ws, 256,
                                 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert b"aligned" in lib.qsa_last_error()
    assert lib.qsa_index_score_fp8(C.byref(c), FAKE, 0, FAKE, 1, FAKE, FAKE + 2, 10, FAKE, FAKE, 10, ws, 256,
                                   0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert b"aligned" in lib.qsa_last_error()
    # sizes and workspace
    assert lib.qsa_index_score_fp8(C.byref(c), FAKE, 0, FAKE, -1, FAKE, FAKE, 10, FAKE, FAKE, 10, ws, 256, 0) == \
        qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_pool_keys_fp8(C.byref(c), FAKE, 100, FAKE, FAKE, FAKE, FAKE, 70000, 4, FAKE, FAKE, 25, ws, 256,
                                 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_index_score_fp8(C.byref(c), FAKE, 0, FAKE, 1, FAKE, FAKE, 10, FAKE, FAKE, 10, ws, 128, 0) == \
        qb.QSA_ERR_WORKSPACE_TOO_SMALL
    assert lib.qsa_index_score_fp8(C.byref(cfg(idx_dim=64)), FAKE, 0, FAKE, 1, FAKE, FAKE, 10, FAKE, FAKE, 10, ws,
                                   256, 0) == qb.QSA_ERR_UNSUPPORTED


def test_decode_step_fp8_host_checks(lib):
    c = cfg()
    need = lib.qsa_workspace_size(qb.OP_DECODE_STEP, C.byref(c), 1, 1000)
    args = lambda codes, scales, n_pooled, B: (C.byref(c), FAKE, codes, scales, n_pooled, FAKE, FAKE, FAKE, FAKE,
                                                FAKE, 4001, FAKE, FAKE, B, 1000, FAKE, FAKE, FAKE, 0, FAKE, need, 0)
    assert lib.qsa_decode_step_fp8(*args(0, 0, 0, 0)) == qb.QSA_OK                      # empty batch
    assert lib.qsa_decode_step_fp8(*args(0, FAKE, 1000, 1)) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_decode_step_fp8(*args(FAKE, FAKE + 4, 1000, 1)) == qb.QSA_ERR_INVALID_ARGUMENT
    assert b"aligned" in lib.qsa_last_error()
    assert lib.qsa_decode_step_fp8(*args(FAKE, FAKE, 1001, 1)) == qb.QSA_ERR_INVALID_ARGUMENT
    assert b"multiple of 4" in lib.qsa_last_error()
    assert lib.qsa_decode_step(C.byref(c), FAKE, 0, 1000, FAKE, FAKE, FAKE, FAKE, FAKE, 4001, FAKE, FAKE, 1, 1000,
                               FAKE, FAKE, FAKE, 0, FAKE, need, 0) == qb.QSA_ERR_INVALID_ARGUMENT


def test_fp8_kv_calls_host_checks(lib):
    # the quantiser: empty is a no-op; NULL, misaligned and out-of-range arguments are refused
    assert lib.qsa_quantize_kv_fp8(0, 0, 0, 0, 0) == qb.QSA_OK
    assert lib.qsa_quantize_kv_fp8(FAKE, -1, FAKE, FAKE, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_quantize_kv_fp8(FAKE, (1 << 34) + 1, FAKE, FAKE, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_quantize_kv_fp8(FAKE, 4, FAKE, 0, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_quantize_kv_fp8(FAKE, 4, FAKE + 8, FAKE, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert b"aligned" in lib.qsa_last_error()
    assert lib.qsa_quantize_kv_fp8(FAKE, 4, FAKE, FAKE + 4, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    # the fused step over FP8 K/V: exactly one key format, all four K/V planes, 16-byte alignment
    c = cfg()
    need = lib.qsa_workspace_size(qb.OP_DECODE_STEP, C.byref(c), 1, 1000)

    def call(pooled, codes, scales, kc, ks, vc, vs, B=1):
        return lib.qsa_decode_step_fp8kv(C.byref(c), FAKE, pooled, codes, scales, 1000, FAKE, FAKE, FAKE, kc, ks, vc,
                                         vs, 4001, FAKE, FAKE, B, 1000, FAKE, FAKE, FAKE, 0, FAKE, need, 0)
    assert call(0, 0, 0, 0, 0, 0, 0, B=0) == qb.QSA_OK                                   # empty batch
    assert call(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE) == qb.QSA_ERR_INVALID_ARGUMENT  # both key formats
    assert b"either" in lib.qsa_last_error()
    assert call(0, 0, 0, FAKE, FAKE, FAKE, FAKE) == qb.QSA_ERR_INVALID_ARGUMENT          # neither
    assert call(FAKE, 0, 0, FAKE, 0, FAKE, FAKE) == qb.QSA_ERR_INVALID_ARGUMENT          # NULL k_scales
    assert b"NULL" in lib.qsa_last_error()
    assert call(FAKE, 0, 0, FAKE, FAKE + 8, FAKE, FAKE) == qb.QSA_ERR_INVALID_ARGUMENT   # misaligned scales
    assert b"aligned" in lib.qsa_last_error()
    assert call(0, FAKE, FAKE, FAKE + 4, FAKE, FAKE, FAKE) == qb.QSA_ERR_INVALID_ARGUMENT  # misaligned codes
    assert lib.qsa_decode_step_fp8kv(C.byref(cfg(n_kv_heads=4)), FAKE, FAKE, 0, 0, 1000, FAKE, FAKE, FAKE, FAKE,
                                     FAKE, FAKE, FAKE, 4001, FAKE, FAKE, 1, 1000, FAKE, FAKE, FAKE, 0, FAKE,
                                     need, 0) == qb.QSA_ERR_UNSUPPORTED


def test_rowcache_host_checks(lib):
    # one slot: the token's K and V rows of every KV head, an int64 tag, a uint32 hit epoch
    # (the array rounded up to 8 bytes) and a uint64 claim
    c = cfg()
    assert lib.qsa_rowcache_bytes(C.byref(c), 1000) == 1000 * (2 * 2 * 512 + 8) + 4000 + 1000 * 8
    assert lib.qsa_rowcache_bytes(C.byref(c), 3) == 3 * (2048 + 8) + 16 + 24
    assert lib.qsa_rowcache_bytes(C.byref(cfg(n_q_heads=8, n_kv_heads=1)), 4) == 4 * (1024 + 8) + 16 + 32
    assert lib.qsa_rowcache_bytes(C.byref(c), 0) == 0
    assert lib.qsa_rowcache_bytes(C.byref(cfg(n_kv_heads=4)), 10) == 0
    assert lib.qsa_rowcache_bytes(C.byref(cfg(head_dim=128)), 10) == 0
    need = lib.qsa_rowcache_bytes(C.byref(c), 64)
    assert lib.qsa_rowcache_init(C.byref(c), 0, need, 64, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_rowcache_init(C.byref(c), FAKE + 8, need, 64, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_rowcache_init(C.byref(c), FAKE, need - 1, 64, 0) == qb.QSA_ERR_WORKSPACE_TOO_SMALL
    assert lib.qsa_rowcache_init(C.byref(c), FAKE, need, 0, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    # the fused step with the cache: an empty batch is a no-op; a NULL cache is refused
    ws_need = lib.qsa_workspace_size(qb.OP_DECODE_STEP, C.byref(c), 1, 1000)

    def step(cache, n_slots, epoch, B=1):
        return lib.qsa_decode_step_rowcache(C.byref(c), FAKE, FAKE, 1000, FAKE, FAKE, FAKE, FAKE, FAKE, 4001, FAKE,
                                            FAKE, B, 1000, FAKE, FAKE, FAKE, 0, FAKE, ws_need, cache, need, n_slots,
                                            epoch, 0)
    assert step(0, 64, 1, B=0) == qb.QSA_OK
    assert step(0, 64, 1) == qb.QSA_ERR_INVALID_ARGUMENT


def test_prefill_staged_host_checks(lib):
    c = cfg()
    ws_need = lib.qsa_workspace_size(qb.OP_SPARSE_PREFILL_CHUNK, C.byref(c), 40, 0)
    rows = 1000 + 40
    need = 2 * rows * 2 * 256 * 2

    def call(stage, stage_bytes, nc=40):
        return lib.qsa_sparse_prefill_chunk_staged(C.byref(c), FAKE, 1000, nc, FAKE, FAKE, FAKE, FAKE, 1024, FAKE, 0,
                                                   FAKE, ws_need, stage, stage_bytes, 0)
    assert call(0, 0, nc=0) == qb.QSA_OK                               # empty chunk
    assert call(0, need) == qb.QSA_ERR_INVALID_ARGUMENT                # no stage
    assert call(FAKE + 8, need) == qb.QSA_ERR_INVALID_ARGUMENT         # misaligned
    assert call(FAKE, need - 1) == qb.QSA_ERR_WORKSPACE_TOO_SMALL
    assert b"stage" in lib.qsa_last_error()


def test_fp8_kv_prefill_and_dequantiser_host_checks(lib):
    # the dequantiser: empty is a no-op; NULL, misaligned and out-of-range arguments are refused
    assert lib.qsa_dequantize_kv_fp8(0, 0, 0, 0, 0) == qb.QSA_OK
    assert lib.qsa_dequantize_kv_fp8(FAKE, FAKE, -1, FAKE, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_dequantize_kv_fp8(FAKE, FAKE, (1 << 34) + 1, FAKE, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_dequantize_kv_fp8(FAKE, 0, 4, FAKE, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_dequantize_kv_fp8(FAKE + 8, FAKE, 4, FAKE, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert b"aligned" in lib.qsa_last_error()
    assert lib.qsa_dequantize_kv_fp8(FAKE, FAKE + 4, 4, FAKE, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert lib.qsa_dequantize_kv_fp8(FAKE, FAKE, 4, FAKE + 8, 0) == qb.QSA_ERR_INVALID_ARGUMENT
    # the FP8 K/V prefill: the stage and the four row planes are checked before anything runs
    c = cfg()
    ws_need = lib.qsa_workspace_size(qb.OP_SPARSE_PREFILL_CHUNK, C.byref(c), 40, 0)
    need = 2 * (1000 + 40) * 2 * 256 * 2

    def call(stage, stage_bytes, nc=40, kc=FAKE, ks=FAKE, vc=FAKE, vs=FAKE, interval=1024, ws_bytes=ws_need):
        return lib.qsa_sparse_prefill_chunk_fp8kv(C.byref(c), FAKE, 1000, nc, kc, ks, vc, vs, FAKE, FAKE, interval,
                                                  FAKE, 0, FAKE, ws_bytes, stage, stage_bytes, 0)
    assert call(0, 0, nc=0) == qb.QSA_OK                               # empty chunk
    assert call(FAKE, need, interval=1000) == qb.QSA_ERR_INVALID_ARGUMENT       # refused before staging
    assert b"interval" in lib.qsa_last_error()
    assert call(FAKE, need, ws_bytes=ws_need - 1) == qb.QSA_ERR_WORKSPACE_TOO_SMALL
    assert call(0, need) == qb.QSA_ERR_INVALID_ARGUMENT                # no stage
    assert call(FAKE + 8, need) == qb.QSA_ERR_INVALID_ARGUMENT         # misaligned stage
    assert call(FAKE, need - 1) == qb.QSA_ERR_WORKSPACE_TOO_SMALL
    assert b"stage" in lib.qsa_last_error()
    assert call(FAKE, need, vs=0) == qb.QSA_ERR_INVALID_ARGUMENT
    assert call(FAKE, need, kc=FAKE + 8) == qb.QSA_ERR_INVALID_ARGUMENT
    assert call(FAKE, need, ks=FAKE + 4) == qb.QSA_ERR_INVALID_ARGUMENT


def test_sparse_mla_host_checks(lib):
    need = lib.qsa_sparse_mla_workspace_size(64, 4, 2048)
    # status block + the partials: up to 256 persistent CTAs + one per query of 64 heads x 512
    # fp32 (two latent halves of 256 per (query, half) above 64 heads fit the same bytes), and a
    # (max, sum) pair per head for up to 256 + 2 per query segments, + slack
    assert need == 256 + (256 + 4) * 64 * 512 * 4 + (256 + 2 * 4) * 64 * 2 * 4 + 256
    assert lib.qsa_sparse_mla_workspace_size(0, 4, 2048) == 0
    assert lib.qsa_sparse_mla_workspace_size(129, 4, 2048) == 0
    assert lib.qsa_sparse_mla_workspace_size(64, 4, 70000) == 0
    args = lambda q, heads, B, ws_bytes: (q, heads, FAKE, 1000, FAKE, FAKE, 2048, B, C.c_float(0.0), FAKE, 0, FAKE,
                                          ws_bytes, 0)
    assert lib.qsa_sparse_mla_decode(*args(FAKE, 64, 0, need)) == qb.QSA_OK                # empty batch
    assert lib.qsa_sparse_mla_decode(*args(FAKE, 200, 4, need)) == qb.QSA_ERR_UNSUPPORTED
    assert lib.qsa_sparse_mla_decode(*args(FAKE, 64, 4, need - 1)) == qb.QSA_ERR_WORKSPACE_TOO_SMALL
    assert lib.qsa_sparse_mla_decode(*args(FAKE + 8, 64, 4, need)) == qb.QSA_ERR_INVALID_ARGUMENT
    assert b"aligned" in lib.qsa_last_error()
    assert lib.qsa_sparse_mla_decode(*args(0, 64, 4, need)) == qb.QSA_ERR_INVALID_ARGUMENT
