"""ctypes binding of libqsa.so: argument marshalling only.

Every function named ``qsa_*`` here calls the C entry point of the same name with
the device pointers of the torch tensors it is given; all work runs in the
library's CUDA kernels. PyTorch only supplies device memory and streams. If the
library is missing, :func:`load` raises: there is no fallback path.
"""

from __future__ import annotations

import ctypes as C
import os

import torch

from .build import LIB_PATH

QSA_OK = 0
QSA_ERR_INVALID_ARGUMENT = 1
QSA_ERR_UNSUPPORTED = 2
QSA_ERR_WORKSPACE_TOO_SMALL = 3
QSA_ERR_CUDA = 4
QSA_ERR_DEVICE_TIMEOUT = 5
QSA_ERR_DEVICE_BOUNDS = 6

(OP_POOL_KEYS, OP_INDEX_SCORE, OP_TOPK_BLOCKS, OP_SPARSE_DECODE, OP_SPARSE_PREFILL_CHUNK, OP_DECODE_STEP,
 OP_PREFILL_SELECT) = range(7)
BLOCK_TOPK = 512


class QsaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class qsa_config(C.Structure):
    _fields_ = [("n_q_heads", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("idx_dim", C.c_int32), ("indexer_compress_ratio", C.c_int32), ("indexer_budget", C.c_int32),
                ("softmax_scale", C.c_float)]


def make_config(n_q_heads: int, n_kv_heads: int = 2, head_dim: int = 256, idx_dim: int = 128,
                ratio: int = 4, budget: int = 2048, softmax_scale: float = 0.0) -> qsa_config:
    return qsa_config(n_q_heads, n_kv_heads, head_dim, idx_dim, ratio, budget, softmax_scale)


_P = C.c_void_p
_I32 = C.c_int32
_I64 = C.c_int64
_SZ = C.c_size_t
_CFG = C.POINTER(qsa_config)

_SIGNATURES = {
    "qsa_workspace_size": (_SZ, [_I32, _CFG, _I32, _I64]),
    "qsa_workspace_init": (_I32, [_P, _SZ, _P]),
    "qsa_read_device_status": (_I32, [_P, _P, C.POINTER(_I32), C.POINTER(_I32)]),
    "qsa_pool_keys": (_I32, [_CFG, _P, _I64, _P, _P, _P, _P, _I32, _I64, _P, _I64, _P, _SZ, _P]),
    "qsa_index_score": (_I32, [_CFG, _P, _P, _P, _I32, _P, _I64, _P, _P, _I64, _P, _SZ, _P]),
    "qsa_topk_blocks": (_I32, [_CFG, _P, _I64, _P, _I32, _P, _P, _P, _SZ, _P]),
    "qsa_sparse_decode": (_I32, [_CFG, _P, _P, _P, _I64, _P, _P, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
    "qsa_sparse_prefill_chunk": (_I32, [_CFG, _P, _I32, _I32, _P, _P, _P, _P, _I32, _P, _P, _P, _SZ, _P]),
    "qsa_sparse_prefill_chunk_staged": (_I32, [_CFG, _P, _I32, _I32, _P, _P, _P, _P, _I32, _P, _P, _P, _SZ, _P, _SZ,
                                               _P]),
    "qsa_decode_step": (_I32, [_CFG, _P, _P, _I64, _P, _P, _P, _P, _P, _I64, _P, _P, _I32, _I64, _P, _P, _P, _P,
                                _P, _SZ, _P]),
    "qsa_decode_step_prefetch": (_I32, [_CFG, _P, _P, _I64, _P, _P, _P, _P, _P, _I64, _P, _P, _I32, _I64, _P, _P,
                                         _P, _P, _P, _SZ, _P, _SZ, _P]),
    "qsa_decode_step_fp8_prefetch": (_I32, [_CFG, _P, _P, _P, _I64, _P, _P, _P, _P, _P, _I64, _P, _P, _I32, _I64,
                                             _P, _P, _P, _P, _P, _SZ, _P, _SZ, _P]),
    "qsa_sparse_decode_noalloc": (_I32, [_CFG, _P, _P, _P, _I64, _P, _P, _I32, _P, _P, _P, _P, _P]),
    "qsa_copy_rows": (_I32, [_P, _SZ, _P, _SZ, _SZ, _SZ, _P]),
    "qsa_prefill_select": (_I32, [_CFG, _P, _P, _I32, _P, _I64, _P, _P, _I64, _P, _P, _P, _SZ, _P]),
    "qsa_pool_keys_fp8": (_I32, [_CFG, _P, _I64, _P, _P, _P, _P, _I32, _I64, _P, _P, _I64, _P, _SZ, _P]),
    "qsa_index_score_fp8": (_I32, [_CFG, _P, _P, _P, _I32, _P, _P, _I64, _P, _P, _I64, _P, _SZ, _P]),
    "qsa_decode_step_fp8": (_I32, [_CFG, _P, _P, _P, _I64, _P, _P, _P, _P, _P, _I64, _P, _P, _I32, _I64, _P, _P,
                                    _P, _P, _P, _SZ, _P]),
    "qsa_decode_step_fp8kv": (_I32, [_CFG, _P, _P, _P, _P, _I64, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _P, _I32,
                                      _I64, _P, _P, _P, _P, _P, _SZ, _P]),
    "qsa_quantize_kv_fp8": (_I32, [_P, _I64, _P, _P, _P]),
    "qsa_dequantize_kv_fp8": (_I32, [_P, _P, _I64, _P, _P]),
    "qsa_sparse_prefill_chunk_fp8kv": (_I32, [_CFG, _P, _I32, _I32, _P, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _SZ,
                                              _P, _SZ, _P]),
    "qsa_rowcache_bytes": (_SZ, [_CFG, _I64]),
    "qsa_rowcache_init": (_I32, [_CFG, _P, _SZ, _I64, _P]),
    "qsa_decode_step_rowcache": (_I32, [_CFG, _P, _P, _I64, _P, _P, _P, _P, _P, _I64, _P, _P, _I32, _I64, _P, _P,
                                        _P, _P, _P, _SZ, _P, _SZ, _I64, C.c_uint32, _P]),
    "qsa_sparse_mla_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "qsa_sparse_mla_decode": (_I32, [_P, _I32, _P, _I64, _P, _P, _I32, _I32, C.c_float, _P, _P, _P, _SZ, _P]),
    "qsa_status_string": (C.c_char_p, [_I32]),
    "qsa_last_error": (C.c_char_p, []),
    "qsa_version": (C.c_char_p, []),
}

_LIB = None


def load(path: str | None = None):
    """Load libqsa.so (built in-tree by ``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() (no CPU fallback exists)")
    lib = C.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t, dtype=None, name="tensor") -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _check(status: int, what: str):
    if status != QSA_OK:
        lib = load()
        raise QsaError(status, f"{what}: {lib.qsa_status_string(status).decode()}: {lib.qsa_last_error().decode()}")


def workspace_size(op: int, cfg: qsa_config, n_rows: int, max_blocks: int = 0) -> int:
    return int(load().qsa_workspace_size(op, C.byref(cfg), n_rows, max_blocks))


def make_workspace(op: int, cfg: qsa_config, n_rows: int, max_blocks: int = 0, device="cuda", stream=None):
    """A zero-initialised workspace tensor for ``op`` (allocated by torch)."""
    n = workspace_size(op, cfg, n_rows, max_blocks)
    if n == 0:
        raise QsaError(QSA_ERR_UNSUPPORTED, "unsupported geometry for workspace")
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n]
    qsa_workspace_init(ws, stream)
    return ws


def qsa_workspace_init(ws, stream=None):
    _check(load().qsa_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "qsa_workspace_init")


def qsa_read_device_status(ws, stream=None):
    st, det = _I32(0), _I32(0)
    _check(load().qsa_read_device_status(_ptr(ws), _stream(stream), C.byref(st), C.byref(det)),
           "qsa_read_device_status")
    return st.value, det.value


def qsa_copy_rows(dst, dst_pitch, src, src_pitch, row_bytes, n_rows, stream=None):
    """Strided row copy between any two memories (pointers or tensors' data pointers)."""
    d = dst if isinstance(dst, int) else dst.data_ptr()
    s = src if isinstance(src, int) else src.data_ptr()
    _check(load().qsa_copy_rows(d, dst_pitch, s, src_pitch, row_bytes, n_rows, _stream(stream)), "qsa_copy_rows")


def _ws_args(ws):
    return _ptr(ws), ws.numel() * ws.element_size()


def qsa_pool_keys(cfg, raw_idx_k, tok_off, blk_off, blk_begin, blk_end, max_blocks_per_seq, pooled, ws, stream=None):
    B = tok_off.numel() - 1
    _check(load().qsa_pool_keys(C.byref(cfg), _ptr(raw_idx_k, torch.bfloat16, "raw_idx_k"), raw_idx_k.shape[0],
                                _ptr(tok_off, torch.int32), _ptr(blk_off, torch.int32), _ptr(blk_begin, torch.int32),
                                _ptr(blk_end, torch.int32), B, int(max_blocks_per_seq),
                                _ptr(pooled, torch.bfloat16, "pooled"), pooled.shape[0], *_ws_args(ws),
                                _stream(stream)), "qsa_pool_keys")


def qsa_index_score(cfg, q_idx, q_seq, q_pos, pooled, blk_off, scores, ws, stream=None):
    _check(load().qsa_index_score(C.byref(cfg), _ptr(q_idx, torch.bfloat16, "q_idx"), _ptr(q_seq, torch.int32),
                                  _ptr(q_pos, torch.int32), q_idx.shape[0], _ptr(pooled, torch.bfloat16, "pooled"),
                                  pooled.shape[0], _ptr(blk_off, torch.int32), _ptr(scores, torch.float32, "scores"),
                                  scores.shape[1], *_ws_args(ws), _stream(stream)), "qsa_index_score")


def qsa_pool_keys_fp8(cfg, raw_idx_k, tok_off, blk_off, blk_begin, blk_end, max_blocks_per_seq, codes, scales, ws,
                      stream=None):
    B = tok_off.numel() - 1
    if codes.shape[0] != scales.shape[0]:
        raise ValueError("codes and scales must have one row per pooled block")
    _check(load().qsa_pool_keys_fp8(C.byref(cfg), _ptr(raw_idx_k, torch.bfloat16, "raw_idx_k"), raw_idx_k.shape[0],
                                    _ptr(tok_off, torch.int32), _ptr(blk_off, torch.int32),
                                    _ptr(blk_begin, torch.int32), _ptr(blk_end, torch.int32), B,
                                    int(max_blocks_per_seq), _ptr(codes, torch.uint8, "codes"),
                                    _ptr(scales, torch.float32, "scales"), codes.shape[0], *_ws_args(ws),
                                    _stream(stream)), "qsa_pool_keys_fp8")


def qsa_index_score_fp8(cfg, q_idx, q_seq, q_pos, codes, scales, blk_off, scores, ws, stream=None):
    if codes.shape[0] != scales.shape[0]:
        raise ValueError("codes and scales must have one row per pooled block")
    _check(load().qsa_index_score_fp8(C.byref(cfg), _ptr(q_idx, torch.bfloat16, "q_idx"), _ptr(q_seq, torch.int32),
                                      _ptr(q_pos, torch.int32), q_idx.shape[0], _ptr(codes, torch.uint8, "codes"),
                                      _ptr(scales, torch.float32, "scales"), codes.shape[0],
                                      _ptr(blk_off, torch.int32), _ptr(scores, torch.float32, "scores"),
                                      scores.shape[1], *_ws_args(ws), _stream(stream)), "qsa_index_score_fp8")


def qsa_prefill_select(cfg, q_idx, q_pos, pooled, blk_off, scores, blocks, count, ws, stream=None):
    _check(load().qsa_prefill_select(C.byref(cfg), _ptr(q_idx, torch.bfloat16, "q_idx"), _ptr(q_pos, torch.int32),
                                     q_idx.shape[0], _ptr(pooled, torch.bfloat16, "pooled"), pooled.shape[0],
                                     _ptr(blk_off, torch.int32), _ptr(scores, torch.float32, "scores"),
                                     scores.shape[1], _ptr(blocks, torch.int32, "blocks"),
                                     _ptr(count, torch.int32, "count"), *_ws_args(ws), _stream(stream)),
           "qsa_prefill_select")


def qsa_topk_blocks(cfg, scores, q_pos, blocks, count, ws, stream=None):
    _check(load().qsa_topk_blocks(C.byref(cfg), _ptr(scores, torch.float32, "scores"), scores.shape[1],
                                  _ptr(q_pos, torch.int32), q_pos.numel(), _ptr(blocks, torch.int32, "blocks"),
                                  _ptr(count, torch.int32, "count"), *_ws_args(ws), _stream(stream)),
           "qsa_topk_blocks")


def qsa_sparse_decode(cfg, q, k_cache, v_cache, tok_off, ctx_len, blocks, count, out, lse, ws, stream=None):
    _check(load().qsa_sparse_decode(C.byref(cfg), _ptr(q, torch.bfloat16, "q"), _ptr(k_cache, torch.bfloat16, "k"),
                                    _ptr(v_cache, torch.bfloat16, "v"), k_cache.shape[0], _ptr(tok_off, torch.int32),
                                    _ptr(ctx_len, torch.int32), ctx_len.numel(), _ptr(blocks, torch.int32),
                                    _ptr(count, torch.int32), _ptr(out, torch.bfloat16, "out"),
                                    _ptr(lse, torch.float32, "lse"), *_ws_args(ws), _stream(stream)),
           "qsa_sparse_decode")


def _next_read(t):
    """(pointer, bytes) of an optional L2 prefetch hint tensor (contiguous, any dtype)."""
    if t is None:
        return None, 0
    if not t.is_contiguous():
        raise ValueError("next_read must be contiguous")
    return t.data_ptr(), t.numel() * t.element_size()


def qsa_decode_step(cfg, raw_idx_k, pooled, blk_off, q_idx, q, k_cache, v_cache, tok_off, ctx_len, max_blocks,
                    blocks, count, out, lse, ws, stream=None, next_read=None):
    """One fused decode layer-step; with `next_read` (the tensor the next call will scan, e.g.
    the next layer's pooled keys) the step also prefetches it into L2 (qsa_decode_step_prefetch)."""
    args = [C.byref(cfg), _ptr(raw_idx_k, torch.bfloat16, "raw_idx_k"), _ptr(pooled, torch.bfloat16, "pooled"),
            pooled.shape[0], _ptr(blk_off, torch.int32), _ptr(q_idx, torch.bfloat16, "q_idx"),
            _ptr(q, torch.bfloat16, "q"), _ptr(k_cache, torch.bfloat16, "k"), _ptr(v_cache, torch.bfloat16, "v"),
            k_cache.shape[0], _ptr(tok_off, torch.int32), _ptr(ctx_len, torch.int32), ctx_len.numel(),
            int(max_blocks), _ptr(blocks, torch.int32), _ptr(count, torch.int32), _ptr(out, torch.bfloat16, "out"),
            _ptr(lse, torch.float32, "lse"), *_ws_args(ws)]
    if next_read is None:
        _check(load().qsa_decode_step(*args, _stream(stream)), "qsa_decode_step")
    else:
        _check(load().qsa_decode_step_prefetch(*args, *_next_read(next_read), _stream(stream)),
               "qsa_decode_step_prefetch")


def qsa_decode_step_fp8(cfg, raw_idx_k, codes, scales, blk_off, q_idx, q, k_cache, v_cache, tok_off, ctx_len,
                        max_blocks, blocks, count, out, lse, ws, stream=None, next_read=None):
    if codes.shape[0] != scales.shape[0]:
        raise ValueError("codes and scales must have one row per pooled block")
    args = [C.byref(cfg), _ptr(raw_idx_k, torch.bfloat16, "raw_idx_k"), _ptr(codes, torch.uint8, "codes"),
            _ptr(scales, torch.float32, "scales"), codes.shape[0], _ptr(blk_off, torch.int32),
            _ptr(q_idx, torch.bfloat16, "q_idx"), _ptr(q, torch.bfloat16, "q"), _ptr(k_cache, torch.bfloat16, "k"),
            _ptr(v_cache, torch.bfloat16, "v"), k_cache.shape[0], _ptr(tok_off, torch.int32),
            _ptr(ctx_len, torch.int32), ctx_len.numel(), int(max_blocks), _ptr(blocks, torch.int32),
            _ptr(count, torch.int32), _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
            *_ws_args(ws)]
    if next_read is None:
        _check(load().qsa_decode_step_fp8(*args, _stream(stream)), "qsa_decode_step_fp8")
    else:
        _check(load().qsa_decode_step_fp8_prefetch(*args, *_next_read(next_read), _stream(stream)),
               "qsa_decode_step_fp8_prefetch")


def qsa_quantize_kv_fp8(x, codes, scales, stream=None):
    """FP8 K/V rows: x [..., 256] bf16 -> codes [..., 256] uint8 and scales [..., 2] fp32."""
    if x.shape[-1] != 256 or codes.shape != x.shape or scales.shape != x.shape[:-1] + (2,):
        raise ValueError("x [..., 256], codes [..., 256], scales [..., 2]")
    n_rows = x.numel() // 256
    _check(load().qsa_quantize_kv_fp8(_ptr(x, torch.bfloat16, "x"), n_rows, _ptr(codes, torch.uint8, "codes"),
                                      _ptr(scales, torch.float32, "scales"), _stream(stream)),
           "qsa_quantize_kv_fp8")


def qsa_dequantize_kv_fp8(codes, scales, x, stream=None):
    """codes [..., 256] uint8 and scales [..., 2] fp32 -> x [..., 256] bf16 (code x scale rounded once)."""
    if codes.shape[-1] != 256 or x.shape != codes.shape or scales.shape != codes.shape[:-1] + (2,):
        raise ValueError("codes [..., 256], scales [..., 2], x [..., 256]")
    n_rows = codes.numel() // 256
    _check(load().qsa_dequantize_kv_fp8(_ptr(codes, torch.uint8, "codes"), _ptr(scales, torch.float32, "scales"),
                                        n_rows, _ptr(x, torch.bfloat16, "x"), _stream(stream)),
           "qsa_dequantize_kv_fp8")


def qsa_decode_step_fp8kv(cfg, raw_idx_k, pooled, codes, scales, blk_off, q_idx, q, k_codes, k_scales, v_codes,
                          v_scales, tok_off, ctx_len, max_blocks, blocks, count, out, lse, ws, stream=None):
    """One fused decode layer-step over FP8 K/V rows (codes [T, Hkv, 256] uint8 + scales [T, Hkv, 2]
    fp32); the indexer keys are bf16 (`pooled`) or FP8 (`codes`, `scales`), the other pair None."""
    n_pooled = pooled.shape[0] if pooled is not None else codes.shape[0]
    if pooled is None and codes.shape[0] != scales.shape[0]:
        raise ValueError("codes and scales must have one row per pooled block")
    args = [C.byref(cfg), _ptr(raw_idx_k, torch.bfloat16, "raw_idx_k"), _ptr(pooled, torch.bfloat16, "pooled"),
            _ptr(codes, torch.uint8, "codes"), _ptr(scales, torch.float32, "scales"), n_pooled,
            _ptr(blk_off, torch.int32), _ptr(q_idx, torch.bfloat16, "q_idx"), _ptr(q, torch.bfloat16, "q"),
            _ptr(k_codes, torch.uint8, "k_codes"), _ptr(k_scales, torch.float32, "k_scales"),
            _ptr(v_codes, torch.uint8, "v_codes"), _ptr(v_scales, torch.float32, "v_scales"), k_codes.shape[0],
            _ptr(tok_off, torch.int32), _ptr(ctx_len, torch.int32), ctx_len.numel(), int(max_blocks),
            _ptr(blocks, torch.int32), _ptr(count, torch.int32), _ptr(out, torch.bfloat16, "out"),
            _ptr(lse, torch.float32, "lse"), *_ws_args(ws)]
    _check(load().qsa_decode_step_fp8kv(*args, _stream(stream)), "qsa_decode_step_fp8kv")


def rowcache_new(cfg, n_slots, device="cuda"):
    """A row cache of n_slots token rows (uint8 device tensor), emptied."""
    nbytes = load().qsa_rowcache_bytes(C.byref(cfg), int(n_slots))
    if nbytes == 0:
        raise ValueError("bad row-cache configuration")
    cache = torch.empty(nbytes, dtype=torch.uint8, device=device)
    qsa_rowcache_init(cfg, cache, n_slots)
    return cache


def qsa_rowcache_init(cfg, cache, n_slots, stream=None):
    _check(load().qsa_rowcache_init(C.byref(cfg), _ptr(cache), cache.numel(), int(n_slots), _stream(stream)),
           "qsa_rowcache_init")


def qsa_decode_step_rowcache(cfg, raw_idx_k, pooled, blk_off, q_idx, q, k_cache, v_cache, tok_off, ctx_len,
                             max_blocks, blocks, count, out, lse, ws, cache, n_slots, epoch, stream=None):
    args = [C.byref(cfg), _ptr(raw_idx_k, torch.bfloat16, "raw_idx_k"), _ptr(pooled, torch.bfloat16, "pooled"),
            pooled.shape[0], _ptr(blk_off, torch.int32), _ptr(q_idx, torch.bfloat16, "q_idx"),
            _ptr(q, torch.bfloat16, "q"), _ptr(k_cache, torch.bfloat16, "k"), _ptr(v_cache, torch.bfloat16, "v"),
            k_cache.shape[0], _ptr(tok_off, torch.int32), _ptr(ctx_len, torch.int32), ctx_len.numel(),
            int(max_blocks), _ptr(blocks, torch.int32), _ptr(count, torch.int32), _ptr(out, torch.bfloat16, "out"),
            _ptr(lse, torch.float32, "lse"), *_ws_args(ws), _ptr(cache), cache.numel(), int(n_slots), int(epoch)]
    _check(load().qsa_decode_step_rowcache(*args, _stream(stream)), "qsa_decode_step_rowcache")


def qsa_sparse_decode_noalloc(cfg, q, k_cache, v_cache, tok_off, ctx_len, blocks, count, out, lse, stream=None):
    _check(load().qsa_sparse_decode_noalloc(C.byref(cfg), _ptr(q, torch.bfloat16, "q"),
                                            _ptr(k_cache, torch.bfloat16, "k"), _ptr(v_cache, torch.bfloat16, "v"),
                                            k_cache.shape[0], _ptr(tok_off, torch.int32), _ptr(ctx_len, torch.int32),
                                            ctx_len.numel(), _ptr(blocks, torch.int32), _ptr(count, torch.int32),
                                            _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
                                            _stream(stream)), "qsa_sparse_decode_noalloc")


def qsa_sparse_prefill_chunk(cfg, q, p0, k_cache, v_cache, blocks, count, interval_tokens, out, lse, ws,
                             stream=None):
    _check(load().qsa_sparse_prefill_chunk(C.byref(cfg), _ptr(q, torch.bfloat16, "q"), int(p0), q.shape[0],
                                           _ptr(k_cache, torch.bfloat16, "k"), _ptr(v_cache, torch.bfloat16, "v"),
                                           _ptr(blocks, torch.int32), _ptr(count, torch.int32), int(interval_tokens),
                                           _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
                                           *_ws_args(ws), _stream(stream)), "qsa_sparse_prefill_chunk")


def qsa_sparse_prefill_chunk_staged(cfg, q, p0, k_cache, v_cache, blocks, count, interval_tokens, out, lse, ws,
                                    stage, stream=None):
    """qsa_sparse_prefill_chunk with K/V (e.g. in pinned host memory) first copied into `stage`
    (a device uint8 tensor of at least 2 x rows x n_kv_heads x head_dim x 2 bytes)."""
    _check(load().qsa_sparse_prefill_chunk_staged(C.byref(cfg), _ptr(q, torch.bfloat16, "q"), int(p0), q.shape[0],
                                                  _ptr(k_cache, torch.bfloat16, "k"), _ptr(v_cache, torch.bfloat16, "v"),
                                                  _ptr(blocks, torch.int32), _ptr(count, torch.int32),
                                                  int(interval_tokens), _ptr(out, torch.bfloat16, "out"),
                                                  _ptr(lse, torch.float32, "lse"), *_ws_args(ws), _ptr(stage),
                                                  stage.numel() * stage.element_size(), _stream(stream)),
           "qsa_sparse_prefill_chunk_staged")


def qsa_sparse_prefill_chunk_fp8kv(cfg, q, p0, kv8, blocks, count, interval_tokens, out, lse, ws, stage,
                                   stream=None):
    """qsa_sparse_prefill_chunk over FP8 K/V rows: kv8 = (k_codes, k_scales, v_codes, v_scales) as
    qsa_quantize_kv_fp8 writes them; `stage` a device uint8 tensor of at least
    2 x rows x n_kv_heads x 512 bytes that receives the dequantised bf16 rows."""
    k_codes, k_scales, v_codes, v_scales = kv8
    _check(load().qsa_sparse_prefill_chunk_fp8kv(C.byref(cfg), _ptr(q, torch.bfloat16, "q"), int(p0), q.shape[0],
                                                 _ptr(k_codes, torch.uint8, "k_codes"),
                                                 _ptr(k_scales, torch.float32, "k_scales"),
                                                 _ptr(v_codes, torch.uint8, "v_codes"),
                                                 _ptr(v_scales, torch.float32, "v_scales"),
                                                 _ptr(blocks, torch.int32), _ptr(count, torch.int32),
                                                 int(interval_tokens), _ptr(out, torch.bfloat16, "out"),
                                                 _ptr(lse, torch.float32, "lse"), *_ws_args(ws), _ptr(stage),
                                                 stage.numel() * stage.element_size(), _stream(stream)),
           "qsa_sparse_prefill_chunk_fp8kv")


def sparse_mla_workspace(n_heads: int, B: int, max_rows: int, device="cuda", stream=None):
    """A zero-initialised workspace for qsa_sparse_mla_decode (allocated by torch)."""
    n = int(load().qsa_sparse_mla_workspace_size(n_heads, B, max_rows))
    if n == 0:
        raise QsaError(QSA_ERR_UNSUPPORTED, "unsupported sparse-MLA geometry")
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n]
    qsa_workspace_init(ws, stream)
    return ws


def qsa_sparse_mla_decode(q, kv_rows, rows, n_rows, out, lse, ws, softmax_scale: float = 0.0, stream=None):
    """q [B, H, 576] bf16; kv_rows [T, 656] uint8; rows [B, max_rows] int32; n_rows [B] int32;
    out [B, H, 512] bf16; lse [B, H] fp32 or None."""
    B, H = q.shape[0], q.shape[1]
    _check(load().qsa_sparse_mla_decode(_ptr(q, torch.bfloat16, "q"), H, _ptr(kv_rows, torch.uint8, "kv_rows"),
                                        kv_rows.shape[0], _ptr(rows, torch.int32, "rows"),
                                        _ptr(n_rows, torch.int32, "n_rows"), rows.shape[1], B, float(softmax_scale),
                                        _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
                                        *_ws_args(ws), _stream(stream)), "qsa_sparse_mla_decode")


def version() -> str:
    return load().qsa_version().decode()
