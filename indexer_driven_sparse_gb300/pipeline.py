"""Device buffers and call sequences for one decode layer-step or one prefill chunk.

Only marshalling: torch allocates the buffers and the metadata tensors, and every
step of the path runs in libqsa.so through the ``qsa_*`` calls of :mod:`.binding`.
"""

from __future__ import annotations

import torch

from . import binding as qb

RATIO = 4


class DecodeBatch:
    """A ragged decode batch: sequence s has its query at p = ctx_len[s] and p + 1
    cached tokens at tok_off[s] .. tok_off[s+1]-1 of the flat K/V arrays."""

    def __init__(self, n_q_heads: int, n_kv_heads: int, ctx_len, device="cuda", softmax_scale: float = 0.0):
        self.cfg = qb.make_config(n_q_heads, n_kv_heads, softmax_scale=softmax_scale)
        self.ctx = [int(p) for p in ctx_len]
        self.B = len(self.ctx)
        self.device = device
        i32 = dict(dtype=torch.int32, device=device)
        tok_off, blk_off, nblk = [0], [0], []
        for p in self.ctx:
            tok_off.append(tok_off[-1] + p + 1)
            nblk.append((p + 1) // RATIO)          # complete blocks among the p+1 cached tokens
            blk_off.append(blk_off[-1] + nblk[-1])
        self.n_tokens = tok_off[-1]
        self.n_pooled = blk_off[-1]
        self.max_blocks = max(nblk) if nblk else 0
        self.ld = max(1, max((p // RATIO for p in self.ctx), default=1))
        self.tok_off = torch.tensor(tok_off, **i32)
        self.blk_off = torch.tensor(blk_off, **i32)
        self.ctx_len = torch.tensor(self.ctx, **i32)
        self.q_seq = torch.arange(self.B, **i32)
        self.blk_begin = torch.zeros(self.B, **i32)
        self.blk_end = torch.tensor(nblk, **i32)
        self.scores = torch.empty(self.B, self.ld, dtype=torch.float32, device=device)
        self.blocks = torch.empty(self.B, qb.BLOCK_TOPK, **i32)
        self.count = torch.empty(self.B, **i32)
        self.out = torch.empty(self.B, n_q_heads, 256, dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(self.B, n_q_heads, dtype=torch.float32, device=device)
        sizes = [qb.workspace_size(qb.OP_POOL_KEYS, self.cfg, self.B, self.max_blocks),
                 qb.workspace_size(qb.OP_INDEX_SCORE, self.cfg, self.B, self.ld),
                 qb.workspace_size(qb.OP_TOPK_BLOCKS, self.cfg, self.B, self.ld),
                 qb.workspace_size(qb.OP_SPARSE_DECODE, self.cfg, self.B, self.ld)]
        self.ws = _workspace(max(sizes), device)
        self.step_ws = None
        if self.B <= 64:
            n = qb.workspace_size(qb.OP_DECODE_STEP, self.cfg, self.B, self.ld)
            if n:
                self.step_ws = _workspace(n, device)

    def new_pooled(self):
        return torch.empty(max(self.n_pooled, 1), 128, dtype=torch.bfloat16, device=self.device)

    def fused_step(self, raw_idx_k, pooled, q_idx, q, k_cache, v_cache, stream=None, next_read=None):
        """One decode layer-step in one launch (qsa_decode_step): re-pool the newest
        block, score, select, attend, merge. `next_read` (e.g. the next layer's pooled
        keys) is prefetched into L2 while the step exchanges keys and partials."""
        qb.qsa_decode_step(self.cfg, raw_idx_k, pooled, self.blk_off, q_idx, q, k_cache, v_cache, self.tok_off,
                           self.ctx_len, self.ld, self.blocks, self.count, self.out, self.lse, self.step_ws, stream,
                           next_read)

    def fused_step_fp8(self, raw_idx_k, codes, scales, q_idx, q, k_cache, v_cache, stream=None, next_read=None):
        """qsa_decode_step over FP8 indexer keys (qsa_decode_step_fp8)."""
        qb.qsa_decode_step_fp8(self.cfg, raw_idx_k, codes, scales, self.blk_off, q_idx, q, k_cache, v_cache,
                               self.tok_off, self.ctx_len, self.ld, self.blocks, self.count, self.out, self.lse,
                               self.step_ws, stream, next_read)

    def fused_step_fp8kv(self, raw_idx_k, keys, q_idx, q, kv8, stream=None):
        """The fused step over FP8 K/V rows (qsa_decode_step_fp8kv). `keys` is the bf16 pooled-key
        tensor or a (codes, scales) pair of FP8 keys; `kv8` is (k_codes, k_scales, v_codes,
        v_scales) as qsa_quantize_kv_fp8 writes them."""
        pooled, codes, scales = (keys, None, None) if torch.is_tensor(keys) else (None, *keys)
        qb.qsa_decode_step_fp8kv(self.cfg, raw_idx_k, pooled, codes, scales, self.blk_off, q_idx, q, *kv8,
                                 self.tok_off, self.ctx_len, self.ld, self.blocks, self.count, self.out, self.lse,
                                 self.step_ws, stream)

    def fused_step_rowcache(self, raw_idx_k, pooled, q_idx, q, k_cache, v_cache, cache, n_slots, epoch, stream=None):
        """qsa_decode_step with the VRAM row cache `cache` (binding.rowcache_new) in front of
        K/V in host memory; `epoch` grows by at least one per call with the same cache."""
        qb.qsa_decode_step_rowcache(self.cfg, raw_idx_k, pooled, self.blk_off, q_idx, q, k_cache, v_cache,
                                    self.tok_off, self.ctx_len, self.ld, self.blocks, self.count, self.out, self.lse,
                                    self.step_ws, cache, n_slots, epoch, stream)

    def fused_status(self, stream=None):
        return qb.qsa_read_device_status(self.step_ws, stream)

    def pool(self, raw_idx_k, pooled, stream=None):
        qb.qsa_pool_keys(self.cfg, raw_idx_k, self.tok_off, self.blk_off, self.blk_begin, self.blk_end,
                         self.max_blocks, pooled, self.ws, stream)

    def score(self, q_idx, pooled, stream=None):
        qb.qsa_index_score(self.cfg, q_idx, self.q_seq, self.ctx_len, pooled, self.blk_off, self.scores, self.ws,
                           stream)

    def topk(self, stream=None):
        qb.qsa_topk_blocks(self.cfg, self.scores, self.ctx_len, self.blocks, self.count, self.ws, stream)

    def attend(self, q, k_cache, v_cache, blocks=None, count=None, stream=None):
        qb.qsa_sparse_decode(self.cfg, q, k_cache, v_cache, self.tok_off, self.ctx_len,
                             self.blocks if blocks is None else blocks, self.count if count is None else count,
                             self.out, self.lse, self.ws, stream)

    def step(self, q_idx, q, k_cache, v_cache, pooled, stream=None):
        """One decode layer-step: score -> top-k -> sparse attention + LSE merge."""
        self.score(q_idx, pooled, stream)
        self.topk(stream)
        self.attend(q, k_cache, v_cache, stream=stream)

    def new_fp8_keys(self):
        """Buffers of the FP8 indexer keys: codes [n, 128] uint8 and scales [n] fp32, n = the
        pooled block count padded to a multiple of 4 (the fused step copies whole groups of 4 scales)."""
        n = max((self.n_pooled + 3) // 4 * 4, 4)
        return (torch.empty(n, 128, dtype=torch.uint8, device=self.device),
                torch.empty(n, dtype=torch.float32, device=self.device))

    def pool_fp8(self, raw_idx_k, codes, scales, stream=None):
        qb.qsa_pool_keys_fp8(self.cfg, raw_idx_k, self.tok_off, self.blk_off, self.blk_begin, self.blk_end,
                             self.max_blocks, codes, scales, self.ws, stream)

    def score_fp8(self, q_idx, codes, scales, stream=None):
        qb.qsa_index_score_fp8(self.cfg, q_idx, self.q_seq, self.ctx_len, codes, scales, self.blk_off, self.scores,
                               self.ws, stream)

    def step_fp8(self, q_idx, q, k_cache, v_cache, codes, scales, stream=None):
        """One decode layer-step with FP8 indexer keys: score -> top-k -> sparse attention."""
        self.score_fp8(q_idx, codes, scales, stream)
        self.topk(stream)
        self.attend(q, k_cache, v_cache, stream=stream)

    def device_status(self, stream=None):
        return qb.qsa_read_device_status(self.ws, stream)


class PrefillChunk:
    """A chunk of Nc queries at positions p0 .. p0+Nc-1 of one sequence whose cache
    holds p0 + Nc tokens (the chunk's K/V already appended)."""

    def __init__(self, n_q_heads: int, n_kv_heads: int, p0: int, n_chunk: int, interval_tokens: int = 8192,
                 device="cuda", softmax_scale: float = 0.0):
        self.cfg = qb.make_config(n_q_heads, n_kv_heads, softmax_scale=softmax_scale)
        self.p0, self.Nc, self.interval = int(p0), int(n_chunk), int(interval_tokens)
        self.device = device
        i32 = dict(dtype=torch.int32, device=device)
        self.n_tokens = self.p0 + self.Nc
        self.n_pooled = self.n_tokens // RATIO
        # score rows padded to 32 floats (128 bytes): aligned line writes and vector reads
        self.ld = max(1, (self.p0 + self.Nc - 1) // RATIO + 31) // 32 * 32
        self.tok_off = torch.tensor([0, self.n_tokens], **i32)
        self.blk_off = torch.zeros(2, **i32)
        self.q_seq = torch.zeros(self.Nc, **i32)
        self.q_pos = torch.arange(self.p0, self.p0 + self.Nc, **i32)
        self.scores = torch.empty(self.Nc, self.ld, dtype=torch.float32, device=device)
        self.blocks = torch.empty(self.Nc, qb.BLOCK_TOPK, **i32)
        self.count = torch.empty(self.Nc, **i32)
        self.out = torch.empty(self.Nc, n_q_heads, 256, dtype=torch.bfloat16, device=device)
        self.lse = torch.empty(self.Nc, n_q_heads, dtype=torch.float32, device=device)
        sizes = [qb.workspace_size(qb.OP_POOL_KEYS, self.cfg, 1, self.n_pooled),
                 qb.workspace_size(qb.OP_INDEX_SCORE, self.cfg, self.Nc, self.ld),
                 qb.workspace_size(qb.OP_TOPK_BLOCKS, self.cfg, self.Nc, self.ld),
                 qb.workspace_size(qb.OP_SPARSE_PREFILL_CHUNK, self.cfg, self.Nc, self.ld)]
        # scoring and top-k fused (no score matrix) for chunks of at least one 128-query tile
        self.fused_select = self.Nc >= 128 and self.n_pooled >= 256
        if self.fused_select:
            sizes.append(qb.workspace_size(qb.OP_PREFILL_SELECT, self.cfg, self.Nc, self.ld))
        self.ws = _workspace(max(sizes), device)

    def new_pooled(self):
        return torch.empty(max(self.n_pooled, 1), 128, dtype=torch.bfloat16, device=self.device)

    def pool(self, raw_idx_k, pooled, first_block: int = 0, stream=None):
        """Pool blocks [first_block, (p0+Nc)//4) (the whole history, or just the chunk's)."""
        i32 = dict(dtype=torch.int32, device=self.device)
        qb.qsa_pool_keys(self.cfg, raw_idx_k, self.tok_off, self.blk_off, torch.tensor([first_block], **i32),
                         torch.tensor([self.n_pooled], **i32), max(0, self.n_pooled - first_block), pooled, self.ws,
                         stream)

    def score(self, q_idx, pooled, stream=None, gemm=True):
        """All chunk queries share one history: with gemm the call passes no per-query
        sequence ids, which selects the tensor-core GEMM; otherwise one query at a time."""
        qb.qsa_index_score(self.cfg, q_idx, None if gemm else self.q_seq, self.q_pos, pooled, self.blk_off,
                           self.scores, self.ws, stream)

    def topk(self, stream=None):
        qb.qsa_topk_blocks(self.cfg, self.scores, self.q_pos, self.blocks, self.count, self.ws, stream)

    def select(self, q_idx, pooled, stream=None):
        """Scores and top-k in one call without the score matrix (qsa_prefill_select)."""
        qb.qsa_prefill_select(self.cfg, q_idx, self.q_pos, pooled, self.blk_off, self.scores, self.blocks, self.count,
                              self.ws, stream)

    def attend(self, q, k_cache, v_cache, blocks=None, count=None, stream=None):
        qb.qsa_sparse_prefill_chunk(self.cfg, q, self.p0, k_cache, v_cache,
                                    self.blocks if blocks is None else blocks,
                                    self.count if count is None else count, self.interval, self.out, self.lse,
                                    self.ws, stream)

    def attend_staged(self, q, k_cache, v_cache, stage, stream=None):
        """attend() with K/V (e.g. in pinned host memory) copied into the device arena `stage`
        first (qsa_sparse_prefill_chunk_staged)."""
        qb.qsa_sparse_prefill_chunk_staged(self.cfg, q, self.p0, k_cache, v_cache, self.blocks, self.count,
                                           self.interval, self.out, self.lse, self.ws, stage, stream)

    def attend_fp8kv(self, q, kv8, stage, stream=None):
        """attend() over FP8 K/V rows kv8 = (k_codes, k_scales, v_codes, v_scales), dequantised
        into the device arena `stage` first (qsa_sparse_prefill_chunk_fp8kv)."""
        qb.qsa_sparse_prefill_chunk_fp8kv(self.cfg, q, self.p0, kv8, self.blocks, self.count, self.interval,
                                          self.out, self.lse, self.ws, stage, stream)

    def run(self, q_idx, q, k_cache, v_cache, pooled, stream=None):
        """The chunk's path after pooling: score -> top-k (fused when the chunk has a full
        query tile) -> interval-walk attention."""
        if self.fused_select:
            self.select(q_idx, pooled, stream)
        else:
            self.score(q_idx, pooled, stream)
            self.topk(stream)
        self.attend(q, k_cache, v_cache, stream=stream)

    def device_status(self, stream=None):
        return qb.qsa_read_device_status(self.ws, stream)


def _workspace(nbytes: int, device):
    ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + nbytes]
    qb.qsa_workspace_init(ws)
    return ws
