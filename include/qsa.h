/*
 * qsa.h — C ABI of the GB300 (sm_103a) indexer-driven sparse attention library (libqsa.so).
 *
 * The method (Qwen Sparse Attention style), as stated on
 * "3090x3で 314 万コンテキスト; KVキャッシュをホストRAMに置けるアーキテクチャの偉大さ":
 *   section "なぜ": an indexer scores every pooled 4-token block of the history
 *     (indexer_compress_ratio = 4) and keeps a fixed budget of 2048 tokens
 *     (indexer_budget = 2048, i.e. the top 512 blocks); up to 4*512+3 = 2051
 *     tokens of context everything is read;
 *   section "VRAM に残す必要があるもの": the pooled key of a block is 128 x bf16 and
 *     the indexer scans all of them every step;
 *   section "カーネルを書き換えずに済む": the gather kernel addresses
 *     K/V as (tok * n_kv_heads + kv_head) * head_dim + d;
 *   section "ちなみにこの欠点": prefill walks the history in fixed intervals
 *     (outer loop) with all chunk tokens inside (inner loop), merging softmax
 *     partials across intervals.
 * Partial results over disjoint token sets are merged by log-sum-exp
 * ("GLM-5.3 最適化 第2部：16基のH200上でのPCP、DCP、およびHybrid HiSparse", section "DCP").
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller. The library
 *    never allocates, never frees, never keeps a pointer after returning and never
 *    synchronises, except qsa_read_device_status, which synchronises the stream it is given.
 *  - The K/V cache (k_cache, v_cache) of the attention calls, and raw_idx_k of
 *    qsa_decode_step, may instead live in pinned host memory mapped into the device's
 *    address space (cudaHostAlloc, or cudaHostRegister with cudaHostRegisterMapped): the
 *    kernels then gather the selected rows over the host link ("3090x3で 314 万コンテキスト",
 *    section "VRAM に残す必要があるもの": only the pooled keys must stay on the GPU). A pointer
 *    the device cannot read at the same address returns QSA_ERR_INVALID_ARGUMENT.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream). Nothing else is launched, so the calls can be captured in a CUDA graph.
 *  - Row-major layouts; bf16 values are passed as raw 16-bit patterns (qsa_bf16).
 *  - Ragged batches are flat token arrays with int32 offsets (tok_off[s] .. tok_off[s+1]).
 *  - Host-side validation failures return immediately with nothing enqueued.
 *    A failed launch returns QSA_ERR_CUDA. Errors found on the device (an index out
 *    of range, a bounded wait that gave up) never trap: the kernel skips the access,
 *    records the first error in the workspace's status word and returns; read it
 *    with qsa_read_device_status. The status word is sticky until qsa_workspace_init.
 *  - Supported geometry: head_dim 256, idx_dim 128, indexer_compress_ratio 4,
 *    indexer_budget 2048, n_q_heads % n_kv_heads == 0, n_q_heads / n_kv_heads <= 16.
 *    Anything else returns QSA_ERR_UNSUPPORTED.
 *  - Per-thread detail of the last host-side error: qsa_last_error().
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define QSA_API __attribute__((visibility("default")))
#else
#define QSA_API
#endif

typedef enum {
    QSA_OK = 0,
    QSA_ERR_INVALID_ARGUMENT = 1,   /* null/misaligned pointer, negative size, bad stride */
    QSA_ERR_UNSUPPORTED = 2,        /* geometry outside the supported set */
    QSA_ERR_WORKSPACE_TOO_SMALL = 3,
    QSA_ERR_CUDA = 4,               /* a CUDA launch or runtime call failed */
    QSA_ERR_DEVICE_TIMEOUT = 5,     /* a bounded device-side wait gave up */
    QSA_ERR_DEVICE_BOUNDS = 6       /* a device-side index/offset check failed */
} qsa_status;

typedef enum {
    QSA_OP_POOL_KEYS = 0,
    QSA_OP_INDEX_SCORE = 1,
    QSA_OP_TOPK_BLOCKS = 2,
    QSA_OP_SPARSE_DECODE = 3,
    QSA_OP_SPARSE_PREFILL_CHUNK = 4,
    QSA_OP_DECODE_STEP = 5,
    QSA_OP_PREFILL_SELECT = 6
} qsa_op;

/* Geometry. Field names follow the model config the page quotes
 * (indexer_budget, indexer_compress_ratio, section "なぜ"). */
typedef struct {
    int32_t n_q_heads;              /* query heads (8 or 16 in the workloads) */
    int32_t n_kv_heads;             /* KV heads (2); query head h reads KV head h / (n_q_heads/n_kv_heads) */
    int32_t head_dim;               /* 256 */
    int32_t idx_dim;                /* 128: width of raw/pooled indexer keys and indexer queries */
    int32_t indexer_compress_ratio; /* 4 tokens per pooled block */
    int32_t indexer_budget;         /* 2048 tokens = 512 blocks kept per query */
    float softmax_scale;            /* <= 0 selects 1/sqrt(head_dim) */
} qsa_config;

typedef uint16_t qsa_bf16;          /* raw bf16 bits */
typedef void *qsa_stream;           /* cudaStream_t */

/* Workspace bytes an op needs for the given sizes (0 on unsupported geometry).
 * n_rows: queries (index_score/topk), sequences (decode), chunk queries (prefill).
 * max_blocks: the largest number of visible blocks of any row (topk: the scores' ld).
 * Every workspace starts with a 256-byte status block; it must be zeroed once with
 * qsa_workspace_init before first use (and after a device error). One workspace
 * may be reused by consecutive calls on the same stream; calls that run
 * concurrently need separate workspaces. */
QSA_API size_t qsa_workspace_size(int32_t op, const qsa_config *cfg, int32_t n_rows, int64_t max_blocks);

/* Zero `ws_bytes` bytes of the workspace on `stream` (clears the status word). */
QSA_API qsa_status qsa_workspace_init(void *ws, size_t ws_bytes, qsa_stream stream);

/* Synchronise `stream`, then copy the workspace's status word to *out and the
 * kernel-specific detail (e.g. the offending row) to *detail (may be NULL). */
QSA_API qsa_status qsa_read_device_status(const void *ws, qsa_stream stream, qsa_status *out, int32_t *detail);

/* Input staging helper (not a step of the method): copies n_rows rows of row_bytes bytes
 * from src (rows src_pitch bytes apart) to dst (rows dst_pitch bytes apart), host or device
 * memory on either side, asynchronously on `stream` (one strided copy, no kernel). Used
 * to append a new token's rows to per-layer caches stacked with a fixed layer stride.
 * Host memory should be pinned for the copy to be asynchronous. Errors: NULL pointers,
 * row_bytes larger than either pitch -> QSA_ERR_INVALID_ARGUMENT; n_rows == 0 copies
 * nothing. */
QSA_API qsa_status qsa_copy_rows(void *dst, size_t dst_pitch, const void *src, size_t src_pitch, size_t row_bytes,
                                 size_t n_rows, qsa_stream stream);

/* a1 — Pool indexer keys ("VRAM に残す必要があるもの": one pooled 128 x bf16 key per
 * 4-token block). For each sequence s < B and each block b in [blk_begin[s], blk_end[s]):
 *   pooled[blk_off[s] + b][d] = bf16_rne( (raw[t0][d] + raw[t0+1][d] + raw[t0+2][d] + raw[t0+3][d]) / 4 ),
 *   t0 = tok_off[s] + 4 b,
 * with the sum exact (accumulated in fp64) and a single round-to-nearest-even.
 *   raw_idx_k  [n_tokens_total, idx_dim] bf16, 16-byte aligned
 *   tok_off    [B+1] int32 (device), blk_off [B+1] int32, blk_begin [B], blk_end [B] int32
 *   pooled     [n_pooled_total, idx_dim] bf16 (written), 16-byte aligned
 *   max_blocks_per_seq: host upper bound of blk_end[s] - blk_begin[s] (sizes the grid)
 * Device checks: 0 <= blk_begin <= blk_end, blk_end - blk_begin <= max_blocks_per_seq,
 * 4*blk_end <= tokens of s, blk_off[s] + blk_end <= n_pooled_total; a failing sequence
 * is skipped and QSA_ERR_DEVICE_BOUNDS recorded. Only complete blocks are pooled. */
QSA_API qsa_status qsa_pool_keys(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, int64_t n_tokens_total,
                                 const int32_t *tok_off, const int32_t *blk_off, const int32_t *blk_begin,
                                 const int32_t *blk_end, int32_t B, int64_t max_blocks_per_seq,
                                 qsa_bf16 *pooled, int64_t n_pooled_total,
                                 void *ws, size_t ws_bytes, qsa_stream stream);

/* a2 — Indexer scores ("なぜ", "VRAM に残す必要があるもの": every pooled block is scored
 * every step). For query r < Nq with p = q_pos[r] history tokens and nb = p / 4:
 *   scores[r * ld + b] = sum_d q_idx[r][d] * pooled[blk_off[q_seq[r]] + b][d],  b < nb,
 * fp32 accumulation of exact bf16 products. Entries b >= nb are not written.
 *   q_idx [Nq, idx_dim] bf16; q_seq [Nq], q_pos [Nq] int32; pooled as above;
 *   blk_off [B+1] int32 (per-sequence pooled offsets); scores [Nq, ld] fp32.
 * q_seq may be NULL: every query then belongs to sequence 0 (a prefill chunk). With
 * Nq >= 128 and n_pooled_total >= 256 that case runs as one tensor-core GEMM ("GLM-5.3
 * 最適化 第2部": prefill scoring is quadratic) in tiles of 128 queries x 256 blocks, the
 * products summed in fp32 in the tensor core's order; otherwise one query at a time.
 * Device checks: nb <= ld, blk_off[s] + nb <= n_pooled_total. */
QSA_API qsa_status qsa_index_score(const qsa_config *cfg, const qsa_bf16 *q_idx, const int32_t *q_seq,
                                   const int32_t *q_pos, int32_t Nq, const qsa_bf16 *pooled,
                                   int64_t n_pooled_total, const int32_t *blk_off, float *scores, int64_t ld,
                                   void *ws, size_t ws_bytes, qsa_stream stream);

/* a1 with FP8 keys — pooled indexer keys stored as 128 FP8 (E4M3) codes plus one fp32 scale
 * per block ("GLM-5.3 最適化 第2部：16基のH200上でのPCP、DCP、およびHybrid HiSparse", footnote on
 * the indexer cache: 128 FP8 values and a 4-byte scale per key), so the scan of every pooled
 * block reads 132 bytes instead of 256. For each block the call first forms the bf16 pooled
 * key exactly as qsa_pool_keys does (key[d]), then
 *   scales[i] = amax / 448 (fp32 IEEE division, amax = max_d |key[d]|),
 *   codes[i][d] = E4M3(key[d] / scales[i]) (fp32 IEEE division; nearest, ties to even;
 *                 saturating at +-448),
 * with i = blk_off[s] + b; a block whose key is all zero (scale 0) gets zero codes.
 *   codes [n_pooled_total, idx_dim] uint8 (written), 16-byte aligned;
 *   scales [n_pooled_total] fp32 (written), 4-byte aligned.
 * Other arguments, the workspace (QSA_OP_POOL_KEYS) and the device checks as qsa_pool_keys. */
QSA_API qsa_status qsa_pool_keys_fp8(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, int64_t n_tokens_total,
                                     const int32_t *tok_off, const int32_t *blk_off, const int32_t *blk_begin,
                                     const int32_t *blk_end, int32_t B, int64_t max_blocks_per_seq, uint8_t *codes,
                                     float *scales, int64_t n_pooled_total, void *ws, size_t ws_bytes,
                                     qsa_stream stream);

/* a2 with FP8 keys — indexer scores against the keys qsa_pool_keys_fp8 writes. For query r
 * with nb = q_pos[r] / 4 and i = blk_off[q_seq[r]] + b:
 *   scores[r * ld + b] = scales[i] * sum_d q_idx[r][d] * codes[i][d],  b < nb,
 * with exact products and an fp32 sum, then one fp32 multiply by the scale. Entries b >= nb
 * are not written. q_seq may be NULL (every query in sequence 0). An HBM stream (no
 * tensor-core path): the CTAs resident in one wave are shared over the queries, each
 * streaming an equal range of its query's blocks. The first call on a device queries that
 * occupancy and should precede stream capture. Workspace QSA_OP_INDEX_SCORE. Device checks:
 * nb <= ld, blk_off[s] + nb <= n_pooled_total. The scores feed qsa_topk_blocks unchanged. */
QSA_API qsa_status qsa_index_score_fp8(const qsa_config *cfg, const qsa_bf16 *q_idx, const int32_t *q_seq,
                                       const int32_t *q_pos, int32_t Nq, const uint8_t *codes, const float *scales,
                                       int64_t n_pooled_total, const int32_t *blk_off, float *scores, int64_t ld,
                                       void *ws, size_t ws_bytes, qsa_stream stream);

/* a2 + a3 fused for a prefill chunk (one sequence, q_seq NULL): the same blocks and counts
 * as qsa_index_score followed by qsa_topk_blocks, without writing the score matrix
 * ("GLM-5.3 最適化 第2部": prefill scoring is quadratic; "なぜ": top-512 per query). The
 * scoring GEMM runs twice: first it keeps each row's maximum over every 64 consecutive
 * visible blocks, whose 512th largest is a floor that at least 512 scores reach; then its
 * epilogue keeps every visible score at or above the floor (exact fp32 scores, as
 * qsa_index_score computes them) and the top-k takes each row's top 512 from those. A row
 * whose candidates overflow (more than 32 in a tile of 256 blocks, e.g. many equal scores)
 * or fall short is finished on the exact path: the full scores are then written to
 * `scores` [Nq, ld] and that row streamed as by qsa_topk_blocks; otherwise `scores` is
 * not touched. Arguments as for those two calls; workspace
 * qsa_workspace_size(QSA_OP_PREFILL_SELECT, cfg, Nq, ld) (about 300 MB for 4096 queries
 * over 66,560 blocks). Needs Nq >= 128, n_pooled_total >= 256, ld <= 524288, else
 * QSA_ERR_UNSUPPORTED. */
QSA_API qsa_status qsa_prefill_select(const qsa_config *cfg, const qsa_bf16 *q_idx, const int32_t *q_pos, int32_t Nq,
                                      const qsa_bf16 *pooled, int64_t n_pooled_total, const int32_t *blk_off,
                                      float *scores, int64_t ld, int32_t *blocks, int32_t *count, void *ws,
                                      size_t ws_bytes, qsa_stream stream);

/* a3 — Fixed-budget block selection ("なぜ": exactly 2048 tokens = 512 blocks beyond 2051
 * tokens of context; all blocks below). For row r with nb = q_pos[r] / 4, k = budget/ratio:
 * the min(k, nb) blocks with the largest scores, ties to the lower block id
 * ("125B MoE を 3090 3 枚で運用する vLLM 最適化編" section 3.3 uses the same rule), written
 * to blocks[r * k ...] in ASCENDING id order; the rest of the row is set to -1;
 * count[r] = min(k, nb). NaN scores rank below every number; -0 equals +0.
 *   scores [Nq, ld] fp32 (only b < nb read); q_pos [Nq]; blocks [Nq, k] int32; count [Nq] int32. */
QSA_API qsa_status qsa_topk_blocks(const qsa_config *cfg, const float *scores, int64_t ld, const int32_t *q_pos,
                                   int32_t Nq, int32_t *blocks, int32_t *count,
                                   void *ws, size_t ws_bytes, qsa_stream stream);

/* a4 + a5 — Sparse GQA decode over the selected blocks with split partials merged by
 * log-sum-exp ("なぜ": 4 MiB of K/V per layer whatever the context; "カーネルを
 * 書き換えずに済む": K/V addressing; "GLM-5.3 最適化 第2部" section DCP: LSE merge).
 * Sequence s has its query at position p = ctx_len[s]; its tokens live at
 * tok_off[s] .. tok_off[s+1]-1 and the current token's K/V is already at index p.
 * Attended tokens J = {4b .. 4b+3 : b in blocks[s][0 .. count[s])} U {4*(p/4) .. p}.
 * For query head h (KV head h / (Hq/Hkv)):
 *   out[s][h] = sum_{j in J} softmax_j(scale * q[s][h] . K[j]) V[j],   lse[s][h] = ln sum_j e^(scale q.K[j])
 *   q [B, Hq, D] bf16; k_cache, v_cache [n_tokens_total, Hkv, D] bf16 (token-major);
 *   blocks [B, k] int32 (as written by qsa_topk_blocks; any order, no duplicates), count [B];
 *   out [B, Hq, D] bf16; lse [B, Hq] fp32 or NULL.
 * Device checks: p + 1 <= tokens of s, count <= min(k, p/4), 0 <= block < p/4. */
QSA_API qsa_status qsa_sparse_decode(const qsa_config *cfg, const qsa_bf16 *q, const qsa_bf16 *k_cache,
                                     const qsa_bf16 *v_cache, int64_t n_tokens_total, const int32_t *tok_off,
                                     const int32_t *ctx_len, int32_t B, const int32_t *blocks,
                                     const int32_t *count, qsa_bf16 *out, float *lse,
                                     void *ws, size_t ws_bytes, qsa_stream stream);

/* a6 — Prefill chunk ("ちなみにこの欠点": each chunk token selects its own 2048 tokens;
 * the history is walked interval by interval with a softmax merge). Chunk query i
 * (0 <= i < Nc) sits at p_i = p0 + i of one sequence whose K/V (history and chunk)
 * occupy tokens 0 .. p0+Nc-1; it attends exactly what qsa_sparse_decode would for
 * p = p_i with its own blocks[i] / count[i]. interval_tokens (a positive multiple of
 * 128) sets the evaluation order only, not the result.
 *   q [Nc, Hq, D] bf16; k_cache, v_cache [p0+Nc, Hkv, D] bf16;
 *   blocks [Nc, k] int32, 16-byte aligned, each row's first count[i] entries strictly
 *   ascending (as qsa_topk_blocks writes them); count [Nc]; out [Nc, Hq, D] bf16;
 *   lse [Nc, Hq] fp32 or NULL. q, k_cache, v_cache and out are 16-byte aligned.
 * With 8 or 16 query heads per KV head the chunk runs on the tensor cores in tiles of
 * 128 (query, head) rows that share each interval's union of selected blocks; a row out
 * of order there is recorded as QSA_ERR_DEVICE_BOUNDS and its tile's outputs are not
 * written. The workspace (qsa_workspace_size) then holds the tiles' chunk plan, about
 * 197 KB per 16 queries. Other head ratios run one CTA per
 * (query, KV head) on the CUDA cores. Requires (p0 + Nc) / 4 < 524288 on the tensor-core
 * path (else QSA_ERR_UNSUPPORTED). */
QSA_API qsa_status qsa_sparse_prefill_chunk(const qsa_config *cfg, const qsa_bf16 *q, int32_t p0, int32_t Nc,
                                            const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                            const int32_t *blocks, const int32_t *count, int32_t interval_tokens,
                                            qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                                            qsa_stream stream);

/* a6 staged, for K/V in host memory ("3090x3で 314 万コンテキスト", section "ちなみにこの欠点":
 * the prefill copies the history over the link into a device staging arena and computes
 * from there, so each row crosses the link once instead of once per tile that gathers it).
 * Rows [0, p0 + Nc) of k_cache and v_cache (any memory the copy engine reaches, pinned host
 * memory for an asynchronous copy) are copied into `stage` (K rows, then V rows:
 * 2 (p0 + Nc) n_kv_heads head_dim x 2 bytes, device memory, 16-byte aligned), then
 * qsa_sparse_prefill_chunk runs on the staged rows: the results are bit-identical to running
 * it on device-resident K/V. A stage shorter than needed -> QSA_ERR_WORKSPACE_TOO_SMALL;
 * a NULL or misaligned stage -> QSA_ERR_INVALID_ARGUMENT. Other arguments and errors as
 * qsa_sparse_prefill_chunk. The caller keeps the stage (an arena it may reuse for every layer). */
QSA_API qsa_status qsa_sparse_prefill_chunk_staged(const qsa_config *cfg, const qsa_bf16 *q, int32_t p0, int32_t Nc,
                                                   const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                                   const int32_t *blocks, const int32_t *count, int32_t interval_tokens,
                                                   qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes, void *stage,
                                                   size_t stage_bytes, qsa_stream stream);

/* a6 over FP8 K/V rows (the row format of qsa_quantize_kv_fp8; "GLM-5.3 最適化 第2部", footnote 1).
 * The prefill multiplies bf16 tiles on the tensor cores, so rows [0, p0 + Nc) of the K and V
 * caches are first dequantised into `stage` as qsa_dequantize_kv_fp8 does (K rows, then V
 * rows: 2 (p0 + Nc) n_kv_heads x 512 bytes of device memory, 16-byte aligned), then
 * qsa_sparse_prefill_chunk runs on the staged rows: the results are bit-identical to running it
 * on the dequantised bf16 caches. Each element is thus code x scale rounded once to bf16 (at
 * most 2^-8 of its magnitude off the exact value) before the attention.
 *   k_codes, v_codes [p0 + Nc][n_kv_heads][256] uint8, 16-byte aligned; k_scales, v_scales
 *   [p0 + Nc][n_kv_heads][2] fp32, 8-byte aligned (device memory or mapped pinned host memory).
 * A stage shorter than needed -> QSA_ERR_WORKSPACE_TOO_SMALL; a NULL or misaligned stage or
 * row pointer -> QSA_ERR_INVALID_ARGUMENT. Other arguments and errors as
 * qsa_sparse_prefill_chunk. The caller keeps the stage (an arena it may reuse for every layer). */
QSA_API qsa_status qsa_sparse_prefill_chunk_fp8kv(const qsa_config *cfg, const qsa_bf16 *q, int32_t p0, int32_t Nc,
                                                  const uint8_t *k_codes, const float *k_scales,
                                                  const uint8_t *v_codes, const float *v_scales,
                                                  const int32_t *blocks, const int32_t *count, int32_t interval_tokens,
                                                  qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes, void *stage,
                                                  size_t stage_bytes, qsa_stream stream);

/* a1-a5 fused — one decode layer-step for a batch of B <= 64 sequences in a single
 * cooperative launch ("なぜ", "VRAM に残す必要があるもの", "カーネルを書き換えずに済む";
 * LSE merge from "GLM-5.3 最適化 第2部" section DCP). For sequence s with p = ctx_len[s],
 * nb = p / 4:
 *   1. pooled[blk_off[s] + nb - 1] is (re)computed from raw_idx_k as in qsa_pool_keys (the
 *      newest block the query scores; blocks below it must already be pooled);
 *   2. every block b < nb is scored as in qsa_index_score (fp32 accumulation);
 *   3. the selection of qsa_topk_blocks is written to blocks[s] (ascending, -1 padded) and
 *      count[s];
 *   4. out[s] and lse[s] are computed as in qsa_sparse_decode over that selection.
 * Arguments have the meaning, layout and alignment they have in those calls.
 * max_blocks: host upper bound of nb over the batch (sizes the workspace:
 * qsa_workspace_size(QSA_OP_DECODE_STEP, cfg, B, max_blocks)). Requires n_kv_heads <= 2 and
 * a batch whose blocks fit the kernel's on-chip limit per CTA (else QSA_ERR_UNSUPPORTED;
 * use the separate calls then). Device errors (bounds, a bounded wait that gave up) go to
 * the workspace status word. The launch is cooperative; the first call on a device sizes
 * the grid and should precede stream capture. */
QSA_API qsa_status qsa_decode_step(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, qsa_bf16 *pooled,
                                   int64_t n_pooled_total, const int32_t *blk_off, const qsa_bf16 *q_idx,
                                   const qsa_bf16 *q, const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                   int64_t n_tokens_total, const int32_t *tok_off, const int32_t *ctx_len, int32_t B,
                                   int64_t max_blocks, int32_t *blocks, int32_t *count, qsa_bf16 *out, float *lse,
                                   void *ws, size_t ws_bytes, qsa_stream stream);

/* a1-a5 fused with FP8 keys — qsa_decode_step over the keys qsa_pool_keys_fp8 writes
 * (128 E4M3 codes + an fp32 scale per block; "GLM-5.3 最適化 第2部：16基のH200上でのPCP、DCP、
 * およびHybrid HiSparse", footnote on the indexer cache), so the scan reads 132 bytes per block
 * instead of 256. For sequence s with p = ctx_len[s], nb = p / 4:
 *   1. block blk_off[s] + nb - 1 is (re)pooled from raw_idx_k and quantised as by
 *      qsa_pool_keys_fp8 (codes and scale written);
 *   2. every block b < nb is scored as by qsa_index_score_fp8 (same products, fp32 sum order
 *      and scale multiply, hence the same fp32 scores);
 *   3.-4. selection and attention as in qsa_decode_step.
 *   codes [n_pooled_total, idx_dim] uint8, 16-byte aligned; scales [n_pooled_total] fp32,
 *   16-byte aligned. n_pooled_total must be a multiple of 4 (the scan copies whole
 *   16-byte groups of scales): pad both arrays to it. Else QSA_ERR_INVALID_ARGUMENT.
 * Other arguments, the workspace (QSA_OP_DECODE_STEP), limits and errors as qsa_decode_step. */
QSA_API qsa_status qsa_decode_step_fp8(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, uint8_t *codes,
                                       float *scales, int64_t n_pooled_total, const int32_t *blk_off,
                                       const qsa_bf16 *q_idx, const qsa_bf16 *q, const qsa_bf16 *k_cache,
                                       const qsa_bf16 *v_cache, int64_t n_tokens_total, const int32_t *tok_off,
                                       const int32_t *ctx_len, int32_t B, int64_t max_blocks, int32_t *blocks,
                                       int32_t *count, qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                                       qsa_stream stream);

/* FP8 K/V rows — the KV-row format of "GLM-5.3 最適化 第2部：16基のH200上でのPCP、DCP、および
 * Hybrid HiSparse" (footnote 1: E4M3 codes in groups of 128 dims, one fp32 scale per group)
 * applied to the GQA cache of this library. Each 256-dim row (one token's K, or V, of one KV
 * head) is two groups; for group g of row r:
 *   scales[r][g] = max_d |x[r][128 g + d]| / 448 (an fp32 IEEE division);
 *   codes[r][128 g + d] = E4M3(x[r][128 g + d] / scales[r][g]) (fp32 IEEE division, nearest
 *   even, saturated at +-448); a group of zeros has scale 0 and zero codes.
 *   x [n_rows][256] bf16, 16-byte aligned (a cache [T][Hkv][256] is n_rows = T x Hkv);
 *   codes [n_rows][256] uint8 (written), 16-byte aligned; scales [n_rows][2] fp32 (written),
 *   8-byte aligned. Device memory or mapped pinned host memory.
 * No workspace, no device-side errors (inputs are not indexed). n_rows = 0 is a no-op;
 * n_rows < 0 or above 2^34, NULL or misaligned pointers: QSA_ERR_INVALID_ARGUMENT. Non-finite
 * inputs are outside the contract. Use it to append the new token's rows to an FP8 cache. */
QSA_API qsa_status qsa_quantize_kv_fp8(const qsa_bf16 *x, int64_t n_rows, uint8_t *codes, float *scales,
                                       qsa_stream stream);

/* The inverse of qsa_quantize_kv_fp8 for computing on bf16 tiles: x[r][d] = the value
 * code_d x scales[r][d / 128] rounded once to bf16 (nearest, ties to even; magnitudes that
 * round past the largest bf16 become infinity; an E4M3 NaN code gives a NaN).
 *   codes [n_rows][256] uint8, 16-byte aligned; scales [n_rows][2] fp32, 8-byte aligned;
 *   x [n_rows][256] bf16 (written), 16-byte aligned. Device memory or mapped pinned host memory.
 * No workspace, no device-side errors. n_rows = 0 is a no-op; n_rows < 0 or above 2^34, NULL
 * or misaligned pointers: QSA_ERR_INVALID_ARGUMENT. */
QSA_API qsa_status qsa_dequantize_kv_fp8(const uint8_t *codes, const float *scales, int64_t n_rows, qsa_bf16 *x,
                                         qsa_stream stream);

/* a1-a5 fused over FP8 K/V rows — qsa_decode_step (bf16 indexer keys: `pooled`) or
 * qsa_decode_step_fp8 (FP8 indexer keys: `codes`, `scales`), with the selected tokens' K and
 * V read from FP8 rows as qsa_quantize_kv_fp8 writes them instead of bf16 rows. Give exactly
 * one key format (the other pointer(s) NULL), else QSA_ERR_INVALID_ARGUMENT.
 *   k_codes, v_codes [n_tokens_total][n_kv_heads][256] uint8, 16-byte aligned;
 *   k_scales, v_scales [n_tokens_total][n_kv_heads][2] fp32, 16-byte aligned.
 * Element d of a row has the value code_d x scale[d / 128]. The logit of query head h and
 * token t is scale_softmax x sum over the two groups of (scale_g x the fp32 sum of the
 * group's exact bf16 x E4M3 products); the output is sum_t softmax_t x (code x scale) in
 * fp32, rounded once to bf16. Selection, outputs, workspace (QSA_OP_DECODE_STEP), limits and
 * errors as qsa_decode_step; the rows (and scales) may live in mapped pinned host memory. */
QSA_API qsa_status qsa_decode_step_fp8kv(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, qsa_bf16 *pooled,
                                         uint8_t *codes, float *scales, int64_t n_pooled_total,
                                         const int32_t *blk_off, const qsa_bf16 *q_idx, const qsa_bf16 *q,
                                         const uint8_t *k_codes, const float *k_scales, const uint8_t *v_codes,
                                         const float *v_scales, int64_t n_tokens_total, const int32_t *tok_off,
                                         const int32_t *ctx_len, int32_t B, int64_t max_blocks, int32_t *blocks,
                                         int32_t *count, qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                                         qsa_stream stream);

/* f1: a VRAM row cache in front of K/V that live in host memory ("125B MoE を 3090 3 枚で運用
 * する vLLM 最適化編", section 5: consecutive decode steps select largely the same rows, so rows
 * read over the host link are kept in unused device memory). A direct-mapped cache of n_slots
 * token rows; a slot holds one token's K and V rows of every KV head (n_kv_heads x 2 x 512 B)
 * with a tag (the token's index in the flat K/V arrays), the epoch of its last hit and the
 * epoch's winning claim. Layout inside the caller's buffer: rows, then int64 tags, uint32 hit
 * epochs, uint64 claims; its size is qsa_rowcache_bytes (0 for a bad configuration, more than
 * 2 KV heads, or n_slots outside [1, 2^31]). The caller owns the buffer (device memory,
 * 16-byte aligned) and keeps one per layer. */
QSA_API size_t qsa_rowcache_bytes(const qsa_config *cfg, int64_t n_slots);

/* Empty every slot of a row cache (tags -1, hit epochs and claims 0). Call it once before the
 * first step, and again whenever rows the cache may hold change in host memory other than by
 * appending new tokens (a sequence's cache reused for another request, blocks reassigned). */
QSA_API qsa_status qsa_rowcache_init(const qsa_config *cfg, void *cache, size_t cache_bytes, int64_t n_slots,
                                     qsa_stream stream);

/* a1-a5 fused with the row cache — qsa_decode_step, for K/V (and raw indexer keys) in mapped
 * pinned host memory (or device memory), with every selected row looked up in `cache` first.
 * Sequence s owns slots [s n_slots / B, (s + 1) n_slots / B); token t of it maps to slot
 * lo_s + t mod (its slot count). Per step (`epoch`: at least 1, larger than at every earlier
 * call with this cache):
 *   - a selected token whose slot's tag is the token's flat index is read from the cache and
 *     the slot is marked as hit in this epoch; any other selected token is read from k_cache /
 *     v_cache and claims its slot with an atomic max of (epoch << 32 | flat index);
 *   - after every CTA of the sequence has read its rows, a claim's winner writes the row and
 *     the tag, unless some token hit the slot in this epoch (the rows of each CTA's last two
 *     chunks of at most 32 tokens each are written, any earlier ones stay uncached this step).
 * The query's own (incomplete) block is always read from k_cache / v_cache and never cached:
 * the caller may still be writing it. Hits return exactly the bytes in host memory, so the
 * outputs equal qsa_decode_step's bit for bit. Cache errors: NULL or misaligned cache,
 * n_slots < B or above 2^31, epoch 0 -> QSA_ERR_INVALID_ARGUMENT; cache_bytes short ->
 * QSA_ERR_WORKSPACE_TOO_SMALL. Everything else (bf16 keys and K/V only) as qsa_decode_step. */
QSA_API qsa_status qsa_decode_step_rowcache(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, qsa_bf16 *pooled,
                                            int64_t n_pooled_total, const int32_t *blk_off, const qsa_bf16 *q_idx,
                                            const qsa_bf16 *q, const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                            int64_t n_tokens_total, const int32_t *tok_off, const int32_t *ctx_len,
                                            int32_t B, int64_t max_blocks, int32_t *blocks, int32_t *count,
                                            qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes, void *cache,
                                            size_t cache_bytes, int64_t n_slots, uint32_t epoch, qsa_stream stream);

/* a1-a5 fused, with an L2 prefetch hint — qsa_decode_step (and qsa_decode_step_fp8) plus
 * the memory the caller's next call will read, typically the next layer's pooled keys (or
 * FP8 codes). Each CTA, once its own pooled-key stream is done, issues L2 prefetch hints for
 * its slice of [next_read, next_read + next_read_bytes), so the bytes the next layer-step
 * scans arrive in L2 while this step exchanges keys and partials (those phases leave HBM
 * idle). The next layer's keys do not depend on this step's output; nothing of the next
 * step is computed here. A hint only: results are bit-identical to qsa_decode_step's.
 *   next_read: 16-byte aligned, device memory or mapped pinned host memory, or NULL (no
 *   hint); next_read_bytes is rounded down to a multiple of 16 (below 16: no hint).
 * Everything else as qsa_decode_step / qsa_decode_step_fp8. A misaligned or unreadable
 * next_read is QSA_ERR_INVALID_ARGUMENT. */
QSA_API qsa_status qsa_decode_step_prefetch(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, qsa_bf16 *pooled,
                                            int64_t n_pooled_total, const int32_t *blk_off, const qsa_bf16 *q_idx,
                                            const qsa_bf16 *q, const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                            int64_t n_tokens_total, const int32_t *tok_off, const int32_t *ctx_len,
                                            int32_t B, int64_t max_blocks, int32_t *blocks, int32_t *count,
                                            qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                                            const void *next_read, size_t next_read_bytes, qsa_stream stream);
QSA_API qsa_status qsa_decode_step_fp8_prefetch(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, uint8_t *codes,
                                                float *scales, int64_t n_pooled_total, const int32_t *blk_off,
                                                const qsa_bf16 *q_idx, const qsa_bf16 *q, const qsa_bf16 *k_cache,
                                                const qsa_bf16 *v_cache, int64_t n_tokens_total,
                                                const int32_t *tok_off, const int32_t *ctx_len, int32_t B,
                                                int64_t max_blocks, int32_t *blocks, int32_t *count, qsa_bf16 *out,
                                                float *lse, void *ws, size_t ws_bytes, const void *next_read,
                                                size_t next_read_bytes, qsa_stream stream);

/* Allocation-free variant of qsa_sparse_decode (the pages have no counterpart; this
 * is a library convenience). Same arguments and result, but no workspace: the split
 * partials live in a 16 MiB static device array inside the library, for callers that
 * cannot allocate device memory at all (a plug-in inside a host application that owns
 * the whole device memory pool, a process whose device memory another allocator has
 * fully reserved, loops that must not risk an allocation's implicit synchronisation).
 *  - Limit: qsa_workspace_size(QSA_OP_SPARSE_DECODE, cfg, B, 0) must not exceed 16 MiB
 *    (B <= 30 at 16 query / 2 KV heads, B <= 61 at 8 / 2); larger batches return
 *    QSA_ERR_WORKSPACE_TOO_SMALL. Every host check (configuration, sizes, pointers, the
 *    stream's device) runs before anything is enqueued.
 *  - `stream` must belong to the current device (else QSA_ERR_INVALID_ARGUMENT): the
 *    array has one address per device.
 *  - The first call on a device resolves the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it.
 *  - The array stays resident on every GPU that loads the library until exit.
 *  - Every call reuses the same array: calls that overlap on the GPU race. Each call
 *    clears the array's status block on `stream`; device-side bounds errors are not
 *    reported (the bad access is still skipped). It never calls cudaMalloc/cudaFree. */
QSA_API qsa_status qsa_sparse_decode_noalloc(const qsa_config *cfg, const qsa_bf16 *q, const qsa_bf16 *k_cache,
                                             const qsa_bf16 *v_cache, int64_t n_tokens_total,
                                             const int32_t *tok_off, const int32_t *ctx_len, int32_t B,
                                             const int32_t *blocks, const int32_t *count, qsa_bf16 *out,
                                             float *lse, qsa_stream stream);

/* f3 — Sparse MLA decode in its MQA form ("GLM-5.3 最適化 第2部：16基のH200上でのPCP、DCP、
 * およびHybrid HiSparse", footnote 1: each query reads 2,048 selected FP8 rows of 656 bytes;
 * QK runs over 576 dims, PV over 512; every row serves all heads). Row layout, 656 bytes:
 *   bytes 0..511   the 512-dim latent as E4M3 codes (dim d at byte d),
 *   bytes 512..527 four fp32 scales (scale g applies to latent dims 128g .. 128g+127),
 *   bytes 528..655 the 64 rotary dims as bf16.
 * With latent_j = code x scale and k_j = [latent_j, rope_j], query b's head h gives
 *   out[b][h] = sum_j softmax_j(scale_qk * q[b][h] . k_j) latent_j,  lse[b][h] = ln sum_j e^(...)
 * over j in rows[b][0 .. n_rows[b]) (token ids, any order, no repeats).
 *   q [B, n_heads, 576] bf16, 16-byte aligned; kv_rows [n_tokens, 656] uint8, 16-byte aligned;
 *   rows [B, max_rows] int32; n_rows [B] int32 (<= max_rows); out [B, n_heads, 512] bf16;
 *   lse [B, n_heads] fp32 or NULL; softmax_scale <= 0 selects 1/sqrt(576).
 * Tensor cores: tiles of 64 selected rows; latent values rounded once to bf16 for the MMA
 * (code x scale in fp32, then bf16), P rounded to bf16; fp32 accumulation; the tiles'
 * partials merged by log-sum-exp. n_heads 1..128 (MMA rows; else QSA_ERR_UNSUPPORTED).
 * Workspace: qsa_sparse_mla_workspace_size(n_heads, B, max_rows) bytes (status block + the
 * tiles' partials); device checks: 0 <= row id < n_tokens (a bad row is skipped and
 * QSA_ERR_DEVICE_BOUNDS recorded); n_rows[b] is clamped to [0, max_rows], a value above
 * max_rows also recording QSA_ERR_DEVICE_BOUNDS. A query with no rows gets out = 0 and
 * lse = -inf. */
QSA_API size_t qsa_sparse_mla_workspace_size(int32_t n_heads, int32_t B, int32_t max_rows);
QSA_API qsa_status qsa_sparse_mla_decode(const qsa_bf16 *q, int32_t n_heads, const uint8_t *kv_rows,
                                         int64_t n_tokens, const int32_t *rows, const int32_t *n_rows,
                                         int32_t max_rows, int32_t B, float softmax_scale, qsa_bf16 *out, float *lse,
                                         void *ws, size_t ws_bytes, qsa_stream stream);

/* Static description of a status code. */
QSA_API const char *qsa_status_string(qsa_status s);

/* Detail of the last host-side error on the calling thread ("" if none). */
QSA_API const char *qsa_last_error(void);

/* Library version, e.g. "qsa-gb300 0.1.0 sm_103a". */
QSA_API const char *qsa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H */
