// extern "C" entry points of libqsa.so: host-side validation, workspace layout and
// launch on the caller's stream. No allocation and no synchronisation happen here
// (except qsa_read_device_status, which synchronises by design).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>

#include "qsa_internal.cuh"
#include "kv_fp8.cuh"

using namespace qsa;

namespace qsa {
// Sparse MLA decode, MQA form, on the tensor cores (mla.cu).
size_t mla_scratch_bytes(int H, int B, int max_rows);
cudaError_t launch_sparse_mla(const uint16_t *q, int H, const uint8_t *kv, int64_t n_tok, const int32_t *rows,
                              const int32_t *n_rows, int max_rows, int B, float scale, uint16_t *out, float *lse,
                              WsHeader *hdr, void *scratch, cudaStream_t st);
}  // namespace qsa

namespace {

thread_local char g_last_error[512] = "";

qsa_status fail(qsa_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return s;
}

qsa_status ok() {
    g_last_error[0] = '\0';
    return QSA_OK;
}

qsa_status cuda_fail(cudaError_t e, const char *what) {
    return fail(QSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qsa_status check_config(const qsa_config *c) {
    if (c == nullptr) return fail(QSA_ERR_INVALID_ARGUMENT, "config is NULL");
    if (c->head_dim != kHeadDim) return fail(QSA_ERR_UNSUPPORTED, "head_dim %d (only 256)", c->head_dim);
    if (c->idx_dim != kIdxDim) return fail(QSA_ERR_UNSUPPORTED, "idx_dim %d (only 128)", c->idx_dim);
    if (c->indexer_compress_ratio != kRatio)
        return fail(QSA_ERR_UNSUPPORTED, "indexer_compress_ratio %d (only 4)", c->indexer_compress_ratio);
    if (c->indexer_budget != kRatio * kBlockTopK)
        return fail(QSA_ERR_UNSUPPORTED, "indexer_budget %d (only 2048)", c->indexer_budget);
    if (c->n_kv_heads < 1 || c->n_q_heads < 1)
        return fail(QSA_ERR_INVALID_ARGUMENT, "head counts must be positive (%d, %d)", c->n_q_heads, c->n_kv_heads);
    if (c->n_q_heads % c->n_kv_heads != 0)
        return fail(QSA_ERR_UNSUPPORTED, "n_q_heads %d not a multiple of n_kv_heads %d", c->n_q_heads, c->n_kv_heads);
    const int g = c->n_q_heads / c->n_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16)
        return fail(QSA_ERR_UNSUPPORTED, "query heads per KV head %d (1, 2, 4, 8 or 16)", g);
    if (c->n_q_heads * (int64_t)kHeadDim > (1 << 20)) return fail(QSA_ERR_UNSUPPORTED, "too many heads");
    if (!(c->softmax_scale <= 0.f) && !isfinite(c->softmax_scale))
        return fail(QSA_ERR_INVALID_ARGUMENT, "softmax_scale must be finite");
    return QSA_OK;
}

float scale_of(const qsa_config *c) {
    return c->softmax_scale > 0.f ? c->softmax_scale : 1.0f / sqrtf((float)c->head_dim);
}

size_t ws_size(int32_t op, const qsa_config *c, int32_t n_rows, int64_t max_blocks) {
    if (n_rows < 0 || max_blocks < 0) return 0;
    switch (op) {
        case QSA_OP_POOL_KEYS:
        case QSA_OP_INDEX_SCORE: return kWsHeaderBytes;
        case QSA_OP_TOPK_BLOCKS: return kWsHeaderBytes + topk_scratch_bytes(n_rows, max_blocks);
        case QSA_OP_SPARSE_DECODE: return kWsHeaderBytes + decode_scratch_bytes(n_rows, c->n_q_heads, c->n_kv_heads);
        case QSA_OP_SPARSE_PREFILL_CHUNK:
            return kWsHeaderBytes + prefill_scratch_bytes(n_rows, c->n_q_heads, c->n_kv_heads);
        case QSA_OP_DECODE_STEP: return decode_step_ws_bytes(n_rows, max_blocks, c->n_q_heads);
        case QSA_OP_PREFILL_SELECT: return kWsHeaderBytes + prefill_select_scratch_bytes(n_rows, max_blocks);
        default: return 0;
    }
}

qsa_status check_ws(int32_t op, const qsa_config *c, int32_t n_rows, int64_t max_blocks, void *ws, size_t bytes) {
    if (ws == nullptr) return fail(QSA_ERR_INVALID_ARGUMENT, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(QSA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
    const size_t need = ws_size(op, c, n_rows, max_blocks);
    if (bytes < need) return fail(QSA_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", bytes, need);
    return QSA_OK;
}

#define QSA_TRY(expr)                         \
    do {                                      \
        const qsa_status _s = (expr);         \
        if (_s != QSA_OK) return _s;          \
    } while (0)

#define QSA_NEED(cond, ...)                                           \
    do {                                                              \
        if (!(cond)) return fail(QSA_ERR_INVALID_ARGUMENT, __VA_ARGS__); \
    } while (0)

constexpr int kMaxGridYZ = 65535;

}  // namespace

qsa_status qsa::host_fail(qsa_status s, const char *what, const char *detail) {
    return fail(s, "%s: %s", what, detail);
}

extern "C" {

QSA_API size_t qsa_workspace_size(int32_t op, const qsa_config *cfg, int32_t n_rows, int64_t max_blocks) {
    if (check_config(cfg) != QSA_OK) return 0;
    return ws_size(op, cfg, n_rows, max_blocks);
}

// The GPU reads p at the same address: device or managed memory, or pinned host memory mapped
// into the device's address space (cudaHostAlloc; cudaHostRegister with the mapped flag) -
// the K/V cache may live in host memory and be gathered over the host link.
static bool device_accessible(const void *p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    switch (at.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged: return true;
        case cudaMemoryTypeHost: return at.devicePointer == p;
        default: return false;
    }
}

QSA_API qsa_status qsa_workspace_init(void *ws, size_t ws_bytes, qsa_stream stream) {
    QSA_NEED(ws != nullptr, "workspace is NULL");
    QSA_NEED(ws_bytes >= kWsHeaderBytes, "workspace smaller than its 256-byte status block");
    const cudaError_t e = cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    return ok();
}

QSA_API qsa_status qsa_copy_rows(void *dst, size_t dst_pitch, const void *src, size_t src_pitch, size_t row_bytes,
                                 size_t n_rows, qsa_stream stream) {
    if (n_rows == 0 || row_bytes == 0) return ok();
    QSA_NEED(dst != nullptr && src != nullptr, "dst and src must be non-NULL");
    QSA_NEED(row_bytes <= dst_pitch && row_bytes <= src_pitch, "row_bytes exceeds a pitch");
    const cudaError_t e = cudaMemcpy2DAsync(dst, dst_pitch, src, src_pitch, row_bytes, n_rows, cudaMemcpyDefault,
                                            static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy2DAsync");
    return ok();
}

QSA_API qsa_status qsa_read_device_status(const void *ws, qsa_stream stream, qsa_status *out, int32_t *detail) {
    QSA_NEED(ws != nullptr && out != nullptr, "workspace and out must be non-NULL");
    int32_t h[3] = {0, 0, 0};
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    e = cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy status");
    *out = static_cast<qsa_status>(h[0]);
    if (detail != nullptr) *detail = h[1];
    return ok();
}

QSA_API qsa_status qsa_pool_keys(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, int64_t n_tokens_total,
                                 const int32_t *tok_off, const int32_t *blk_off, const int32_t *blk_begin,
                                 const int32_t *blk_end, int32_t B, int64_t max_blocks_per_seq, qsa_bf16 *pooled,
                                 int64_t n_pooled_total, void *ws, size_t ws_bytes, qsa_stream stream) {
    QSA_TRY(check_config(cfg));
    QSA_NEED(B >= 0 && B <= kMaxGridYZ, "B = %d out of range [0, 65535]", B);
    QSA_NEED(n_tokens_total >= 0 && n_pooled_total >= 0 && max_blocks_per_seq >= 0, "negative size");
    QSA_NEED(max_blocks_per_seq <= (int64_t)1 << 28, "max_blocks_per_seq too large");
    QSA_TRY(check_ws(QSA_OP_POOL_KEYS, cfg, B, max_blocks_per_seq, ws, ws_bytes));
    if (B == 0 || max_blocks_per_seq == 0) return ok();
    QSA_NEED(raw_idx_k && pooled && tok_off && blk_off && blk_begin && blk_end, "NULL tensor pointer");
    QSA_NEED(aligned(raw_idx_k, 16) && aligned(pooled, 16), "raw_idx_k and pooled must be 16-byte aligned");
    const cudaError_t e = launch_pool_keys(raw_idx_k, n_tokens_total, tok_off, blk_off, blk_begin, blk_end, B,
                                           max_blocks_per_seq, pooled, n_pooled_total,
                                           static_cast<WsHeader *>(ws), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pool_keys launch");
    return ok();
}

QSA_API qsa_status qsa_index_score(const qsa_config *cfg, const qsa_bf16 *q_idx, const int32_t *q_seq,
                                   const int32_t *q_pos, int32_t Nq, const qsa_bf16 *pooled, int64_t n_pooled_total,
                                   const int32_t *blk_off, float *scores, int64_t ld, void *ws, size_t ws_bytes,
                                   qsa_stream stream) {
    QSA_TRY(check_config(cfg));
    QSA_NEED(Nq >= 0 && Nq <= kMaxGridYZ, "Nq = %d out of range [0, 65535]", Nq);
    QSA_NEED(ld >= 0 && n_pooled_total >= 0, "negative size");
    QSA_NEED(ld <= (int64_t)1 << 28, "ld too large");
    QSA_TRY(check_ws(QSA_OP_INDEX_SCORE, cfg, Nq, ld, ws, ws_bytes));
    if (Nq == 0 || ld == 0) return ok();
    QSA_NEED(q_idx && q_pos && pooled && blk_off && scores, "NULL tensor pointer");
    QSA_NEED(aligned(q_idx, 16) && aligned(pooled, 16), "q_idx and pooled must be 16-byte aligned");
    QSA_NEED(aligned(scores, 4), "scores must be 4-byte aligned");
    // one sequence with many queries (a prefill chunk): a tensor-core GEMM
    const bool gemm = q_seq == nullptr && score_tc_supported(Nq, n_pooled_total);
    const cudaError_t e =
        gemm ? launch_score_tc(q_idx, q_pos, Nq, pooled, n_pooled_total, blk_off, scores, ld,
                               static_cast<WsHeader *>(ws), static_cast<cudaStream_t>(stream))
             : launch_index_score(q_idx, q_seq, q_pos, Nq, pooled, n_pooled_total, blk_off, scores, ld,
                                  static_cast<WsHeader *>(ws), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "index_score launch");
    return ok();
}

QSA_API qsa_status qsa_pool_keys_fp8(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, int64_t n_tokens_total,
                                     const int32_t *tok_off, const int32_t *blk_off, const int32_t *blk_begin,
                                     const int32_t *blk_end, int32_t B, int64_t max_blocks_per_seq, uint8_t *codes,
                                     float *scales, int64_t n_pooled_total, void *ws, size_t ws_bytes,
                                     qsa_stream stream) {
    QSA_TRY(check_config(cfg));
    QSA_NEED(B >= 0 && B <= kMaxGridYZ, "B = %d out of range [0, 65535]", B);
    QSA_NEED(n_tokens_total >= 0 && n_pooled_total >= 0 && max_blocks_per_seq >= 0, "negative size");
    QSA_NEED(max_blocks_per_seq <= (int64_t)1 << 28, "max_blocks_per_seq too large");
    QSA_TRY(check_ws(QSA_OP_POOL_KEYS, cfg, B, max_blocks_per_seq, ws, ws_bytes));
    if (B == 0 || max_blocks_per_seq == 0) return ok();
    QSA_NEED(raw_idx_k && codes && scales && tok_off && blk_off && blk_begin && blk_end, "NULL tensor pointer");
    QSA_NEED(aligned(raw_idx_k, 16) && aligned(codes, 16), "raw_idx_k and codes must be 16-byte aligned");
    QSA_NEED(aligned(scales, 4), "scales must be 4-byte aligned");
    const cudaError_t e = launch_pool_keys_fp8(raw_idx_k, n_tokens_total, tok_off, blk_off, blk_begin, blk_end, B,
                                               max_blocks_per_seq, codes, scales, n_pooled_total,
                                               static_cast<WsHeader *>(ws), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "pool_keys_fp8 launch");
    return ok();
}

QSA_API qsa_status qsa_index_score_fp8(const qsa_config *cfg, const qsa_bf16 *q_idx, const int32_t *q_seq,
                                       const int32_t *q_pos, int32_t Nq, const uint8_t *codes, const float *scales,
                                       int64_t n_pooled_total, const int32_t *blk_off, float *scores, int64_t ld,
                                       void *ws, size_t ws_bytes, qsa_stream stream) {
    QSA_TRY(check_config(cfg));
    QSA_NEED(Nq >= 0 && Nq <= kMaxGridYZ, "Nq = %d out of range [0, 65535]", Nq);
    QSA_NEED(ld >= 0 && n_pooled_total >= 0, "negative size");
    QSA_NEED(ld <= (int64_t)1 << 28, "ld too large");
    QSA_TRY(check_ws(QSA_OP_INDEX_SCORE, cfg, Nq, ld, ws, ws_bytes));
    if (Nq == 0 || ld == 0) return ok();
    QSA_NEED(q_idx && q_pos && codes && scales && blk_off && scores, "NULL tensor pointer");
    QSA_NEED(aligned(q_idx, 16) && aligned(codes, 16), "q_idx and codes must be 16-byte aligned");
    QSA_NEED(aligned(scales, 4) && aligned(scores, 4), "scales and scores must be 4-byte aligned");
    const cudaError_t e = launch_index_score_fp8(q_idx, q_seq, q_pos, Nq, codes, scales, n_pooled_total, blk_off,
                                                 scores, ld, static_cast<WsHeader *>(ws),
                                                 static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "index_score_fp8 launch");
    return ok();
}

QSA_API qsa_status qsa_prefill_select(const qsa_config *cfg, const qsa_bf16 *q_idx, const int32_t *q_pos, int32_t Nq,
                                      const qsa_bf16 *pooled, int64_t n_pooled_total, const int32_t *blk_off,
                                      float *scores, int64_t ld, int32_t *blocks, int32_t *count, void *ws,
                                      size_t ws_bytes, qsa_stream stream) {
    QSA_TRY(check_config(cfg));
    QSA_NEED(Nq >= 0 && Nq <= kMaxGridYZ, "Nq = %d out of range [0, 65535]", Nq);
    QSA_NEED(ld >= 0 && n_pooled_total >= 0, "negative size");
    QSA_NEED(ld <= (int64_t)1 << 28, "ld too large");
    QSA_TRY(check_ws(QSA_OP_PREFILL_SELECT, cfg, Nq, ld, ws, ws_bytes));
    if (Nq == 0) return ok();
    if (!prefill_select_supported(Nq, n_pooled_total, ld))
        return fail(QSA_ERR_UNSUPPORTED, "prefill select needs Nq >= 128, n_pooled >= 256 and ld <= 524288");
    QSA_NEED(q_idx && q_pos && pooled && blk_off && scores && blocks && count, "NULL tensor pointer");
    QSA_NEED(aligned(q_idx, 16) && aligned(pooled, 16), "q_idx and pooled must be 16-byte aligned");
    QSA_NEED(aligned(scores, 4), "scores must be 4-byte aligned");
    char *w = static_cast<char *>(ws);
    const cudaError_t e = launch_prefill_select(q_idx, q_pos, Nq, pooled, n_pooled_total, blk_off, scores, ld, blocks,
                                                count, reinterpret_cast<WsHeader *>(w), w + kWsHeaderBytes,
                                                ws_bytes - kWsHeaderBytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "prefill_select launch");
    return ok();
}

QSA_API qsa_status qsa_topk_blocks(const qsa_config *cfg, const float *scores, int64_t ld, const int32_t *q_pos,
                                   int32_t Nq, int32_t *blocks, int32_t *count, void *ws, size_t ws_bytes,
                                   qsa_stream stream) {
    QSA_TRY(check_config(cfg));
    QSA_NEED(Nq >= 0 && Nq <= (1 << 30), "Nq = %d out of range", Nq);
    QSA_NEED(ld >= 0 && ld <= (int64_t)1 << 28, "ld out of range");
    QSA_TRY(check_ws(QSA_OP_TOPK_BLOCKS, cfg, Nq, ld, ws, ws_bytes));
    if (Nq == 0) return ok();
    QSA_NEED(scores && q_pos && blocks && count, "NULL tensor pointer");
    char *w = static_cast<char *>(ws);
    const cudaError_t e = launch_topk_blocks(scores, ld, q_pos, Nq, blocks, count, reinterpret_cast<WsHeader *>(w),
                                             w + kWsHeaderBytes, ws_bytes - kWsHeaderBytes,
                                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "topk_blocks launch");
    return ok();
}

}  // extern "C"

qsa_status qsa::sparse_decode_shape_check(const qsa_config *cfg, int32_t B, int64_t n_tokens_total) {
    QSA_TRY(check_config(cfg));
    QSA_NEED(B >= 0 && B <= kMaxGridYZ, "B = %d out of range [0, 65535]", B);
    QSA_NEED(n_tokens_total >= 0, "negative size");
    return QSA_OK;
}

qsa_status qsa::sparse_decode_pointer_check(const qsa_bf16 *q, const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                            const int32_t *tok_off, const int32_t *ctx_len, const int32_t *blocks,
                                            const int32_t *count, const qsa_bf16 *out) {
    QSA_NEED(q && k_cache && v_cache && tok_off && ctx_len && blocks && count && out, "NULL tensor pointer");
    QSA_NEED(aligned(k_cache, 16) && aligned(v_cache, 16) && aligned(q, 16) && aligned(out, 16),
             "q, k_cache, v_cache and out must be 16-byte aligned");
    QSA_NEED(device_accessible(k_cache) && device_accessible(v_cache),
             "k_cache and v_cache must be device memory or mapped pinned host memory");
    return QSA_OK;
}

extern "C" {

QSA_API qsa_status qsa_sparse_decode(const qsa_config *cfg, const qsa_bf16 *q, const qsa_bf16 *k_cache,
                                     const qsa_bf16 *v_cache, int64_t n_tokens_total, const int32_t *tok_off,
                                     const int32_t *ctx_len, int32_t B, const int32_t *blocks, const int32_t *count,
                                     qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes, qsa_stream stream) {
    QSA_TRY(sparse_decode_shape_check(cfg, B, n_tokens_total));
    QSA_TRY(check_ws(QSA_OP_SPARSE_DECODE, cfg, B, 0, ws, ws_bytes));
    if (B == 0) return ok();
    QSA_TRY(sparse_decode_pointer_check(q, k_cache, v_cache, tok_off, ctx_len, blocks, count, out));
    char *w = static_cast<char *>(ws);
    AttnArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.n_tok = n_tokens_total;
    a.tok_off = tok_off;
    a.ctx_len = ctx_len;
    a.p0 = 0;
    a.rows = B;
    a.blocks = blocks;
    a.count = count;
    a.out = out;
    a.lse = lse;
    a.n_q_heads = cfg->n_q_heads;
    a.n_kv_heads = cfg->n_kv_heads;
    a.scale_log2 = scale_of(cfg) * kLog2e;
    a.where = kWhereDecode;
    const cudaError_t e = launch_sparse_decode(a, reinterpret_cast<WsHeader *>(w), w + kWsHeaderBytes,
                                               ws_bytes - kWsHeaderBytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sparse_decode launch");
    return ok();
}

// The prefill's checks that do not look at the K/V pointers, shared by the staged entry points
// so that nothing is copied or dequantised for a call that would be refused.
static qsa_status check_prefill_args(const qsa_config *cfg, int32_t p0, int32_t Nc, int32_t interval_tokens,
                                     void *ws, size_t ws_bytes) {
    QSA_TRY(check_config(cfg));
    QSA_NEED(p0 >= 0 && Nc >= 0 && Nc <= kMaxGridYZ, "p0 = %d / Nc = %d out of range", p0, Nc);
    QSA_NEED((int64_t)p0 + Nc <= INT32_MAX, "p0 + Nc overflows int32");
    QSA_NEED(interval_tokens > 0 && interval_tokens % 128 == 0,
             "interval_tokens = %d must be a positive multiple of 128", interval_tokens);
    QSA_TRY(check_ws(QSA_OP_SPARSE_PREFILL_CHUNK, cfg, Nc, 0, ws, ws_bytes));
    if (Nc == 0) return ok();
    if (prefill_tc_supported(cfg->n_q_heads, cfg->n_kv_heads) && ((int64_t)p0 + Nc) / kRatio + 1 > kPrefillTcMaxBlocks)
        return fail(QSA_ERR_UNSUPPORTED, "p0 + Nc = %lld exceeds the tensor-core prefill's %lld blocks",
                    (long long)p0 + Nc, (long long)kPrefillTcMaxBlocks);
    return ok();
}

QSA_API qsa_status qsa_sparse_prefill_chunk(const qsa_config *cfg, const qsa_bf16 *q, int32_t p0, int32_t Nc,
                                            const qsa_bf16 *k_cache, const qsa_bf16 *v_cache, const int32_t *blocks,
                                            const int32_t *count, int32_t interval_tokens, qsa_bf16 *out, float *lse,
                                            void *ws, size_t ws_bytes, qsa_stream stream) {
    QSA_TRY(check_prefill_args(cfg, p0, Nc, interval_tokens, ws, ws_bytes));
    if (Nc == 0) return ok();
    QSA_NEED(q && k_cache && v_cache && blocks && count && out, "NULL tensor pointer");
    QSA_NEED(aligned(k_cache, 16) && aligned(v_cache, 16) && aligned(q, 16) && aligned(out, 16) && aligned(blocks, 16),
             "q, k_cache, v_cache, out and blocks must be 16-byte aligned");
    QSA_NEED(device_accessible(k_cache) && device_accessible(v_cache),
             "k_cache and v_cache must be device memory or mapped pinned host memory");
    char *w = static_cast<char *>(ws);
    AttnArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.n_tok = (int64_t)p0 + Nc;
    a.tok_off = nullptr;
    a.ctx_len = nullptr;
    a.p0 = p0;
    a.rows = Nc;
    a.blocks = blocks;
    a.count = count;
    a.out = out;
    a.lse = lse;
    a.n_q_heads = cfg->n_q_heads;
    a.n_kv_heads = cfg->n_kv_heads;
    a.scale_log2 = scale_of(cfg) * kLog2e;
    a.where = kWherePrefill;
    const cudaError_t e = launch_sparse_prefill(a, interval_tokens, reinterpret_cast<WsHeader *>(w),
                                                w + kWsHeaderBytes, ws_bytes - kWsHeaderBytes,
                                                static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sparse_prefill_chunk launch");
    return ok();
}

}  // extern "C"

namespace {

// The fused step with bf16 keys (pooled) or FP8 keys (codes + scales).
// K/V rows of the fused step: bf16 rows, or FP8 codes + scales planes.
struct StepKv {
    const qsa_bf16 *k_cache = nullptr, *v_cache = nullptr;
    const uint8_t *k_codes = nullptr, *v_codes = nullptr;
    const float *k_scales = nullptr, *v_scales = nullptr;
    bool is_fp8 = false;
    bool fp8() const { return is_fp8; }
};

// The VRAM row cache of qsa_decode_step_rowcache (cache == nullptr: none).
struct StepRc {
    void *cache = nullptr;
    size_t bytes = 0;
    int64_t slots = 0;
    uint32_t epoch = 0;
};

qsa_status decode_step_common(const char *name, const qsa_config *cfg, const qsa_bf16 *raw_idx_k, qsa_bf16 *pooled,
                              uint8_t *codes, float *scales, int64_t n_pooled_total, const int32_t *blk_off,
                              const qsa_bf16 *q_idx, const qsa_bf16 *q, const StepKv &kv, int64_t n_tokens_total,
                              const int32_t *tok_off, const int32_t *ctx_len, int32_t B, int64_t max_blocks,
                              int32_t *blocks, int32_t *count, qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                              qsa_stream stream, const void *next_read = nullptr, size_t next_read_bytes = 0,
                              const StepRc &rc = StepRc()) {
    const bool fp8 = pooled == nullptr;
    const bool kv8 = kv.fp8();
    QSA_TRY(check_config(cfg));
    QSA_NEED(B >= 0 && B <= kMaxStepRows, "B = %d out of range [0, 64]", B);
    QSA_NEED(max_blocks >= 0 && max_blocks <= (int64_t)1 << 28, "max_blocks out of range");
    QSA_NEED(n_tokens_total >= 0 && n_pooled_total >= 0, "negative size");
    if (cfg->n_kv_heads > 2) return fail(QSA_ERR_UNSUPPORTED, "%s supports n_kv_heads <= 2", name);
    QSA_TRY(check_ws(QSA_OP_DECODE_STEP, cfg, B, max_blocks, ws, ws_bytes));
    if (B == 0) return ok();
    QSA_NEED(raw_idx_k && (fp8 ? codes && scales : pooled != nullptr) && blk_off && q_idx && q &&
                 (kv8 ? kv.k_codes && kv.k_scales && kv.v_codes && kv.v_scales : kv.k_cache && kv.v_cache) &&
                 tok_off && ctx_len && blocks && count && out,
             "NULL tensor pointer");
    const void *k_rows = kv8 ? static_cast<const void *>(kv.k_codes) : kv.k_cache;
    const void *v_rows = kv8 ? static_cast<const void *>(kv.v_codes) : kv.v_cache;
    QSA_NEED(aligned(raw_idx_k, 16) && aligned(q_idx, 16) && aligned(k_rows, 16) && aligned(v_rows, 16) &&
                 aligned(q, 16) && (fp8 ? aligned(codes, 16) && aligned(scales, 16) : aligned(pooled, 16)) &&
                 (!kv8 || (aligned(kv.k_scales, 16) && aligned(kv.v_scales, 16))),
             "bf16 tensors, codes and scales must be 16-byte aligned");
    if (fp8)
        QSA_NEED(n_pooled_total % 4 == 0, "n_pooled_total = %lld must be a multiple of 4 with FP8 keys",
                 (long long)n_pooled_total);
    QSA_NEED(device_accessible(raw_idx_k) && device_accessible(k_rows) && device_accessible(v_rows) &&
                 (!kv8 || (device_accessible(kv.k_scales) && device_accessible(kv.v_scales))),
             "raw_idx_k and the K/V rows (and their scales) must be device memory or mapped pinned host memory");
    const bool use_rc = rc.cache != nullptr;
    if (use_rc) {
        QSA_NEED(aligned(rc.cache, 16), "the row cache must be 16-byte aligned");
        QSA_NEED(rc.slots >= B && rc.slots <= ((int64_t)1 << 31), "n_slots = %lld must be in [B, 2^31]",
                 (long long)rc.slots);
        QSA_NEED(rc.epoch >= 1, "epoch must be at least 1");
        const RowCacheLayout L = row_cache_layout(cfg->n_kv_heads, rc.slots);
        if (rc.bytes < L.total)
            return fail(QSA_ERR_WORKSPACE_TOO_SMALL, "row cache %zu bytes < %zu needed", rc.bytes, L.total);
        QSA_NEED(device_accessible(rc.cache), "the row cache must be device memory");
    }
    if (next_read != nullptr && next_read_bytes >= 16) {
        QSA_NEED(aligned(next_read, 16), "next_read must be 16-byte aligned");
        QSA_NEED(device_accessible(next_read), "next_read must be device memory or mapped pinned host memory");
    }
    const int G = cfg->n_q_heads / cfg->n_kv_heads;
    const int ctas = decode_step_grid(G, fp8, kv8, use_rc);
    if (ctas == 0) return fail(QSA_ERR_CUDA, "%s: cannot size the cooperative grid on this device", name);
    if (B > ctas) return fail(QSA_ERR_UNSUPPORTED, "%s: B = %d exceeds %d co-resident CTAs", name, B, ctas);
    // every CTA keeps at most decode_step_max_keys() scores on chip; bound the worst row
    const int64_t K = 16384;
    const int64_t worst = ctas > B ? (int64_t)B * (max_blocks + K) / (ctas - B) + 1 : max_blocks;
    if (std::min<int64_t>(worst, max_blocks) > decode_step_max_keys())
        return fail(QSA_ERR_UNSUPPORTED, "%s: %lld blocks per CTA exceed the on-chip limit %d", name,
                    (long long)std::min<int64_t>(worst, max_blocks), decode_step_max_keys());
    StepArgs a{};
    a.raw_idx_k = raw_idx_k;
    a.pooled = pooled;
    a.codes = fp8 ? codes : nullptr;
    a.scales = fp8 ? scales : nullptr;
    a.n_pooled = n_pooled_total;
    a.blk_off = blk_off;
    a.q_idx = q_idx;
    a.q = q;
    a.k_cache = kv8 ? nullptr : kv.k_cache;
    a.v_cache = kv8 ? nullptr : kv.v_cache;
    a.k_codes = kv8 ? kv.k_codes : nullptr;
    a.k_scales = kv8 ? kv.k_scales : nullptr;
    a.v_codes = kv8 ? kv.v_codes : nullptr;
    a.v_scales = kv8 ? kv.v_scales : nullptr;
    a.n_tok = n_tokens_total;
    a.tok_off = tok_off;
    a.ctx_len = ctx_len;
    a.B = B;
    a.max_blocks = max_blocks;
    a.blocks = blocks;
    a.count = count;
    a.out = out;
    a.lse = lse;
    a.n_q_heads = cfg->n_q_heads;
    a.n_kv_heads = cfg->n_kv_heads;
    a.scale_log2 = scale_of(cfg) * kLog2e;
    if (use_rc) {
        const RowCacheLayout L = row_cache_layout(cfg->n_kv_heads, rc.slots);
        char *c = static_cast<char *>(rc.cache);
        a.rc_rows = reinterpret_cast<uint16_t *>(c + L.rows);
        a.rc_tag = reinterpret_cast<int64_t *>(c + L.tag);
        a.rc_hit = reinterpret_cast<uint32_t *>(c + L.hit);
        a.rc_claim = reinterpret_cast<unsigned long long *>(c + L.claim);
        a.rc_slots = rc.slots;
        a.rc_epoch = rc.epoch;
    }
    a.next_read = next_read_bytes >= 16 ? static_cast<const unsigned char *>(next_read) : nullptr;
    a.next_read_bytes = a.next_read ? (int64_t)(next_read_bytes & ~(size_t)15) : 0;
    const cudaError_t e = launch_decode_step(a, ws, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode_step launch");
    return ok();
}

StepKv bf16_kv(const qsa_bf16 *k_cache, const qsa_bf16 *v_cache) {
    StepKv kv;
    kv.k_cache = k_cache;
    kv.v_cache = v_cache;
    return kv;
}

}  // namespace

extern "C" {

QSA_API qsa_status qsa_decode_step(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, qsa_bf16 *pooled,
                                   int64_t n_pooled_total, const int32_t *blk_off, const qsa_bf16 *q_idx,
                                   const qsa_bf16 *q, const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                   int64_t n_tokens_total, const int32_t *tok_off, const int32_t *ctx_len, int32_t B,
                                   int64_t max_blocks, int32_t *blocks, int32_t *count, qsa_bf16 *out, float *lse,
                                   void *ws, size_t ws_bytes, qsa_stream stream) {
    if (pooled == nullptr && B > 0) return fail(QSA_ERR_INVALID_ARGUMENT, "pooled is NULL");
    return decode_step_common("qsa_decode_step", cfg, raw_idx_k, pooled, nullptr, nullptr, n_pooled_total, blk_off,
                              q_idx, q, bf16_kv(k_cache, v_cache), n_tokens_total, tok_off, ctx_len, B, max_blocks, blocks,
                              count, out, lse, ws, ws_bytes, stream);
}

QSA_API qsa_status qsa_decode_step_fp8(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, uint8_t *codes,
                                       float *scales, int64_t n_pooled_total, const int32_t *blk_off,
                                       const qsa_bf16 *q_idx, const qsa_bf16 *q, const qsa_bf16 *k_cache,
                                       const qsa_bf16 *v_cache, int64_t n_tokens_total, const int32_t *tok_off,
                                       const int32_t *ctx_len, int32_t B, int64_t max_blocks, int32_t *blocks,
                                       int32_t *count, qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                                       qsa_stream stream) {
    if ((codes == nullptr || scales == nullptr) && B > 0)
        return fail(QSA_ERR_INVALID_ARGUMENT, "codes and scales must be non-NULL");
    return decode_step_common("qsa_decode_step_fp8", cfg, raw_idx_k, nullptr, codes, scales, n_pooled_total,
                              blk_off, q_idx, q, bf16_kv(k_cache, v_cache), n_tokens_total, tok_off, ctx_len, B, max_blocks,
                              blocks, count, out, lse, ws, ws_bytes, stream);
}

QSA_API qsa_status qsa_decode_step_prefetch(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, qsa_bf16 *pooled,
                                            int64_t n_pooled_total, const int32_t *blk_off, const qsa_bf16 *q_idx,
                                            const qsa_bf16 *q, const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                            int64_t n_tokens_total, const int32_t *tok_off, const int32_t *ctx_len,
                                            int32_t B, int64_t max_blocks, int32_t *blocks, int32_t *count,
                                            qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                                            const void *next_read, size_t next_read_bytes, qsa_stream stream) {
    if (pooled == nullptr && B > 0) return fail(QSA_ERR_INVALID_ARGUMENT, "pooled is NULL");
    return decode_step_common("qsa_decode_step_prefetch", cfg, raw_idx_k, pooled, nullptr, nullptr, n_pooled_total,
                              blk_off, q_idx, q, bf16_kv(k_cache, v_cache), n_tokens_total, tok_off, ctx_len, B, max_blocks,
                              blocks, count, out, lse, ws, ws_bytes, stream, next_read, next_read_bytes);
}

QSA_API qsa_status qsa_decode_step_fp8_prefetch(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, uint8_t *codes,
                                                float *scales, int64_t n_pooled_total, const int32_t *blk_off,
                                                const qsa_bf16 *q_idx, const qsa_bf16 *q, const qsa_bf16 *k_cache,
                                                const qsa_bf16 *v_cache, int64_t n_tokens_total,
                                                const int32_t *tok_off, const int32_t *ctx_len, int32_t B,
                                                int64_t max_blocks, int32_t *blocks, int32_t *count, qsa_bf16 *out,
                                                float *lse, void *ws, size_t ws_bytes, const void *next_read,
                                                size_t next_read_bytes, qsa_stream stream) {
    if ((codes == nullptr || scales == nullptr) && B > 0)
        return fail(QSA_ERR_INVALID_ARGUMENT, "codes and scales must be non-NULL");
    return decode_step_common("qsa_decode_step_fp8_prefetch", cfg, raw_idx_k, nullptr, codes, scales,
                              n_pooled_total, blk_off, q_idx, q, bf16_kv(k_cache, v_cache), n_tokens_total, tok_off, ctx_len,
                              B, max_blocks, blocks, count, out, lse, ws, ws_bytes, stream, next_read,
                              next_read_bytes);
}

QSA_API qsa_status qsa_decode_step_fp8kv(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, qsa_bf16 *pooled,
                                         uint8_t *codes, float *scales, int64_t n_pooled_total,
                                         const int32_t *blk_off, const qsa_bf16 *q_idx, const qsa_bf16 *q,
                                         const uint8_t *k_codes, const float *k_scales, const uint8_t *v_codes,
                                         const float *v_scales, int64_t n_tokens_total, const int32_t *tok_off,
                                         const int32_t *ctx_len, int32_t B, int64_t max_blocks, int32_t *blocks,
                                         int32_t *count, qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                                         qsa_stream stream) {
    if (B > 0 && (pooled == nullptr) == (codes == nullptr || scales == nullptr))
        return fail(QSA_ERR_INVALID_ARGUMENT, "give either pooled or codes and scales");
    StepKv kv;
    kv.is_fp8 = true;
    kv.k_codes = k_codes;
    kv.k_scales = k_scales;
    kv.v_codes = v_codes;
    kv.v_scales = v_scales;
    return decode_step_common("qsa_decode_step_fp8kv", cfg, raw_idx_k, pooled, pooled ? nullptr : codes,
                              pooled ? nullptr : scales, n_pooled_total, blk_off, q_idx, q, kv, n_tokens_total,
                              tok_off, ctx_len, B, max_blocks, blocks, count, out, lse, ws, ws_bytes, stream);
}

QSA_API qsa_status qsa_sparse_prefill_chunk_staged(const qsa_config *cfg, const qsa_bf16 *q, int32_t p0, int32_t Nc,
                                                   const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                                   const int32_t *blocks, const int32_t *count, int32_t interval_tokens,
                                                   qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes, void *stage,
                                                   size_t stage_bytes, qsa_stream stream) {
    QSA_TRY(check_prefill_args(cfg, p0, Nc, interval_tokens, ws, ws_bytes));
    if (Nc == 0) return ok();
    const size_t rows_bytes = ((size_t)p0 + Nc) * cfg->n_kv_heads * cfg->head_dim * 2;
    QSA_NEED(stage != nullptr && aligned(stage, 16), "the stage must be non-NULL and 16-byte aligned");
    if (stage_bytes < 2 * rows_bytes)
        return fail(QSA_ERR_WORKSPACE_TOO_SMALL, "stage %zu bytes < %zu needed", stage_bytes, 2 * rows_bytes);
    QSA_NEED(k_cache && v_cache, "NULL tensor pointer");
    QSA_NEED(device_accessible(stage), "the stage must be device memory");
    // the history and the chunk cross the link once, as two bulk copies, before the chunk runs
    char *sk = static_cast<char *>(stage), *sv = sk + rows_bytes;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(sk, k_cache, rows_bytes, cudaMemcpyDefault, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(sv, v_cache, rows_bytes, cudaMemcpyDefault, st);
    if (e != cudaSuccess) return cuda_fail(e, "prefill staging copy");
    return qsa_sparse_prefill_chunk(cfg, q, p0, Nc, reinterpret_cast<const qsa_bf16 *>(sk),
                                    reinterpret_cast<const qsa_bf16 *>(sv), blocks, count, interval_tokens, out, lse,
                                    ws, ws_bytes, stream);
}

QSA_API size_t qsa_rowcache_bytes(const qsa_config *cfg, int64_t n_slots) {
    if (check_config(cfg) != QSA_OK || cfg->n_kv_heads > 2 || n_slots < 1 || n_slots > ((int64_t)1 << 31)) return 0;
    return row_cache_layout(cfg->n_kv_heads, n_slots).total;
}

QSA_API qsa_status qsa_rowcache_init(const qsa_config *cfg, void *cache, size_t cache_bytes, int64_t n_slots,
                                     qsa_stream stream) {
    const size_t need = qsa_rowcache_bytes(cfg, n_slots);
    QSA_NEED(need > 0, "bad configuration or n_slots = %lld", (long long)n_slots);
    QSA_NEED(cache != nullptr && aligned(cache, 16), "the row cache must be non-NULL and 16-byte aligned");
    if (cache_bytes < need) return fail(QSA_ERR_WORKSPACE_TOO_SMALL, "row cache %zu bytes < %zu needed", cache_bytes, need);
    const RowCacheLayout L = row_cache_layout(cfg->n_kv_heads, n_slots);
    char *c = static_cast<char *>(cache);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(c + L.tag, 0xFF, L.hit - L.tag, st);        // every tag -1: empty
    if (e == cudaSuccess) e = cudaMemsetAsync(c + L.hit, 0, L.total - L.hit, st);  // marks and claims 0
    if (e != cudaSuccess) return cuda_fail(e, "rowcache_init");
    return ok();
}

QSA_API qsa_status qsa_decode_step_rowcache(const qsa_config *cfg, const qsa_bf16 *raw_idx_k, qsa_bf16 *pooled,
                                            int64_t n_pooled_total, const int32_t *blk_off, const qsa_bf16 *q_idx,
                                            const qsa_bf16 *q, const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                            int64_t n_tokens_total, const int32_t *tok_off, const int32_t *ctx_len,
                                            int32_t B, int64_t max_blocks, int32_t *blocks, int32_t *count,
                                            qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes, void *cache,
                                            size_t cache_bytes, int64_t n_slots, uint32_t epoch, qsa_stream stream) {
    if (B > 0 && (pooled == nullptr || cache == nullptr))
        return fail(QSA_ERR_INVALID_ARGUMENT, "pooled and the row cache must be non-NULL");
    StepRc rc;
    rc.cache = cache;
    rc.bytes = cache_bytes;
    rc.slots = n_slots;
    rc.epoch = epoch;
    return decode_step_common("qsa_decode_step_rowcache", cfg, raw_idx_k, pooled, nullptr, nullptr, n_pooled_total,
                              blk_off, q_idx, q, bf16_kv(k_cache, v_cache), n_tokens_total, tok_off, ctx_len, B,
                              max_blocks, blocks, count, out, lse, ws, ws_bytes, stream, nullptr, 0, rc);
}

QSA_API qsa_status qsa_quantize_kv_fp8(const qsa_bf16 *x, int64_t n_rows, uint8_t *codes, float *scales,
                                       qsa_stream stream) {
    QSA_NEED(n_rows >= 0 && n_rows <= ((int64_t)1 << 34), "n_rows = %lld out of range", (long long)n_rows);
    if (n_rows == 0) return ok();
    QSA_NEED(x && codes && scales, "NULL tensor pointer");
    QSA_NEED(aligned(x, 16) && aligned(codes, 16) && aligned(scales, 8), "x and codes must be 16-byte aligned, "
             "scales 8-byte aligned");
    QSA_NEED(device_accessible(x) && device_accessible(codes) && device_accessible(scales),
             "x, codes and scales must be device memory or mapped pinned host memory");
    const cudaError_t e = launch_quantize_kv_fp8(x, n_rows, codes, scales, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "quantize_kv_fp8 launch");
    return ok();
}

QSA_API qsa_status qsa_dequantize_kv_fp8(const uint8_t *codes, const float *scales, int64_t n_rows, qsa_bf16 *x,
                                         qsa_stream stream) {
    QSA_NEED(n_rows >= 0 && n_rows <= ((int64_t)1 << 34), "n_rows = %lld out of range", (long long)n_rows);
    if (n_rows == 0) return ok();
    QSA_NEED(x && codes && scales, "NULL tensor pointer");
    QSA_NEED(aligned(x, 16) && aligned(codes, 16) && aligned(scales, 8), "codes and x must be 16-byte aligned, "
             "scales 8-byte aligned");
    QSA_NEED(device_accessible(x) && device_accessible(codes) && device_accessible(scales),
             "codes, scales and x must be device memory or mapped pinned host memory");
    const cudaError_t e = launch_dequantize_kv_fp8(codes, scales, x, nullptr, nullptr, nullptr, n_rows,
                                                   static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "dequantize_kv_fp8 launch");
    return ok();
}

QSA_API qsa_status qsa_sparse_prefill_chunk_fp8kv(const qsa_config *cfg, const qsa_bf16 *q, int32_t p0, int32_t Nc,
                                                  const uint8_t *k_codes, const float *k_scales,
                                                  const uint8_t *v_codes, const float *v_scales,
                                                  const int32_t *blocks, const int32_t *count, int32_t interval_tokens,
                                                  qsa_bf16 *out, float *lse, void *ws, size_t ws_bytes, void *stage,
                                                  size_t stage_bytes, qsa_stream stream) {
    QSA_TRY(check_prefill_args(cfg, p0, Nc, interval_tokens, ws, ws_bytes));
    if (Nc == 0) return ok();
    const int64_t n_rows = ((int64_t)p0 + Nc) * cfg->n_kv_heads;          // 256-dim rows of K (and of V)
    const size_t rows_bytes = (size_t)n_rows * cfg->head_dim * 2;
    QSA_NEED(stage != nullptr && aligned(stage, 16), "the stage must be non-NULL and 16-byte aligned");
    if (stage_bytes < 2 * rows_bytes)
        return fail(QSA_ERR_WORKSPACE_TOO_SMALL, "stage %zu bytes < %zu needed", stage_bytes, 2 * rows_bytes);
    QSA_NEED(k_codes && k_scales && v_codes && v_scales, "NULL tensor pointer");
    QSA_NEED(aligned(k_codes, 16) && aligned(v_codes, 16) && aligned(k_scales, 8) && aligned(v_scales, 8),
             "codes must be 16-byte aligned, scales 8-byte aligned");
    QSA_NEED(device_accessible(stage), "the stage must be device memory");
    QSA_NEED(device_accessible(k_codes) && device_accessible(k_scales) && device_accessible(v_codes) &&
             device_accessible(v_scales), "codes and scales must be device memory or mapped pinned host memory");
    // the history and the chunk dequantised once into the stage, then the bf16 prefill on it
    uint16_t *sk = static_cast<uint16_t *>(stage), *sv = sk + (size_t)n_rows * cfg->head_dim;
    const cudaError_t e = launch_dequantize_kv_fp8(k_codes, k_scales, sk, v_codes, v_scales, sv, n_rows,
                                                   static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "dequantize_kv_fp8 launch");
    return qsa_sparse_prefill_chunk(cfg, q, p0, Nc, reinterpret_cast<const qsa_bf16 *>(sk),
                                    reinterpret_cast<const qsa_bf16 *>(sv), blocks, count, interval_tokens, out, lse,
                                    ws, ws_bytes, stream);
}

QSA_API size_t qsa_sparse_mla_workspace_size(int32_t n_heads, int32_t B, int32_t max_rows) {
    if (n_heads < 1 || n_heads > 128 || B < 0 || B > kMaxGridYZ || max_rows < 0 || max_rows > 65536) return 0;
    return kWsHeaderBytes + mla_scratch_bytes(n_heads, B, max_rows);
}

QSA_API qsa_status qsa_sparse_mla_decode(const qsa_bf16 *q, int32_t n_heads, const uint8_t *kv_rows,
                                         int64_t n_tokens, const int32_t *rows, const int32_t *n_rows,
                                         int32_t max_rows, int32_t B, float softmax_scale, qsa_bf16 *out, float *lse,
                                         void *ws, size_t ws_bytes, qsa_stream stream) {
    if (n_heads < 1 || n_heads > 128) return fail(QSA_ERR_UNSUPPORTED, "n_heads = %d (1 .. 128)", n_heads);
    QSA_NEED(B >= 0 && B <= kMaxGridYZ, "B = %d out of range [0, 65535]", B);
    QSA_NEED(max_rows >= 0 && max_rows <= 65536, "max_rows = %d out of range [0, 65536]", max_rows);
    QSA_NEED(n_tokens >= 0, "negative size");
    QSA_NEED(!(softmax_scale > 0.f) || isfinite(softmax_scale), "softmax_scale must be finite");
    QSA_NEED(ws != nullptr && aligned(ws, 256), "workspace must be non-NULL and 256-byte aligned");
    const size_t need = qsa_sparse_mla_workspace_size(n_heads, B, max_rows);
    if (ws_bytes < need) return fail(QSA_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", ws_bytes, need);
    if (B == 0) return ok();
    QSA_NEED(q && kv_rows && rows && n_rows && out, "NULL tensor pointer");
    QSA_NEED(aligned(q, 16) && aligned(kv_rows, 16), "q and kv_rows must be 16-byte aligned");
    QSA_NEED(aligned(out, 2) && aligned(rows, 4) && aligned(n_rows, 4) && aligned(lse, 4), "misaligned output");
    const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(576.0f);
    char *w = static_cast<char *>(ws);
    const cudaError_t e = launch_sparse_mla(q, n_heads, kv_rows, n_tokens, rows, n_rows, max_rows, B, scale, out, lse,
                                            reinterpret_cast<WsHeader *>(w), w + kWsHeaderBytes,
                                            static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sparse_mla_decode launch");
    return ok();
}

QSA_API const char *qsa_status_string(qsa_status s) {
    switch (s) {
        case QSA_OK: return "ok";
        case QSA_ERR_INVALID_ARGUMENT: return "invalid argument";
        case QSA_ERR_UNSUPPORTED: return "unsupported geometry";
        case QSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case QSA_ERR_CUDA: return "CUDA error";
        case QSA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case QSA_ERR_DEVICE_BOUNDS: return "device-side bounds check failed";
        default: return "unknown status";
    }
}

QSA_API const char *qsa_last_error(void) { return g_last_error; }

QSA_API const char *qsa_version(void) { return "qsa-gb300 0.1.0 sm_103a"; }

}  // extern "C"
