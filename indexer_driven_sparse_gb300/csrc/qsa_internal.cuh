// Internal declarations shared by the CUDA translation units of libqsa.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "qsa.h"

namespace qsa {

constexpr int kHeadDim = 256;
constexpr int kIdxDim = 128;
constexpr int kRatio = 4;
constexpr int kBlockTopK = 512;              // indexer_budget / ratio
constexpr int kMaxGroup = 16;                // max query heads per KV head
constexpr int kMaxAttended = kRatio * kBlockTopK + kRatio;   // 2052 = 2048 selected + own block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// First 256 bytes of every workspace.
struct WsHeader {
    int32_t status;      // first device-side error (qsa_status), 0 = none
    int32_t detail;      // kernel-specific detail (row, index)
    int32_t where;       // which kernel recorded it
    int32_t debug;       // test knob: kDebugStallBarrier makes the first row barrier never complete
    uint32_t sem[60];    // self-resetting counters (last-CTA-done, grid barriers)
};
static_assert(sizeof(WsHeader) == 256, "status block must be 256 bytes");
constexpr size_t kWsHeaderBytes = 256;
constexpr int32_t kDebugStallBarrier = 0x5741171;   // written only by the device-timeout test
constexpr int32_t kDebugTrace = 0x7ACE;             // record per-CTA phase timestamps (qsa_decode_step)
constexpr int kTraceSlots = 16;
constexpr uint64_t kWaitLimitNs = 250ull * 1000 * 1000;   // every device-side wait gives up after 250 ms

enum Where : int32_t {
    kWherePool = 1, kWhereScore = 2, kWhereTopk = 3, kWhereDecode = 4, kWhereMerge = 5, kWherePrefill = 6,
    kWhereStep = 7,
};

__device__ __forceinline__ void record_error(WsHeader *h, int32_t code, int32_t where, int32_t detail) {
    if (h == nullptr) return;
    if (atomicCAS(&h->status, 0, code) == 0) {
        h->detail = detail;
        h->where = where;
    }
}

// bf16 bits -> float (exact).
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Unpack 8 bf16 values from a 16-byte vector.
__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
    f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xFFFF0000u);
    f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xFFFF0000u);
    f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xFFFF0000u);
    f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

// Read-only 16-byte global load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// fp32 -> bf16 bits, round to nearest even (CUDA intrinsic).
__device__ __forceinline__ uint16_t float_to_bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Round a double to the nearest bf16 (ties to even) in one step. bf16 keeps 8
// significant bits with fp32's exponent range: near |x| in [2^e, 2^(e+1)) the spacing is
// 2^(e-7), and 2^-133 below 2^-126.
// Normal range: round the 52-bit fp64 fraction at bit 45 with integer arithmetic (add
// half an ulp minus one plus the kept lsb, clear the dropped bits); the result has 8
// significant bits and converts to fp32 exactly. Elsewhere (zero, subnormal bf16, inf,
// NaN): scale by a power of two (exact), rint() (half to even), scale back.
__device__ __forceinline__ uint16_t double_to_bf16_rne(double x) {
    const unsigned long long b = (unsigned long long)__double_as_longlong(x);
    const unsigned e = (unsigned)(b >> 52) & 0x7FFu;
    const uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
    if (e >= 1023u - 126u && e < 1023u + 128u) {
        const unsigned long long lsb = (b >> 45) & 1ull;
        unsigned long long r = b + 0x00000FFFFFFFFFFFull + lsb;
        r &= ~0x00001FFFFFFFFFFFull;
        if ((((unsigned)(r >> 52)) & 0x7FFu) >= 1023u + 128u) return sign | 0x7F80;
        return (uint16_t)(__float_as_uint((float)__longlong_as_double((long long)r)) >> 16);
    }
    if (isnan(x)) return 0x7FC0;
    const double ax = fabs(x);
    if (isinf(ax)) return sign | 0x7F80;
    if (ax >= 0x1p127) return sign | 0x7F80;    // |x| >= 2^128: overflow
    const double r = ldexp(rint(ldexp(ax, 133)), -133);
    return sign | (uint16_t)(__float_as_uint((float)r) >> 16);
}

// ---------------------------------------------------------------------------- FP8 (E4M3) keys
constexpr float kE4m3Max = 448.f;   // largest finite E4M3 value: 1.75 * 2^8

// Two fp32 values -> two E4M3 codes (nearest even, saturating at +-448); `lo` lands in
// bits 0-7, `hi` in bits 8-15 (the instruction puts its first source in the upper byte).
__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Sixteen E4M3 codes (byte k = dim k) -> fp32, exactly: E4M3 -> f16 is exact, f16 -> f32 too.
__device__ __forceinline__ void e4m3x16_to_f32(const uint4 &v, float (&f)[16]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h0, h1;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h0) : "h"((uint16_t)(w[i] & 0xFFFFu)));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h1) : "h"((uint16_t)(w[i] >> 16)));
        f[4 * i + 0] = __half2float(__ushort_as_half((unsigned short)(h0 & 0xFFFFu)));
        f[4 * i + 1] = __half2float(__ushort_as_half((unsigned short)(h0 >> 16)));
        f[4 * i + 2] = __half2float(__ushort_as_half((unsigned short)(h1 & 0xFFFFu)));
        f[4 * i + 3] = __half2float(__ushort_as_half((unsigned short)(h1 >> 16)));
    }
}

// The indexer score's evaluation order, shared by every bf16 scan (index_score_kernel and
// the fused step) so that their scores agree bit for bit: lane l of a warp holds dims
// 4l .. 4l+3 of the 128-dim row and of the query; its partial is x0 q0 + x1 q1 + x2 q2 + x3 q3
// as one product and three fused multiply-adds (bf16 x bf16 products are exact in fp32);
// the row's score is the butterfly sum of the 32 partials over lane distances 16, 8, 4, 2, 1.
__device__ __forceinline__ float dot4_bf16(uint2 x, const float (&q)[4]) {
    float t = __uint_as_float(x.x << 16) * q[0];
    t = fmaf(__uint_as_float(x.x & 0xFFFF0000u), q[1], t);
    t = fmaf(__uint_as_float(x.y << 16), q[2], t);
    return fmaf(__uint_as_float(x.y & 0xFFFF0000u), q[3], t);
}

__device__ __forceinline__ void load_q4(const uint16_t *q_row, int lane, float (&q)[4]) {
    const uint2 v = *reinterpret_cast<const uint2 *>(q_row + 4 * lane);
    q[0] = __uint_as_float(v.x << 16);
    q[1] = __uint_as_float(v.x & 0xFFFF0000u);
    q[2] = __uint_as_float(v.y << 16);
    q[3] = __uint_as_float(v.y & 0xFFFF0000u);
}

// Reduce-scatter of NV rows' partials (NV a power of two <= 32) over the warp in the
// butterfly order above: afterwards every lane holds the full score of row
// row_of_lane<NV>(lane) (the rows' sums are identical to a per-row butterfly).
template <int NV>
__device__ __forceinline__ float reduce_rows(float (&v)[NV], int lane) {
#pragma unroll
    for (int level = 0; (NV >> level) > 1; ++level) {
        const int n = NV >> level, o = 16 >> level;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float r = v[0];
#pragma unroll
    for (int o = 16 / NV; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

// Row index whose total lane `lane` holds after reduce_rows<NV>: the top log2(NV) lane bits.
constexpr int ilog2(int n) { return n <= 1 ? 0 : 1 + ilog2(n >> 1); }

template <int NV>
__device__ __forceinline__ int row_of_lane(int lane) {
    return (lane >> (5 - ilog2(NV))) & (NV - 1);
}

// Order-preserving map of an fp32 score to uint32: larger score -> larger key.
// -0 is folded onto +0 and NaN onto the smallest key.
__device__ __forceinline__ uint32_t score_key(float s) {
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u) u = 0u;
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------- launchers
// Each returns cudaGetLastError() of its launches.
cudaError_t launch_pool_keys(const uint16_t *raw, int64_t n_tok, const int32_t *tok_off, const int32_t *blk_off,
                             const int32_t *blk_begin, const int32_t *blk_end, int B, int64_t max_blocks,
                             uint16_t *pooled, int64_t n_pooled, WsHeader *hdr, cudaStream_t st);

cudaError_t launch_index_score(const uint16_t *q_idx, const int32_t *q_seq, const int32_t *q_pos, int Nq,
                               const uint16_t *pooled, int64_t n_pooled, const int32_t *blk_off, float *scores,
                               int64_t ld, WsHeader *hdr, cudaStream_t st);

// FP8 (E4M3) indexer keys with a per-block fp32 scale (fp8_keys.cu).
cudaError_t launch_pool_keys_fp8(const uint16_t *raw, int64_t n_tok, const int32_t *tok_off, const int32_t *blk_off,
                                 const int32_t *blk_begin, const int32_t *blk_end, int B, int64_t max_blocks,
                                 uint8_t *codes, float *scales, int64_t n_pooled, WsHeader *hdr, cudaStream_t st);
cudaError_t launch_index_score_fp8(const uint16_t *q_idx, const int32_t *q_seq, const int32_t *q_pos, int Nq,
                                   const uint8_t *codes, const float *scales, int64_t n_pooled,
                                   const int32_t *blk_off, float *scores, int64_t ld, WsHeader *hdr,
                                   cudaStream_t st);

size_t topk_scratch_bytes(int Nq, int64_t ld);
// Tensor-core scoring of many queries of one sequence (score_tc.cu).
bool score_tc_supported(int Nq, int64_t n_pooled);
cudaError_t launch_score_tc(const uint16_t *q_idx, const int32_t *q_pos, int Nq, const uint16_t *pooled,
                            int64_t n_pooled, const int32_t *blk_off, float *scores, int64_t ld, WsHeader *hdr,
                            cudaStream_t st);
cudaError_t launch_topk_blocks(const float *scores, int64_t ld, const int32_t *q_pos, int Nq, int32_t *blocks,
                               int32_t *count, WsHeader *hdr, void *scratch, size_t scratch_bytes, cudaStream_t st);

// ---------------------------------------------------------------------------- fused prefill selection
// Scoring and top-k of a prefill chunk without materialising the score matrix:
//   1. the scoring GEMM keeps, per row, the max of every 64 consecutive visible blocks;
//   2. each row's floor T = the 512th largest of those maxima (at least 512 scores reach it);
//   3. the GEMM runs again and its epilogue keeps every visible score >= T as a 64-bit key in
//      per-(row, 256-block tile) slots;
//   4. the top-k kernel takes each row's exact top 512 from its candidates;
//   5. rows whose candidates overflowed a tile's slots (or fell short) are left to the exact
//      path: the GEMM stores the full scores and the top-k kernel streams those rows only
//      (both launches return at once when no row needs them).
constexpr int kSelGroup = 64;                 // blocks per maximum
constexpr int kSelSlots = 16;                 // candidate slots per (row, half a tile: 128 blocks)
constexpr int kSelSegsPerThread = 8;          // top-k: half-tile segments of a row per thread
constexpr int kSelMaxTiles = 512 * kSelSegsPerThread / 2;   // 2048 tiles of 256 blocks

struct TopkCandidates {
    const uint64_t *slots = nullptr;   // [Nq][n_segs][kSelSlots] candidate keys (nullptr: stream the scores)
    const uint8_t *scnt = nullptr;     // [Nq][n_segs] candidates per segment (> kSelSlots: overflowed)
    int32_t n_segs = 0;                // segments of a row: two per tile of 256 blocks
    int32_t *fb_rows = nullptr;        // [Nq] rows left to the exact path
    int32_t *fb_any = nullptr;         // set when some row is
    int32_t fallback_only = 0;         // run only the rows of fb_rows (on the stored scores)
};

cudaError_t launch_topk_with(const float *scores, int64_t ld, const int32_t *q_pos, int Nq, int32_t *blocks,
                             int32_t *count, WsHeader *hdr, const TopkCandidates &tc, cudaStream_t st);
size_t prefill_select_scratch_bytes(int Nq, int64_t ld);
bool prefill_select_supported(int Nq, int64_t n_pooled, int64_t ld);
cudaError_t launch_prefill_select(const uint16_t *q_idx, const int32_t *q_pos, int Nq, const uint16_t *pooled,
                                  int64_t n_pooled, const int32_t *blk_off, float *scores, int64_t ld, int32_t *blocks,
                                  int32_t *count, WsHeader *hdr, void *scratch, size_t scratch_bytes, cudaStream_t st);

struct AttnArgs {
    const uint16_t *q;        // [rows, Hq, D]
    const uint16_t *k_cache;  // [T, Hkv, D]
    const uint16_t *v_cache;
    int64_t n_tok;
    const int32_t *tok_off;   // decode: [B+1]; prefill: nullptr (one sequence from token 0)
    const int32_t *ctx_len;   // decode: [B]; prefill: nullptr (p = p0 + row)
    int32_t p0;
    int32_t rows;
    const int32_t *blocks;    // [rows, kBlockTopK]
    const int32_t *count;     // [rows]
    uint16_t *out;            // [rows, Hq, D]
    float *lse;               // [rows, Hq] or nullptr
    int32_t n_q_heads, n_kv_heads;
    float scale_log2;         // softmax scale * log2(e)
    int32_t where;
};
size_t decode_scratch_bytes(int B, int Hq, int Hkv);
cudaError_t launch_sparse_decode(const AttnArgs &a, WsHeader *hdr, void *scratch, size_t scratch_bytes,
                                 cudaStream_t st);

// One CTA per (row, KV head) over the row's whole token set (no split partials).
cudaError_t launch_attn_rows(const AttnArgs &a, WsHeader *hdr, cudaStream_t st);

size_t prefill_scratch_bytes(int Nc, int Hq, int Hkv);
bool prefill_tc_supported(int Hq, int Hkv);
constexpr int64_t kPrefillTcMaxBlocks = 2048 * 256;   // pooled blocks the tile tables cover
size_t prefill_tc_plan_bytes(int Nc, int Hq, int Hkv);
cudaError_t launch_prefill_tc(const AttnArgs &a, int interval_tokens, WsHeader *hdr, void *scratch,
                              size_t scratch_bytes, cudaStream_t st);

// Fused decode layer-step (decode_step.cu).
constexpr int kMaxStepCtas = 256;
constexpr int kMaxStepRows = 64;
struct StepArgs {
    const uint16_t *raw_idx_k;
    uint16_t *pooled;           // bf16 keys [n_pooled][128] (nullptr with FP8 keys)
    uint8_t *codes;             // FP8 keys: codes [n_pooled][128] and scales [n_pooled] (else nullptr)
    float *scales;
    int64_t n_pooled;
    const int32_t *blk_off;
    const uint16_t *q_idx;
    const uint16_t *q;
    const uint16_t *k_cache;    // bf16 K/V rows [n_tok][Hkv][256] (nullptr with FP8 K/V)
    const uint16_t *v_cache;
    const uint8_t *k_codes;     // FP8 K/V: codes [n_tok][Hkv][256], scales [n_tok][Hkv][2] (else nullptr)
    const float *k_scales;
    const uint8_t *v_codes;
    const float *v_scales;
    int64_t n_tok;
    const int32_t *tok_off;
    const int32_t *ctx_len;
    int32_t B;
    int64_t max_blocks;
    int32_t *blocks;
    int32_t *count;
    uint16_t *out;
    float *lse;
    int32_t n_q_heads, n_kv_heads;
    float scale_log2;
    const unsigned char *next_read;   // optional L2 prefetch hint (16-byte aligned) or nullptr
    int64_t next_read_bytes;
    // VRAM row cache (nullptr: none): rows [rc_slots][2][Hkv][256] bf16, tags, hit marks, claims
    uint16_t *rc_rows;
    int64_t *rc_tag;
    uint32_t *rc_hit;
    unsigned long long *rc_claim;
    int64_t rc_slots;
    uint32_t rc_epoch;
    // workspace views (set by launch_decode_step)
    WsHeader *hdr;
    void *rows;
    uint32_t *hist;
    unsigned long long *cands;
    float *part;
    unsigned long long *pub;     // [kMaxStepCtas][513] published local top-K keys + flag
    unsigned long long *trace;   // [kMaxStepCtas][kTraceSlots] globaltimer stamps
};
struct StepLayout {
    size_t rows, hist, cands, part, pub, trace, total;
};
StepLayout step_layout(int B, int64_t max_blocks, int Hq);
size_t decode_step_ws_bytes(int B, int64_t max_blocks, int Hq);
int decode_step_max_keys();
// Number of CTAs the cooperative step kernel runs with on the current device (0 on error),
// for FP8 or bf16 indexer keys, FP8 or bf16 K/V rows, with or without the row cache.
int decode_step_grid(int G, bool fp8_keys, bool fp8_kv, bool row_cache = false);
// Bytes of a row cache of n_slots token rows for n_kv_heads, and its parts' offsets.
struct RowCacheLayout {
    size_t rows, tag, hit, claim, total;
};
RowCacheLayout row_cache_layout(int n_kv_heads, int64_t n_slots);
cudaError_t launch_decode_step(StepArgs a, void *ws, cudaStream_t st);

// FP8 K/V rows: x [n_rows][256] bf16 -> codes [n_rows][256] E4M3, scales [n_rows][2] fp32.
cudaError_t launch_quantize_kv_fp8(const uint16_t *x, int64_t n_rows, uint8_t *codes, float *scales,
                                   cudaStream_t st);

// Set the calling thread's qsa_last_error() text to "<what>: <detail>" and return s.
qsa_status host_fail(qsa_status s, const char *what, const char *detail);
// The host checks of qsa_sparse_decode, in its order: the configuration, B and the token
// count first; the tensor pointers (non-NULL, 16-byte alignment, readable by the device) once
// the workspace has been checked and B > 0. Each records its message as qsa_last_error.
qsa_status sparse_decode_shape_check(const qsa_config *cfg, int32_t B, int64_t n_tokens_total);
qsa_status sparse_decode_pointer_check(const qsa_bf16 *q, const qsa_bf16 *k_cache, const qsa_bf16 *v_cache,
                                       const int32_t *tok_off, const int32_t *ctx_len, const int32_t *blocks,
                                       const int32_t *count, const qsa_bf16 *out);
cudaError_t launch_sparse_prefill(const AttnArgs &a, int interval_tokens, WsHeader *hdr, void *scratch,
                                  size_t scratch_bytes, cudaStream_t st);

}  // namespace qsa
