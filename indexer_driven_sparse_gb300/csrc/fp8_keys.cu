// FP8 indexer keys: each pooled block stored as 128 E4M3 codes plus one fp32 scale
// ("GLM-5.3 最適化 第2部：16基のH200上でのPCP、DCP、およびHybrid HiSparse", footnote on the
// indexer cache: 128 FP8 values and a 4-byte scale per key). The pooled-key scan of
// "3090x3で 314 万コンテキスト" (section "VRAM に残す必要があるもの") then reads 132 bytes per
// block instead of 256.
//
//   pool_keys_fp8_kernel:  pooled bf16 key (exact mean, one RNE, as pool_keys_kernel), then
//                          scale = max|key| / 448 and code = E4M3(key / scale), both fp32
//                          IEEE divisions, the code rounded to nearest even and saturated;
//                          an all-zero key has scale 0 and zero codes.
//   index_score_fp8_kernel: s_b = scale_b * sum_d q_idx[d] * code_b[d]; every product of a
//                          bf16 and an E4M3 value is exact in fp32, summed in fp32.
//   quantize_kv_fp8_kernel: FP8 K/V rows for the fused decode step ("GLM-5.3 最適化 第2部",
//                          footnote 1: KV rows as E4M3 codes in 128-dim groups with an fp32
//                          scale each): every 128-dim group of a 256-dim K or V row is
//                          quantised exactly as a pooled key above.
//   dequantize_kv_fp8_kernel: the inverse for the tensor-core prefill, which multiplies bf16
//                          tiles: element d of a row becomes code_d x scale[d / 128] rounded
//                          once to bf16 (nearest, ties to even).
#include "qsa_internal.cuh"
#include "kv_fp8.cuh"
#include "qsa_ptx.cuh"

#include <algorithm>

namespace qsa {

// 16 threads per pooled block, each owning 8 of the 128 dims; the block's |max| is reduced
// over its 16 threads (one half-warp).
__global__ void __launch_bounds__(256) pool_keys_fp8_kernel(const uint16_t *__restrict__ raw, int64_t n_tok,
                                                            const int32_t *tok_off, const int32_t *blk_off,
                                                            const int32_t *blk_begin, const int32_t *blk_end,
                                                            int64_t max_blocks, uint8_t *__restrict__ codes,
                                                            float *__restrict__ scales, int64_t n_pooled,
                                                            WsHeader *hdr) {
    const int s = blockIdx.y;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t b_rel = t >> 4;
    const int c = (int)(t & 15);
    const int64_t t0 = tok_off[s], t1 = tok_off[s + 1];
    const int64_t bb = blk_begin[s], be = blk_end[s], bo = blk_off[s];
    const bool ok = t0 >= 0 && t0 <= t1 && t1 <= n_tok && bb >= 0 && be >= bb && be - bb <= max_blocks &&
                    kRatio * be <= t1 - t0 && bo >= 0 && bo + be <= n_pooled;
    if (!ok) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(hdr, QSA_ERR_DEVICE_BOUNDS, kWherePool, s);
        return;
    }
    const int64_t b = bb + b_rel;
    if (b >= be) return;   // the 16 threads of one pooled block leave together
    const uint16_t *src = raw + (t0 + kRatio * b) * kIdxDim + c * 8;
    float f0[8], f1[8], f2[8], f3[8];
    unpack8(ldg_nc_v4(src), f0);
    unpack8(ldg_nc_v4(src + kIdxDim), f1);
    unpack8(ldg_nc_v4(src + 2 * kIdxDim), f2);
    unpack8(ldg_nc_v4(src + 3 * kIdxDim), f3);
    float x[8];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const double sum = (((double)f0[i] + (double)f1[i]) + (double)f2[i]) + (double)f3[i];
        x[i] = bf16_bits_to_float(double_to_bf16_rne(sum * 0.25));   // the pooled bf16 key, exact in fp32
        amax = fmaxf(amax, fabsf(x[i]));
    }
    const unsigned grp = 0xFFFFu << (threadIdx.x & 16);
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(grp, amax, o, 16));
    const float scale = __fdiv_rn(amax, kE4m3Max);
    uint32_t w0 = 0u, w1 = 0u;
    if (scale > 0.f) {
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = __fdiv_rn(x[i], scale);
        w0 = e4m3x2_of(y[0], y[1]) | (e4m3x2_of(y[2], y[3]) << 16);
        w1 = e4m3x2_of(y[4], y[5]) | (e4m3x2_of(y[6], y[7]) << 16);
    }
    *reinterpret_cast<uint2 *>(codes + (bo + b) * kIdxDim + c * 8) = make_uint2(w0, w1);
    if (c == 0) scales[bo + b] = scale;
}

constexpr int kF8Threads = 256;
constexpr int kF8TileRows = 128;                                     // 16 KiB of codes per stage
constexpr int kF8Stages = 4;
constexpr int kF8TileBytes = kF8TileRows * kIdxDim;
constexpr int kF8Smem = kF8Stages * kF8TileBytes + 8 * kF8Stages;   // ring + full mbarriers

// The CTAs of a query row (gridDim.x of them) split its visible blocks into equal contiguous
// ranges. A CTA streams its range through a 4-stage shared-memory ring of 128-row tiles
// filled by bulk async copies (TMA engine), so every stage's bytes are requested without
// holding registers; a tile is scored from shared memory (8 lanes per row, 16 dims per lane)
// while later tiles are in flight. Each lane loads its rows' scales one tile ahead.
__global__ void __launch_bounds__(kF8Threads) index_score_fp8_kernel(const uint16_t *__restrict__ q_idx,
                                                                     const int32_t *q_seq, const int32_t *q_pos,
                                                                     const uint8_t *__restrict__ codes,
                                                                     const float *__restrict__ scales,
                                                                     int64_t n_pooled, const int32_t *blk_off,
                                                                     float *__restrict__ scores, int64_t ld,
                                                                     WsHeader *hdr) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int r = blockIdx.y;
    const int p = q_pos[r];
    const int64_t nb = p >= 0 ? (p >> 2) : -1;
    const int64_t off = blk_off[q_seq != nullptr ? q_seq[r] : 0];   // NULL: one sequence
    if (nb < 0 || nb > ld || off < 0 || off + nb > n_pooled) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(hdr, QSA_ERR_DEVICE_BOUNDS, kWhereScore, r);
        return;
    }
    const int64_t lo = nb * blockIdx.x / gridDim.x, hi = nb * (blockIdx.x + 1) / gridDim.x;
    if (lo >= hi) return;   // the whole CTA leaves
    const int n_tiles = (int)((hi - lo + kF8TileRows - 1) / kF8TileRows);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 3, c = lane & 7;
    const uint32_t ring = smem_u32(smem), bar = smem_u32(smem + kF8Stages * kF8TileBytes);
    const uint8_t *src = codes + (off + lo) * kIdxDim;
    auto issue = [&](int t) {                      // thread 0: tile t into stage t % kF8Stages
        const int st = t % kF8Stages;
        const int64_t left = hi - lo - (int64_t)t * kF8TileRows;
        const uint32_t bytes = (uint32_t)(left < kF8TileRows ? left : (int64_t)kF8TileRows) * kIdxDim;
        mbar_arrive_expect_tx(bar + 8 * st, bytes);
        bulk_g2s(ring + st * kF8TileBytes, src + (int64_t)t * kF8TileBytes, bytes, bar + 8 * st);
    };
    if (tid == 0) {
        for (int i = 0; i < kF8Stages; ++i) mbar_init(bar + 8 * i, 1);
        fence_mbar_init();
        for (int t = 0; t < n_tiles && t < kF8Stages; ++t) issue(t);
    }
    float qf[16];
    {
        float a[8], b[8];
        unpack8(ldg_nc_v4(q_idx + (int64_t)r * kIdxDim + c * 16), a);
        unpack8(ldg_nc_v4(q_idx + (int64_t)r * kIdxDim + c * 16 + 8), b);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            qf[e] = a[e];
            qf[8 + e] = b[e];
        }
    }
    // warp w scores rows 16w .. 16w+15 of a tile; lane L < 16 holds the scale of row 16w + L
    auto scale_at = [&](int t) {
        const int64_t row = lo + (int64_t)t * kF8TileRows + warp * 16 + (lane & 15);
        return row < hi ? __ldg(scales + off + row) : 0.f;
    };
    float sc_next = scale_at(0);
    __syncthreads();                               // mbarriers initialised
    for (int t = 0; t < n_tiles; ++t) {
        const int st = t % kF8Stages;
        const float sc = sc_next;
        if (t + 1 < n_tiles) sc_next = scale_at(t + 1);
        const bool late = !mbar_wait_bounded(bar + 8 * st, (t / kF8Stages) & 1, kWaitLimitNs);
        if (__syncthreads_or(late)) {              // every thread leaves together
            if (tid == 0) {
                record_error(hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereScore, r);
                for (int t2 = t; t2 < n_tiles && t2 < t + kF8Stages; ++t2)   // copies still in flight
                    mbar_wait_bounded(bar + 8 * (t2 % kF8Stages), (t2 / kF8Stages) & 1, kWaitLimitNs);
            }
            return;
        }
        const int64_t row0 = lo + (int64_t)t * kF8TileRows;
        const int rows = (int)(hi - row0 < kF8TileRows ? hi - row0 : (int64_t)kF8TileRows);
        const uint8_t *buf = smem + st * kF8TileBytes;
        float part[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int rr = warp * 16 + 4 * j + g;
            float s = 0.f;
            if (rr < rows) {
                float f[16];
                e4m3x16_to_f32(*reinterpret_cast<const uint4 *>(buf + rr * kIdxDim + c * 16), f);
#pragma unroll
                for (int e = 0; e < 16; ++e) s = fmaf(f[e], qf[e], s);
            }
#pragma unroll
            for (int o = 4; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            part[j] = s;
        }
        // row 16w + 4j + g sits in every lane of group g: lane L < 16 takes row 16w + L
        float mine = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float v = __shfl_sync(0xffffffffu, part[j], (lane & 3) * 8);
            if (j == ((lane & 15) >> 2)) mine = v;
        }
        const int my = warp * 16 + lane;
        if (lane < 16 && my < rows) scores[(int64_t)r * ld + row0 + my] = mine * sc;
        __syncthreads();                           // the stage has been read
        if (tid == 0 && t + kF8Stages < n_tiles) {
            fence_proxy_async_smem();
            issue(t + kF8Stages);
        }
    }
}

// 16 threads per 128-dim group (8 dims each; a warp is one 256-dim row), grid-stride.
__global__ void __launch_bounds__(256) quantize_kv_fp8_kernel(const uint16_t *__restrict__ x, int64_t n_groups,
                                                              uint8_t *__restrict__ codes,
                                                              float *__restrict__ scales) {
    const int c = threadIdx.x & 15;
    const unsigned grp = 0xFFFFu << (threadIdx.x & 16);
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 4);
    for (int64_t g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 4; g < n_groups; g += stride) {
        float v[8];
        unpack8(ldg_nc_v4(x + g * 128 + c * 8), v);
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(grp, amax, o, 16));
        const float scale = __fdiv_rn(amax, kE4m3Max);
        uint32_t w0 = 0u, w1 = 0u;
        if (scale > 0.f) {
            float y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = __fdiv_rn(v[i], scale);
            w0 = e4m3x2_of(y[0], y[1]) | (e4m3x2_of(y[2], y[3]) << 16);
            w1 = e4m3x2_of(y[4], y[5]) | (e4m3x2_of(y[6], y[7]) << 16);
        }
        *reinterpret_cast<uint2 *>(codes + g * 128 + c * 8) = make_uint2(w0, w1);
        if (c == 0) scales[g] = scale;
    }
}

cudaError_t launch_quantize_kv_fp8(const uint16_t *x, int64_t n_rows, uint8_t *codes, float *scales,
                                   cudaStream_t st) {
    const int64_t n_groups = 2 * n_rows;                      // two 128-dim groups per 256-dim row
    const int64_t blocks = std::min<int64_t>((n_groups * 16 + 255) / 256, (int64_t)1 << 20);
    quantize_kv_fp8_kernel<<<(unsigned)blocks, 256, 0, st>>>(x, n_groups, codes, scales);
    return cudaGetLastError();
}

// bf16 bits of a x s rounded once (nearest, ties to even), for an E4M3 value a and an fp32 s.
// The fp32 product is rounded, but every point where bf16 rounding changes direction (a
// midpoint between two bf16 values) is itself an fp32 value, and rounding to fp32 is monotone:
// the fp32 product and the exact one lie on the same side of every midpoint unless the fp32
// product is a midpoint. So the fp32 product rounds to the right bf16 except when it is a
// midpoint, zero, below the normal range (where a flush to zero may have lost it), infinite
// or NaN; those take the exact product in fp64 (a 4-bit by 24-bit product fits its 53 bits).
// Not inlined: the caller branches to it only for those rare elements, where an inlined copy
// was if-converted and ran its fp64 arithmetic for every element.
__device__ __noinline__ uint32_t bf16_of_product(float a, float s) {
    const float p = a * s;
    const uint32_t u = __float_as_uint(p), mag = u & 0x7FFFFFFFu;
    if ((u & 0xFFFFu) != 0x8000u && mag >= 0x00800000u && mag < 0x7F800000u) return float_to_bf16_bits(p);
    return double_to_bf16_rne((double)a * (double)s);
}

// True when a byte of w is an E4M3 NaN code (0x7F or 0xFF).
__device__ __forceinline__ bool has_e4m3_nan(uint32_t w) {
    const uint32_t v = (w & 0x7F7F7F7Fu) ^ 0x7F7F7F7Fu;   // a zero byte where the code is NaN
    return ((v - 0x01010101u) & ~v & 0x80808080u) != 0u;
}

// Eight E4M3 codes (byte k = element k) -> fp32, exactly (E4M3 -> f16 -> f32).
__device__ __forceinline__ void e4m3x8_to_f32(uint2 c, float (&a)[8]) {
    const uint32_t w[2] = {c.x, c.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            uint32_t h;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)(w[i] >> (16 * j))));
            const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&h));
            a[4 * i + 2 * j] = x.x;
            a[4 * i + 2 * j + 1] = x.y;
        }
    }
}

// Eight codes by the exact route of bf16_of_product (see dequant8 for when). Not inlined, for
// the same reason as bf16_of_product.
__device__ __noinline__ uint4 dequant8_exact(uint2 c, float s) {
    float a[8];
    e4m3x8_to_f32(c, a);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = bf16_of_product(a[2 * i], s) | (bf16_of_product(a[2 * i + 1], s) << 16);
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Eight codes (byte k = element k) times s, each rounded once to bf16. The fp32 product p is
// converted by the packed round-to-nearest-even instruction, which is right unless p lies
// exactly on a bf16 midpoint while the exact product does not (see bf16_of_product); the
// residual a s - p of one fused multiply-add, exact while p is a normal number, tells the two
// apart. Exact midpoints are common (when a group's scale has few significant bits many
// products are exact and sit on midpoints) and are right as converted; only a granule with an
// inexact one, a NaN code, or a scale below 2^-117 (where a nonzero product, at least 2^-9 s,
// may be subnormal) takes the exact route.
__device__ __forceinline__ uint4 dequant8(uint2 c, float s) {
    float a[8];
    e4m3x8_to_f32(c, a);
    uint32_t o[4];
    bool slow = has_e4m3_nan(c.x) | has_e4m3_nan(c.y) | !(fabsf(s) >= 0x1p-117f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float p0 = a[2 * i] * s, p1 = a[2 * i + 1] * s;
        const float r0 = fmaf(a[2 * i], s, -p0), r1 = fmaf(a[2 * i + 1], s, -p1);
        slow |= (((__float_as_uint(p0) & 0xFFFFu) == 0x8000u) & (r0 != 0.f)) |
                (((__float_as_uint(p1) & 0xFFFFu) == 0x8000u) & (r1 != 0.f));
        const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
        o[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    if (slow) return dequant8_exact(c, s);
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// A thread takes 8 codes (an 8-byte load; 16 bytes of bf16 written, so a warp's stores cover 512
// contiguous bytes) of kDqUnroll granules a block-width apart, all loaded before any is
// converted; a 128-dim group is 16 granules sharing one scale. The grid is one wave of
// resident CTAs striding over the rows. blockIdx.y selects K (0) or V (1).
constexpr int kDqUnroll = 4, kDqThreads = 256;
struct DequantKvArgs {
    const uint8_t *codes[2];
    const float *scales[2];
    uint16_t *out[2];
    int64_t n_gran;                                  // 8-code granules per tensor
};

__global__ void __launch_bounds__(kDqThreads) dequantize_kv_fp8_kernel(DequantKvArgs a) {
    const bool v = blockIdx.y != 0;                  // selects, not indexes, the parameters
    const uint8_t *__restrict__ codes = v ? a.codes[1] : a.codes[0];
    const float *__restrict__ scales = v ? a.scales[1] : a.scales[0];
    uint16_t *__restrict__ out = v ? a.out[1] : a.out[0];
    const int64_t step = (int64_t)gridDim.x * kDqThreads * kDqUnroll;
    for (int64_t g0 = (int64_t)blockIdx.x * kDqThreads * kDqUnroll + threadIdx.x; g0 < a.n_gran; g0 += step) {
        uint2 c[kDqUnroll];
        float sc[kDqUnroll];
#pragma unroll
        for (int k = 0; k < kDqUnroll; ++k) {
            const int64_t g = g0 + (int64_t)k * kDqThreads;
            c[k] = g < a.n_gran ? __ldg(reinterpret_cast<const uint2 *>(codes + g * 8)) : make_uint2(0u, 0u);
            sc[k] = g < a.n_gran ? __ldg(scales + (g >> 4)) : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kDqUnroll; ++k) {
            const int64_t g = g0 + (int64_t)k * kDqThreads;
            if (g < a.n_gran) *reinterpret_cast<uint4 *>(out + g * 8) = dequant8(c[k], sc[k]);
        }
    }
}

int g_dq_resident[64];   // per device: co-resident dequantiser CTAs, 0 = unknown

int dq_resident() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int &slot = g_dq_resident[dev];
    if (slot == 0) {
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dequantize_kv_fp8_kernel, kDqThreads, 0) !=
                cudaSuccess ||
            per_sm < 1)
            return 0;
        slot = sms * per_sm;
    }
    return slot;
}

cudaError_t launch_dequantize_kv_fp8(const uint8_t *k_codes, const float *k_scales, uint16_t *k_out,
                                     const uint8_t *v_codes, const float *v_scales, uint16_t *v_out, int64_t n_rows,
                                     cudaStream_t st) {
    DequantKvArgs a{{k_codes, v_codes}, {k_scales, v_scales}, {k_out, v_out}, n_rows * 32};
    const int resident = dq_resident();
    if (resident == 0) return cudaErrorInvalidConfiguration;
    const unsigned ny = v_codes ? 2u : 1u;
    const int64_t need = (a.n_gran + kDqThreads * kDqUnroll - 1) / (kDqThreads * kDqUnroll);
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(need, resident / ny));
    dequantize_kv_fp8_kernel<<<dim3((unsigned)blocks, ny), kDqThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_pool_keys_fp8(const uint16_t *raw, int64_t n_tok, const int32_t *tok_off, const int32_t *blk_off,
                                 const int32_t *blk_begin, const int32_t *blk_end, int B, int64_t max_blocks,
                                 uint8_t *codes, float *scales, int64_t n_pooled, WsHeader *hdr, cudaStream_t st) {
    if (B == 0 || max_blocks == 0) return cudaSuccess;
    const int64_t threads = max_blocks * 16;
    dim3 grid((unsigned)((threads + 255) / 256), (unsigned)B);
    pool_keys_fp8_kernel<<<grid, 256, 0, st>>>(raw, n_tok, tok_off, blk_off, blk_begin, blk_end, max_blocks, codes,
                                               scales, n_pooled, hdr);
    return cudaGetLastError();
}

namespace {
int g_f8_resident[64];   // per device: co-resident scan CTAs, 0 = unknown

int f8_resident() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int &slot = g_f8_resident[dev];
    if (slot == 0) {
        if (cudaFuncSetAttribute(index_score_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kF8Smem) !=
            cudaSuccess)
            return 0;
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, index_score_fp8_kernel, kF8Threads, kF8Smem) !=
                cudaSuccess ||
            per_sm < 1)
            return 0;
        slot = sms * per_sm;
    }
    return slot;
}
}  // namespace

cudaError_t launch_index_score_fp8(const uint16_t *q_idx, const int32_t *q_seq, const int32_t *q_pos, int Nq,
                                   const uint8_t *codes, const float *scales, int64_t n_pooled,
                                   const int32_t *blk_off, float *scores, int64_t ld, WsHeader *hdr,
                                   cudaStream_t st) {
    if (Nq == 0 || ld == 0) return cudaSuccess;
    const int resident = f8_resident();
    if (resident == 0) return cudaErrorInvalidConfiguration;
    // one wave: the resident CTAs shared over the rows, at most one per 128-row tile of the longest
    const int64_t tiles = (ld + kF8TileRows - 1) / kF8TileRows;
    const int64_t per_row = std::max<int64_t>(1, std::min<int64_t>(tiles, resident / Nq));
    dim3 grid((unsigned)per_row, (unsigned)Nq);
    index_score_fp8_kernel<<<grid, kF8Threads, kF8Smem, st>>>(q_idx, q_seq, q_pos, codes, scales, n_pooled, blk_off,
                                                             scores, ld, hdr);
    return cudaGetLastError();
}

}  // namespace qsa
