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
#include "qsa_internal.cuh"

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
constexpr int kF8RowsPerWarp = 32;
constexpr int kF8RowsPerCta = kF8RowsPerWarp * (kF8Threads / 32);   // 256 rows = 32 KiB of codes

// Each warp covers 32 consecutive 128-byte code rows: a row is 8 lanes x 16 bytes (16 dims
// per lane), so one 16-byte load instruction of the warp covers 4 rows; all 8 loads of a
// lane are issued before use. The 32 scales of the warp's rows are one coalesced load.
__global__ void __launch_bounds__(kF8Threads) index_score_fp8_kernel(const uint16_t *__restrict__ q_idx,
                                                                     const int32_t *q_seq, const int32_t *q_pos,
                                                                     const uint8_t *__restrict__ codes,
                                                                     const float *__restrict__ scales,
                                                                     int64_t n_pooled, const int32_t *blk_off,
                                                                     float *__restrict__ scores, int64_t ld,
                                                                     WsHeader *hdr) {
    const int r = blockIdx.y;
    const int p = q_pos[r];
    const int64_t nb = p >= 0 ? (p >> 2) : -1;
    const int64_t off = blk_off[q_seq != nullptr ? q_seq[r] : 0];   // NULL: one sequence
    if (nb < 0 || nb > ld || off < 0 || off + nb > n_pooled) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(hdr, QSA_ERR_DEVICE_BOUNDS, kWhereScore, r);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row0 = (int64_t)blockIdx.x * kF8RowsPerCta + warp * kF8RowsPerWarp;
    if (row0 >= nb) return;   // whole warps leave
    const int g = lane >> 3, c = lane & 7;
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
    const uint8_t *base = codes + (off + row0) * kIdxDim + c * 16;
    uint4 v[kF8RowsPerWarp / 4];
#pragma unroll
    for (int j = 0; j < kF8RowsPerWarp / 4; ++j) {
        const int64_t row = row0 + 4 * j + g;
        v[j] = row < nb ? ldg_nc_v4(base + (int64_t)(4 * j + g) * kIdxDim) : make_uint4(0, 0, 0, 0);
    }
    const int64_t my_row = row0 + lane;
    const float sc = my_row < nb ? __ldg(scales + off + my_row) : 0.f;
    float part[kF8RowsPerWarp / 4];
#pragma unroll
    for (int j = 0; j < kF8RowsPerWarp / 4; ++j) {
        float f[16];
        e4m3x16_to_f32(v[j], f);
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) s = fmaf(f[e], qf[e], s);
        part[j] = s;
    }
#pragma unroll
    for (int j = 0; j < kF8RowsPerWarp / 4; ++j) {
#pragma unroll
        for (int o = 4; o >= 1; o >>= 1) part[j] += __shfl_xor_sync(0xffffffffu, part[j], o);
    }
    // row 4j + g sits in every lane of group g: lane L takes row L = 4 (L >> 2) + (L & 3)
    float mine = 0.f;
#pragma unroll
    for (int j = 0; j < kF8RowsPerWarp / 4; ++j) {
        const float a = __shfl_sync(0xffffffffu, part[j], (lane & 3) * 8);
        if (j == (lane >> 2)) mine = a;
    }
    if (my_row < nb) scores[(int64_t)r * ld + my_row] = mine * sc;
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

cudaError_t launch_index_score_fp8(const uint16_t *q_idx, const int32_t *q_seq, const int32_t *q_pos, int Nq,
                                   const uint8_t *codes, const float *scales, int64_t n_pooled,
                                   const int32_t *blk_off, float *scores, int64_t ld, WsHeader *hdr,
                                   cudaStream_t st) {
    if (Nq == 0 || ld == 0) return cudaSuccess;
    dim3 grid((unsigned)((ld + kF8RowsPerCta - 1) / kF8RowsPerCta), (unsigned)Nq);
    index_score_fp8_kernel<<<grid, kF8Threads, 0, st>>>(q_idx, q_seq, q_pos, codes, scales, n_pooled, blk_off,
                                                        scores, ld, hdr);
    return cudaGetLastError();
}

}  // namespace qsa
