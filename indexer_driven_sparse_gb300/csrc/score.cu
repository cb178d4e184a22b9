// a2 — indexer scores of every visible pooled block ("3090x3で 314 万コンテキスト",
// sections "なぜ" and "VRAM に残す必要があるもの": the scan over all pooled keys is the
// one read that grows with context). HBM-bound streaming dot products: each warp
// covers 32 consecutive 256-byte rows with 128-bit coalesced non-allocating loads
// (a half-warp per row, 8 dims per lane), all 16 loads of a lane issued before use.
#include "qsa_internal.cuh"

namespace qsa {

constexpr int kScoreThreads = 256;
constexpr int kRowsPerWarp = 32;
constexpr int kRowsPerCta = kRowsPerWarp * (kScoreThreads / 32);   // 256 rows = 64 KiB

__global__ void __launch_bounds__(kScoreThreads) index_score_kernel(const uint16_t *__restrict__ q_idx,
                                                                    const int32_t *q_seq, const int32_t *q_pos,
                                                                    const uint16_t *__restrict__ pooled,
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
    const int64_t row0 = (int64_t)blockIdx.x * kRowsPerCta + warp * kRowsPerWarp;
    if (row0 >= nb) return;
    const int half = lane >> 4, c = lane & 15;
    float qf[8];
    unpack8(ldg_nc_v4(q_idx + (int64_t)r * kIdxDim + c * 8), qf);
    const uint16_t *base = pooled + (off + row0) * kIdxDim + c * 8;
    uint4 v[kRowsPerWarp / 2];
#pragma unroll
    for (int j = 0; j < kRowsPerWarp / 2; ++j) {
        const int64_t row = row0 + 2 * j + half;
        v[j] = row < nb ? ldg_nc_v4(base + (int64_t)(2 * j + half) * kIdxDim) : make_uint4(0, 0, 0, 0);
    }
    float part[kRowsPerWarp / 2];
#pragma unroll
    for (int j = 0; j < kRowsPerWarp / 2; ++j) {
        float f[8];
        unpack8(v[j], f);
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) s = fmaf(f[e], qf[e], s);
        part[j] = s;
    }
#pragma unroll
    for (int j = 0; j < kRowsPerWarp / 2; ++j) {
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) part[j] += __shfl_xor_sync(0xffffffffu, part[j], o);
    }
    // lane 0 holds rows 2j, lane 16 rows 2j+1: let lane 2j+half write row 2j+half.
    float mine = 0.f;
#pragma unroll
    for (int j = 0; j < kRowsPerWarp / 2; ++j) {
        const float a = __shfl_sync(0xffffffffu, part[j], 0);
        const float b = __shfl_sync(0xffffffffu, part[j], 16);
        if (lane == 2 * j) mine = a;
        if (lane == 2 * j + 1) mine = b;
    }
    const int64_t my_row = row0 + lane;
    if (my_row < nb) scores[(int64_t)r * ld + my_row] = mine;
}

cudaError_t launch_index_score(const uint16_t *q_idx, const int32_t *q_seq, const int32_t *q_pos, int Nq,
                               const uint16_t *pooled, int64_t n_pooled, const int32_t *blk_off, float *scores,
                               int64_t ld, WsHeader *hdr, cudaStream_t st) {
    if (Nq == 0 || ld == 0) return cudaSuccess;
    dim3 grid((unsigned)((ld + kRowsPerCta - 1) / kRowsPerCta), (unsigned)Nq);
    index_score_kernel<<<grid, kScoreThreads, 0, st>>>(q_idx, q_seq, q_pos, pooled, n_pooled, blk_off, scores, ld,
                                                       hdr);
    return cudaGetLastError();
}

}  // namespace qsa
