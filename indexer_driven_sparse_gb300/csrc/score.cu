// a2 — indexer scores of every visible pooled block ("3090x3で 314 万コンテキスト",
// sections "なぜ" and "VRAM に残す必要があるもの": the scan over all pooled keys is the
// one read that grows with context). HBM-bound streaming dot products: each warp
// covers 32 consecutive 256-byte rows; lane l loads dims 4l .. 4l+3 of every row (8-byte
// coalesced non-allocating loads, all 32 issued before use) and a reduce-scatter over the
// 32 rows leaves row l's score in lane l, in the evaluation order of dot4_bf16.
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
    float q4[4];
    load_q4(q_idx + (int64_t)r * kIdxDim, lane, q4);
    const uint16_t *base = pooled + (off + row0) * kIdxDim + 4 * lane;
    uint2 x[kRowsPerWarp];
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) {
        const int64_t row = row0 + j;
        if (row < nb) {
            asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                         : "=r"(x[j].x), "=r"(x[j].y) : "l"(base + (int64_t)j * kIdxDim));
        } else {
            x[j] = make_uint2(0, 0);
        }
    }
    float part[kRowsPerWarp];
#pragma unroll
    for (int j = 0; j < kRowsPerWarp; ++j) part[j] = dot4_bf16(x[j], q4);
    const float mine = reduce_rows<kRowsPerWarp>(part, lane);      // row row_of_lane<32>(lane) = lane
    const int64_t my_row = row0 + row_of_lane<kRowsPerWarp>(lane);
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
