// a1 — pooled indexer keys: one 128 x bf16 key per complete 4-token block
// ("3090x3で 314 万コンテキスト", section "VRAM に残す必要があるもの"). The mean of the
// four raw keys is formed exactly in fp64 and rounded once to bf16 (nearest-even).
#include "qsa_internal.cuh"

namespace qsa {

// 16 threads per block, each owning 8 of the 128 dims (16-byte loads and stores).
__global__ void __launch_bounds__(256) pool_keys_kernel(const uint16_t *__restrict__ raw, int64_t n_tok,
                                                        const int32_t *tok_off, const int32_t *blk_off,
                                                        const int32_t *blk_begin, const int32_t *blk_end,
                                                        int64_t max_blocks, uint16_t *__restrict__ pooled,
                                                        int64_t n_pooled, WsHeader *hdr) {
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
    if (b >= be) return;
    const uint16_t *src = raw + (t0 + kRatio * b) * kIdxDim + c * 8;
    float f0[8], f1[8], f2[8], f3[8];
    unpack8(ldg_nc_v4(src), f0);
    unpack8(ldg_nc_v4(src + kIdxDim), f1);
    unpack8(ldg_nc_v4(src + 2 * kIdxDim), f2);
    unpack8(ldg_nc_v4(src + 3 * kIdxDim), f3);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const double s0 = (((double)f0[2 * i] + (double)f1[2 * i]) + (double)f2[2 * i]) + (double)f3[2 * i];
        const double s1 = (((double)f0[2 * i + 1] + (double)f1[2 * i + 1]) + (double)f2[2 * i + 1]) +
                          (double)f3[2 * i + 1];
        w[i] = (uint32_t)double_to_bf16_rne(s0 * 0.25) | ((uint32_t)double_to_bf16_rne(s1 * 0.25) << 16);
    }
    *reinterpret_cast<uint4 *>(pooled + (bo + b) * kIdxDim + c * 8) = make_uint4(w[0], w[1], w[2], w[3]);
}

cudaError_t launch_pool_keys(const uint16_t *raw, int64_t n_tok, const int32_t *tok_off, const int32_t *blk_off,
                             const int32_t *blk_begin, const int32_t *blk_end, int B, int64_t max_blocks,
                             uint16_t *pooled, int64_t n_pooled, WsHeader *hdr, cudaStream_t st) {
    if (B == 0 || max_blocks == 0) return cudaSuccess;
    const int64_t threads = max_blocks * 16;
    dim3 grid((unsigned)((threads + 255) / 256), (unsigned)B);
    pool_keys_kernel<<<grid, 256, 0, st>>>(raw, n_tok, tok_off, blk_off, blk_begin, blk_end, max_blocks, pooled,
                                           n_pooled, hdr);
    return cudaGetLastError();
}

}  // namespace qsa
