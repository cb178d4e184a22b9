// a3 — fixed-budget block selection: the min(512, nb) best blocks of each row,
// ties to the lower block id, written in ascending id order ("3090x3で 314 万コンテキスト",
// section "なぜ"; tie rule as in "125B MoE を 3090 3 枚で運用する vLLM 最適化編" section 3.3).
//
// One CTA per row: a three-digit (11/11/10-bit) radix select on order-preserving
// 32-bit score keys finds the exact key T of the k-th best block and how many blocks
// with key == T to keep; a final pass in index order emits every block with key > T
// and the first `need` blocks with key == T, so the output is ascending by construction.
#include "qsa_internal.cuh"

namespace qsa {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kBins = 2048;

// Find the digit d (bins high -> low) where the running count from the top first
// reaches `need`. Returns d and the count strictly above d. Uses warp 0 only.
__device__ __forceinline__ void find_digit(const uint32_t *hist, int nbins, uint32_t need, int *d_out,
                                           uint32_t *above_out) {
    const int lane = threadIdx.x & 31;
    const int per = nbins / 32;
    // lane L owns bins [L*per, (L+1)*per)
    uint32_t sum = 0;
    for (int i = 0; i < per; ++i) sum += hist[lane * per + i];
    // inclusive suffix sum over lanes (from lane 31 down)
    uint32_t suf = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += v;
    }
    const uint32_t above_lane = suf - sum;   // count in bins of higher lanes
    const bool hit = above_lane < need && suf >= need;
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    const int L = 31 - __clz(m);             // exactly one lane hits (counts are monotone)
    if (lane == L) {
        uint32_t run = above_lane;
        int d = (L + 1) * per - 1;
        for (; d >= L * per; --d) {
            if (run + hist[d] >= need) break;
            run += hist[d];
        }
        *d_out = d;
        *above_out = run;
    }
}

__global__ void __launch_bounds__(kTopkThreads) topk_rows_kernel(const float *__restrict__ scores, int64_t ld,
                                                                 const int32_t *q_pos, int32_t *__restrict__ blocks,
                                                                 int32_t *__restrict__ count, WsHeader *hdr) {
    __shared__ uint32_t hist[kBins];
    __shared__ int s_digit;
    __shared__ uint32_t s_above;
    __shared__ uint32_t s_wsum[2][kTopkWarps];

    const int row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int p = q_pos[row];
    const int64_t nb = p >= 0 ? (p >> 2) : -1;
    int32_t *out = blocks + (int64_t)row * kBlockTopK;
    if (nb < 0 || nb > ld) {
        if (tid == 0) {
            record_error(hdr, QSA_ERR_DEVICE_BOUNDS, kWhereTopk, row);
            count[row] = 0;
        }
        for (int i = tid; i < kBlockTopK; i += kTopkThreads) out[i] = -1;
        return;
    }
    if (nb <= kBlockTopK) {                  // the budget covers the whole history: dense
        for (int i = tid; i < kBlockTopK; i += kTopkThreads) out[i] = i < nb ? i : -1;
        if (tid == 0) count[row] = (int32_t)nb;
        return;
    }
    const float *s = scores + (int64_t)row * ld;

    uint32_t prefix = 0, pmask = 0, need = kBlockTopK;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = shifts[pass];
        const uint32_t dmask = (1u << widths[pass]) - 1u;
        const int nbins = 1 << widths[pass];
        for (int i = tid; i < nbins; i += kTopkThreads) hist[i] = 0;
        __syncthreads();
        for (int64_t i = tid; i < nb; i += kTopkThreads) {
            const uint32_t key = score_key(__ldg(s + i));
            if ((key & pmask) == prefix) atomicAdd(&hist[(key >> sh) & dmask], 1u);
        }
        __syncthreads();
        if (warp == 0) find_digit(hist, nbins, need, &s_digit, &s_above);
        __syncthreads();
        prefix |= (uint32_t)s_digit << sh;
        pmask |= dmask << sh;
        need -= s_above;
        __syncthreads();
    }
    const uint32_t T = prefix;               // exact key of the k-th best block
    const uint32_t need_eq = need;           // how many blocks with key == T are kept (>= 1)

    uint32_t written = 0, eq_seen = 0;
    for (int64_t base = 0; base < nb; base += kTopkThreads) {
        const int64_t i = base + tid;
        const uint32_t key = i < nb ? score_key(__ldg(s + i)) : 0u;
        const bool gt = i < nb && key > T;
        const bool eq = i < nb && key == T;
        const unsigned beq = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) s_wsum[0][warp] = __popc(beq);
        __syncthreads();
        uint32_t eq_before = eq_seen, eq_total = 0;
        for (int w = 0; w < kTopkWarps; ++w) {
            const uint32_t c = s_wsum[0][w];
            if (w < warp) eq_before += c;
            eq_total += c;
        }
        eq_before += __popc(beq & ((1u << lane) - 1u));
        const bool take = gt || (eq && eq_before < need_eq);
        const unsigned bt = __ballot_sync(0xffffffffu, take);
        if (lane == 0) s_wsum[1][warp] = __popc(bt);
        __syncthreads();
        uint32_t pos = written, t_total = 0;
        for (int w = 0; w < kTopkWarps; ++w) {
            const uint32_t c = s_wsum[1][w];
            if (w < warp) pos += c;
            t_total += c;
        }
        pos += __popc(bt & ((1u << lane) - 1u));
        if (take && pos < kBlockTopK) out[pos] = (int32_t)i;
        written += t_total;
        eq_seen += eq_total;
        __syncthreads();
    }
    if (tid == 0) {
        count[row] = kBlockTopK;
        if (written != kBlockTopK) record_error(hdr, QSA_ERR_DEVICE_BOUNDS, kWhereTopk, row);
    }
}

size_t topk_scratch_bytes(int Nq, int64_t ld) {
    (void)Nq;
    (void)ld;
    return 0;
}

cudaError_t launch_topk_blocks(const float *scores, int64_t ld, const int32_t *q_pos, int Nq, int32_t *blocks,
                               int32_t *count, WsHeader *hdr, void *scratch, size_t scratch_bytes, cudaStream_t st) {
    (void)scratch;
    (void)scratch_bytes;
    if (Nq == 0) return cudaSuccess;
    topk_rows_kernel<<<Nq, kTopkThreads, 0, st>>>(scores, ld, q_pos, blocks, count, hdr);
    return cudaGetLastError();
}

}  // namespace qsa
