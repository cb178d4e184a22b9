// Fused decode layer-step for a small batch: a1 (pool the newest block), a2 (score every
// visible block), a3 (exact top-512, ties to the lower id), a4 (gathered GQA attention)
// and a5 (log-sum-exp merge) in ONE cooperative launch.
//
//   "3090x3で 314 万コンテキスト", section "なぜ": a token reads K/V of exactly 2048 selected
//   tokens; "VRAM に残す必要があるもの": the pooled-key scan is the only read that grows with
//   context; "カーネルを書き換えずに済む": row address (tok * n_kv_heads + kv) * head_dim + d.
//   "GLM-5.3 最適化 第2部", section "DCP": partials over disjoint key sets merge by LSE.
//   "125B MoE を 3090 3 枚で運用する vLLM 最適化編", section 3.3: ordered-integer top-k keys
//   with the id in the low bits, and a last-CTA-done finaliser.
//
// Layout of the work: each sequence (row) owns a contiguous group of CTAs (sized by its
// context); CTA j of a row owns the contiguous block range [nb*j/c, nb*(j+1)/c).
//   1. The CTA owning block nb-1 re-pools it from the raw keys (exact fp64 mean).
//   2. Each CTA streams its pooled rows through a 4-stage shared-memory ring filled by
//      bulk async copies (TMA engine), keeps the 32-bit order-preserving score keys of its
//      range in shared memory and histograms their top 12 bits.
//   3. Row barrier; the last CTA to arrive finds the threshold bin and how many of its
//      members are still needed.
//   4. Each CTA counts its blocks above the bin and appends the bin's members (64-bit
//      key = score key << 32 | ~block) to a candidate list.
//   5. Row barrier; the last arriver radix-selects the exact 64-bit threshold among the
//      candidates and publishes every CTA's output offset.
//   6. Each CTA writes its selected ids (ascending) and attends its own selected tokens
//      (plus the query's own block, in the row's last CTA), producing an (m, l, acc) partial.
//   7. Row barrier; the CTAs of the row merge all partials by LSE, each a slice of outputs.
// Rows with nb <= 512 (dense) skip steps 2-5. Every wait is bounded: a barrier or mbarrier
// that gives up records QSA_ERR_DEVICE_TIMEOUT and the CTA returns.
#include "qsa_internal.cuh"
#include "qsa_ptx.cuh"

namespace qsa {

constexpr int kStepThreads = 512;
constexpr int kStepWarps = kStepThreads / 32;
constexpr int kHistBins = 4096;                       // top 12 bits of the score key
constexpr int kHistShift = 20;
constexpr int kRingStages = 4;
constexpr int kChunkRows = 128;                       // 128 pooled rows = 32 KiB per stage
constexpr int kChunkBytes = kChunkRows * kIdxDim * 2;
constexpr int kMaxKeys = 12288;                       // score keys per CTA kept on chip
constexpr int kAttnTok = 32;                          // tokens per attention step
constexpr int kAttnWeightBlocks = 16384;              // attention cost of a row, in scanned blocks

constexpr size_t kRingOff = 0;
constexpr size_t kKeysOff = kRingOff + (size_t)kRingStages * kChunkBytes;
constexpr size_t kHistOff = kKeysOff + (size_t)kMaxKeys * 4;
constexpr size_t kNewRowOff = kHistOff + (size_t)kHistBins * 4;
constexpr size_t kMbarOff = kNewRowOff + 256;
constexpr size_t kStepSmem = kMbarOff + 64;

struct StepRowState {
    uint32_t bar_count;
    uint32_t bar_gen;
    int32_t t1;                 // threshold bin (top 12 key bits)
    int32_t need;               // members of the threshold bin still to take
    unsigned long long t64;     // exact 64-bit threshold key
    uint32_t cand_count;
    int32_t pad;
    int32_t definite[kMaxStepCtas];
    int32_t offset[kMaxStepCtas];
};

constexpr size_t kRowStateBytes = (sizeof(StepRowState) + 255) / 256 * 256;
__host__ __device__ constexpr size_t step_row_state_bytes() { return kRowStateBytes; }

StepLayout step_layout(int B, int64_t max_blocks, int Hq) {
    StepLayout L;
    L.rows = kWsHeaderBytes;
    L.hist = L.rows + (size_t)B * step_row_state_bytes();
    L.cands = L.hist + (size_t)B * kHistBins * 4;
    L.part = L.cands + ((size_t)B * (size_t)max_blocks * 8 + 255) / 256 * 256;
    L.total = L.part + (size_t)kMaxStepCtas * Hq * (kHeadDim + 2) * 4;
    return L;
}

struct RowPart {
    int row, jj, cr, first;
};

__device__ __forceinline__ int64_t row_weight(const int32_t *ctx_len, int r) {
    const int p = ctx_len[r];
    return (p >= 0 ? (int64_t)(p >> 2) : 0) + kAttnWeightBlocks;
}

// Warp 0: split gridDim.x CTAs over B <= 64 rows (1 each + a share by weight) and find
// this CTA's row. Every CTA computes the same split.
__device__ void partition_rows(const int32_t *ctx_len, int B, RowPart *out) {
    const int lane = threadIdx.x & 31;
    const int C = gridDim.x;
    const int64_t w0 = lane < B ? row_weight(ctx_len, lane) : 0;
    const int64_t w1 = lane + 32 < B ? row_weight(ctx_len, lane + 32) : 0;
    int64_t W = w0 + w1;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    const int64_t R = C - B;
    const int e0 = lane < B ? (int)(R * w0 / W) : 0;
    const int e1 = lane + 32 < B ? (int)(R * w1 / W) : 0;
    int E = e0 + e1;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) E += __shfl_xor_sync(0xffffffffu, E, o);
    const int left = (int)R - E;
    const int c0 = lane < B ? 1 + e0 + (lane < left ? 1 : 0) : 0;
    const int c1 = lane + 32 < B ? 1 + e1 + (lane + 32 < left ? 1 : 0) : 0;
    int s0 = c0, s1 = c1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, s0, o);
        const int b = __shfl_up_sync(0xffffffffu, s1, o);
        if (lane >= o) {
            s0 += a;
            s1 += b;
        }
    }
    s1 += __shfl_sync(0xffffffffu, s0, 31);
    const int bid = blockIdx.x;
    const bool in0 = lane < B && bid >= s0 - c0 && bid < s0;
    const bool in1 = lane + 32 < B && bid >= s1 - c1 && bid < s1;
    if (in0) *out = RowPart{lane, bid - (s0 - c0), c0, s0 - c0};
    if (in1) *out = RowPart{lane + 32, bid - (s1 - c1), c1, s1 - c1};
}

// Arrive at the row barrier. Returns 1 for the last CTA to arrive (which must call
// row_release after its exclusive work), 0 for the others once released, -1 on timeout.
__device__ int row_arrive(StepRowState *rs, int n, WsHeader *hdr, int row, int *s_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t gen = ld_acquire_u32(&rs->bar_gen);
        __threadfence();
        const uint32_t arrived = atomicAdd(&rs->bar_count, 1u) + 1u;
        int res = 1;
        if (arrived != (uint32_t)n) {
            res = 0;
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_u32(&rs->bar_gen) == gen) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    record_error(hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereStep, row);
                    res = -1;
                    break;
                }
                __nanosleep(100);
            }
        }
        __threadfence();
        *s_flag = res;
    }
    __syncthreads();
    return *s_flag;
}

__device__ void row_release(StepRowState *rs) {
    __syncthreads();
    if (threadIdx.x == 0) {
        rs->bar_count = 0;
        __threadfence();
        atomicAdd(&rs->bar_gen, 1u);
    }
}

// Warp 0: in hist[0..nbins) (bins high = better), find the bin where the count from the
// top first reaches `need`; returns it and the count strictly above it.
__device__ void warp_find_bin(const uint32_t *hist, int nbins, uint32_t need, int *d_out, uint32_t *above_out) {
    const int lane = threadIdx.x & 31;
    const int per = nbins / 32;
    uint32_t sum = 0;
    for (int i = 0; i < per; ++i) sum += hist[lane * per + i];
    uint32_t suf = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += v;
    }
    const uint32_t above_lane = suf - sum;
    const unsigned m = __ballot_sync(0xffffffffu, above_lane < need && suf >= need);
    const int L = m ? 31 - __clz(m) : 0;
    if (lane == L) {
        uint32_t run = above_lane;
        int d = (L + 1) * per - 1;
        for (; d > L * per; --d) {
            if (run + hist[d] >= need) break;
            run += hist[d];
        }
        *d_out = d;
        *above_out = run;
    }
}

// CTA-wide: the need-th largest of n 64-bit keys in global memory whose bits above
// `start` are all equal. 11-bit radix passes, stopping early once the chosen bin holds
// exactly the keys still needed.
__device__ unsigned long long select_kth_key64(const unsigned long long *keys, uint32_t n, uint32_t need,
                                               int start, uint32_t *hist, int *s_d, uint32_t *s_above) {
    unsigned long long prefix = (__ldcg(&keys[0]) >> start) << start;
    int hi = start;
    while (hi > 0) {
        const int width = hi >= 11 ? 11 : hi;
        const int shift = hi - width;
        const int nbins = 1 << width;
        for (int i = threadIdx.x; i < 2048; i += kStepThreads) hist[i] = 0;
        __syncthreads();
        for (uint32_t i = threadIdx.x; i < n; i += kStepThreads) {
            const unsigned long long k = __ldcg(&keys[i]);
            if ((k >> hi) == (prefix >> hi)) atomicAdd(&hist[(uint32_t)(k >> shift) & (nbins - 1)], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) warp_find_bin(hist, nbins < 32 ? 32 : nbins, need, s_d, s_above);
        __syncthreads();
        const int d = *s_d;
        const uint32_t in_bin = hist[d];
        prefix |= (unsigned long long)d << shift;
        need -= *s_above;
        __syncthreads();
        if (in_bin == need) return prefix;           // the whole bin is kept
        hi = shift;
    }
    return prefix;
}

template <int G>
__global__ void __launch_bounds__(kStepThreads, 1) decode_step_kernel(StepArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem + kKeysOff);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + kHistOff);
    uint16_t *newrow = reinterpret_cast<uint16_t *>(smem + kNewRowOff);
    const uint32_t mbar0 = smem_u32(smem + kMbarOff);
    const uint32_t ring0 = smem_u32(smem + kRingOff);

    __shared__ RowPart s_part;
    __shared__ int s_flag, s_d, s_bad;
    __shared__ uint32_t s_above;
    __shared__ int32_t s_sel[kBlockTopK];
    __shared__ int s_nsel;
    __shared__ uint32_t s_cnt[kMaxStepCtas];
    __shared__ uint32_t s_wsum[kStepWarps];
    __shared__ float s_m[2 * kMaxGroup], s_l[2 * kMaxGroup], s_alpha[2 * kMaxGroup];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hq = a.n_q_heads, Hkv = a.n_kv_heads;

    if (warp == 0) partition_rows(a.ctx_len, a.B, &s_part);
    __syncthreads();
    const int row = s_part.row, jj = s_part.jj, cr = s_part.cr, first = s_part.first;

    // ---- row geometry (identical in every CTA of the row)
    const int p = a.ctx_len[row];
    const int64_t base = a.tok_off[row], end = a.tok_off[row + 1];
    const int64_t boff = a.blk_off[row];
    const int64_t nb = p >= 0 ? (p >> 2) : 0;
    const int64_t max_range = (nb + cr - 1) / cr;
    const bool ok = p >= 0 && base >= 0 && end <= a.n_tok && base + p + 1 <= end && boff >= 0 &&
                    boff + nb <= a.n_pooled && nb <= a.max_blocks && max_range <= kMaxKeys;
    if (!ok) {
        if (jj == 0 && tid == 0) record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereStep, row);
        return;
    }
    StepRowState *rs = reinterpret_cast<StepRowState *>(reinterpret_cast<char *>(a.rows) +
                                                        (size_t)row * step_row_state_bytes());
    const int64_t lo = nb * jj / cr, hi = nb * (jj + 1) / cr;
    const int n_mine = (int)(hi - lo);
    const bool dense = nb <= kBlockTopK;
    const bool owner_new = nb >= 1 && hi == nb && lo < hi;     // owns block nb-1

    // ---- 1. re-pool block nb-1 (exact mean of its four raw keys)
    if (owner_new && warp == 0 && lane < 16) {
        const uint16_t *src = a.raw_idx_k + (base + kRatio * (nb - 1)) * kIdxDim + lane * 8;
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
        const uint4 v = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4 *>(a.pooled + (boff + nb - 1) * kIdxDim + lane * 8) = v;
        *reinterpret_cast<uint4 *>(newrow + lane * 8) = v;
    }

    if (!dense) {
        // ---- 2. scan: bulk copies into a 4-stage ring, scores -> keys + histogram
        const int n_tma = owner_new ? n_mine - 1 : n_mine;
        const int n_chunks = (n_tma + kChunkRows - 1) / kChunkRows;
        for (int i = tid; i < kHistBins; i += kStepThreads) hist[i] = 0;
        if (tid == 0) {
            for (int s = 0; s < kRingStages; ++s) mbar_init(mbar0 + 8 * s, 1);
            fence_mbar_init();
        }
        __syncthreads();
        const uint16_t *gsrc = a.pooled + (boff + lo) * kIdxDim;
        if (tid == 0) {
            for (int c = 0; c < n_chunks && c < kRingStages; ++c) {
                const uint32_t bytes = (uint32_t)min(kChunkRows, n_tma - c * kChunkRows) * kIdxDim * 2;
                mbar_arrive_expect_tx(mbar0 + 8 * c, bytes);
                bulk_g2s(ring0 + c * kChunkBytes, gsrc + (int64_t)c * kChunkRows * kIdxDim, bytes, mbar0 + 8 * c);
            }
        }
        float qf[8];
        unpack8(ldg_nc_v4(a.q_idx + (int64_t)row * kIdxDim + (lane & 15) * 8), qf);
        const int half = lane >> 4, c16 = lane & 15;
        for (int c = 0; c < n_chunks; ++c) {
            const int stage = c % kRingStages;
            if (!mbar_wait_bounded(mbar0 + 8 * stage, (c / kRingStages) & 1, kWaitLimitNs)) {
                // give up: wait (bounded) for every copy still in flight, then leave
                if (tid == 0) {
                    record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereStep, row);
                    for (int c2 = c; c2 < n_chunks && c2 < c + kRingStages; ++c2)
                        mbar_wait_bounded(mbar0 + 8 * (c2 % kRingStages), (c2 / kRingStages) & 1, kWaitLimitNs);
                }
                __syncthreads();
                return;
            }
            const int rows_c = min(kChunkRows, n_tma - c * kChunkRows);
            const uint16_t *buf = reinterpret_cast<const uint16_t *>(smem + kRingOff + (size_t)stage * kChunkBytes);
            // 16 warps x 8 rows: each half-warp takes one row per step
#pragma unroll
            for (int it = 0; it < kChunkRows / (2 * kStepWarps); ++it) {
                const int r = (warp * (kChunkRows / kStepWarps)) + it * 2 + half;
                float s = 0.f;
                if (r < rows_c) {
                    float f[8];
                    unpack8(*reinterpret_cast<const uint4 *>(buf + r * kIdxDim + c16 * 8), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) s = fmaf(f[e], qf[e], s);
                }
#pragma unroll
                for (int o = 8; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (c16 == 0 && r < rows_c) {
                    const uint32_t key = score_key(s);
                    keys[c * kChunkRows + r] = key;
                    atomicAdd(&hist[key >> kHistShift], 1u);
                }
            }
            __syncthreads();
            if (tid == 0 && c + kRingStages < n_chunks) {
                const int cn = c + kRingStages;
                const uint32_t bytes = (uint32_t)min(kChunkRows, n_tma - cn * kChunkRows) * kIdxDim * 2;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(mbar0 + 8 * stage, bytes);
                bulk_g2s(ring0 + stage * kChunkBytes, gsrc + (int64_t)cn * kChunkRows * kIdxDim, bytes,
                         mbar0 + 8 * stage);
            }
        }
        if (owner_new && warp == 0) {          // the freshly pooled block, from shared memory
            float f[8];
            unpack8(*reinterpret_cast<const uint4 *>(newrow + c16 * 8), f);
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) s = fmaf(f[e], qf[e], s);
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) {
                const uint32_t key = score_key(s);
                keys[n_mine - 1] = key;
                atomicAdd(&hist[key >> kHistShift], 1u);
            }
        }
        __syncthreads();
        uint32_t *ghist = a.hist + (size_t)row * kHistBins;
        for (int i = tid; i < kHistBins; i += kStepThreads)
            if (hist[i]) atomicAdd(&ghist[i], hist[i]);

        // ---- 3. threshold bin (last arriver). The test knob adds one arrival that never comes.
        const int stall = __ldcg(&a.hdr->debug) == kDebugStallBarrier ? 1 : 0;
        const int r1 = row_arrive(rs, cr + stall, a.hdr, row, &s_flag);
        if (r1 < 0) return;
        if (r1 == 1) {
            for (int i = tid; i < kHistBins; i += kStepThreads) {
                hist[i] = __ldcg(&ghist[i]);
                ghist[i] = 0;
            }
            __syncthreads();
            if (warp == 0) warp_find_bin(hist, kHistBins, kBlockTopK, &s_d, &s_above);
            __syncthreads();
            if (tid == 0) {
                rs->t1 = s_d;
                rs->need = kBlockTopK - (int)s_above;
            }
            row_release(rs);
        }
        __syncthreads();

        // ---- 4. classify: count blocks above the bin, append the bin's members
        const uint32_t t1 = (uint32_t)__ldcg(&rs->t1);
        unsigned long long *cands = a.cands + (size_t)row * a.max_blocks;
        uint32_t above = 0;
        for (int base_i = 0; base_i < n_mine; base_i += kStepThreads) {
            const int i = base_i + tid;
            const uint32_t key = i < n_mine ? keys[i] : 0u;
            const uint32_t bin = key >> kHistShift;
            const bool is_c = i < n_mine && bin == t1;
            above += (i < n_mine && bin > t1) ? 1u : 0u;
            const unsigned bal = __ballot_sync(0xffffffffu, is_c);
            uint32_t slot0 = 0;
            if (lane == 0 && bal) slot0 = atomicAdd(&rs->cand_count, (uint32_t)__popc(bal));
            slot0 = __shfl_sync(0xffffffffu, slot0, 0);
            const uint32_t slot = slot0 + __popc(bal & ((1u << lane) - 1u));
            if (is_c && slot < (uint32_t)nb) {          // nb <= max_blocks: the row's list capacity
                const uint32_t blk = (uint32_t)(lo + i);
                cands[slot] = ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - blk);
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) above += __shfl_xor_sync(0xffffffffu, above, o);
        if (lane == 0) s_wsum[warp] = above;
        __syncthreads();
        if (tid == 0) {
            uint32_t t = 0;
            for (int w = 0; w < kStepWarps; ++w) t += s_wsum[w];
            rs->definite[jj] = (int32_t)t;
        }

        // ---- 5. exact threshold and per-CTA offsets (last arriver)
        const int r2 = row_arrive(rs, cr, a.hdr, row, &s_flag);
        if (r2 < 0) return;
        if (r2 == 1) {
            const uint32_t n_c = min(__ldcg(&rs->cand_count), (uint32_t)nb);
            const uint32_t need = (uint32_t)__ldcg(&rs->need);
            const unsigned long long t64 = select_kth_key64(cands, n_c, need, 64 - 12, hist, &s_d, &s_above);
            for (int i = tid; i < cr; i += kStepThreads) s_cnt[i] = 0;
            __syncthreads();
            for (uint32_t i = tid; i < n_c; i += kStepThreads) {
                const unsigned long long k = __ldcg(&cands[i]);
                if (k >= t64) {
                    const int64_t b = (int64_t)(0xFFFFFFFFu - (uint32_t)k);
                    int j = (int)(b * cr / nb);
                    while (j + 1 < cr && nb * (j + 1) / cr <= b) ++j;
                    while (j > 0 && nb * j / cr > b) --j;
                    atomicAdd(&s_cnt[j], 1u);
                }
            }
            __syncthreads();
            if (tid == 0) {
                int32_t run = 0;
                for (int j = 0; j < cr; ++j) {
                    rs->offset[j] = run;
                    run += __ldcg(&rs->definite[j]) + (int32_t)s_cnt[j];
                }
                rs->t64 = t64;
                rs->cand_count = 0;
                if (run != kBlockTopK) record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereStep, row);
            }
            row_release(rs);
        }
        __syncthreads();
    }

    // ---- 6a. this CTA's selected blocks, ascending, and their output slots
    const unsigned long long t64 = dense ? 0ull : __ldcg(&rs->t64);
    const int out_off = dense ? (int)lo : __ldcg(&rs->offset[jj]);
    int32_t *blocks_row = a.blocks + (int64_t)row * kBlockTopK;
    int nsel = 0;
    for (int base_i = 0; base_i < n_mine; base_i += kStepThreads) {
        const int i = base_i + tid;
        bool take = false;
        if (i < n_mine) {
            if (dense) {
                take = true;
            } else {
                const uint32_t blk = (uint32_t)(lo + i);
                const unsigned long long k = ((unsigned long long)keys[i] << 32) | (0xFFFFFFFFu - blk);
                take = k >= t64;
            }
        }
        const unsigned bal = __ballot_sync(0xffffffffu, take);
        if (lane == 0) s_wsum[warp] = __popc(bal);
        __syncthreads();
        int before = nsel, total = 0;
        for (int w = 0; w < kStepWarps; ++w) {
            if (w < warp) before += s_wsum[w];
            total += s_wsum[w];
        }
        before += __popc(bal & ((1u << lane) - 1u));
        if (take && before < kBlockTopK && out_off + before < kBlockTopK) {
            s_sel[before] = (int32_t)(lo + i);
            blocks_row[out_off + before] = (int32_t)(lo + i);
        }
        nsel += total;
        __syncthreads();
    }
    nsel = min(nsel, kBlockTopK);
    const int kk = nb < kBlockTopK ? (int)nb : kBlockTopK;
    if (jj == 0) {
        for (int i = kk + tid; i < kBlockTopK; i += kStepThreads) blocks_row[i] = -1;
        if (tid == 0) a.count[row] = kk;
    }

    // ---- 6b. attention over this CTA's tokens (+ the query's own block in the last CTA)
    const bool last_cta = jj == cr - 1;
    const int n_tail = last_cta ? (int)(p - kRatio * nb + 1) : 0;
    const int n_tok = kRatio * nsel + n_tail;
    float *q_s = reinterpret_cast<float *>(smem + kRingOff);                 // [Hq][256], ring reused
    float *pw = q_s + 2 * kMaxGroup * kHeadDim;                              // [Hq][kAttnTok]
    int64_t *toks = reinterpret_cast<int64_t *>(pw + 2 * kMaxGroup * kAttnTok);
    __syncthreads();
    for (int i = tid; i < Hq * kHeadDim; i += kStepThreads)
        q_s[i] = bf16_bits_to_float(a.q[(int64_t)row * Hq * kHeadDim + i]) * a.scale_log2;
    if (tid < Hq) {
        s_m[tid] = -INFINITY;
        s_l[tid] = 0.f;
    }
    const int kv_t = tid >> 8, d_t = tid & 255;          // PV ownership: (KV head, dim)
    float acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = 0.f;
    __syncthreads();
    for (int t0 = 0; t0 < n_tok; t0 += kAttnTok) {
        const int n = min(kAttnTok, n_tok - t0);
        if (tid < n) {
            const int j = t0 + tid;
            const int64_t tk = j < kRatio * nsel ? (int64_t)kRatio * s_sel[j >> 2] + (j & 3)
                                                 : kRatio * nb + (j - kRatio * nsel);
            toks[tid] = base + tk;
        }
        __syncthreads();
        for (int i = warp; i < n; i += kStepWarps) {
            for (int kv = 0; kv < Hkv; ++kv) {
                float kf[8];
                unpack8(ldg_nc_v4(a.k_cache + (toks[i] * Hkv + kv) * kHeadDim + lane * 8), kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float *qh = q_s + (kv * G + g) * kHeadDim + lane * 8;
                    float s = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) s = fmaf(kf[e], qh[e], s);
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                    if (lane == 0) pw[(kv * G + g) * kAttnTok + i] = s;
                }
            }
        }
        __syncthreads();
        for (int h = warp; h < Hq; h += kStepWarps) {
            const float x = lane < n ? pw[h * kAttnTok + lane] : -INFINITY;
            float cm = x;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
            const float mo = s_m[h];
            const float mn = fmaxf(mo, cm);
            const float e = lane < n ? exp2f(x - mn) : 0.f;
            if (lane < n) pw[h * kAttnTok + lane] = e;
            float sm = e;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
            if (lane == 0) {
                const float al = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
                s_alpha[h] = al;
                s_l[h] = s_l[h] * al + sm;
                s_m[h] = mn;
            }
        }
        __syncthreads();
        if (kv_t < Hkv) {
#pragma unroll
            for (int g = 0; g < G; ++g) acc[g] *= s_alpha[kv_t * G + g];
            for (int i = 0; i < n; ++i) {
                const float v = bf16_bits_to_float(__ldg(a.v_cache + (toks[i] * Hkv + kv_t) * kHeadDim + d_t));
#pragma unroll
                for (int g = 0; g < G; ++g) acc[g] = fmaf(pw[(kv_t * G + g) * kAttnTok + i], v, acc[g]);
            }
        }
        __syncthreads();
    }
    // partial of this CTA: m[Hq], l[Hq], acc[Hq][256]
    float *mypart = a.part + (size_t)blockIdx.x * Hq * (kHeadDim + 2);
    if (tid < Hq) {
        mypart[tid] = s_m[tid];
        mypart[Hq + tid] = s_l[tid];
    }
    if (kv_t < Hkv) {
#pragma unroll
        for (int g = 0; g < G; ++g) mypart[2 * Hq + (kv_t * G + g) * kHeadDim + d_t] = acc[g];
    }

    // ---- 7. merge the row's partials; each CTA finishes a slice of the Hq x 256 outputs
    const int r3 = row_arrive(rs, cr, a.hdr, row, &s_flag);
    if (r3 < 0) return;
    if (r3 == 1) row_release(rs);
    __syncthreads();
    const float *parts = a.part + (size_t)first * Hq * (kHeadDim + 2);
    const int stride = Hq * (kHeadDim + 2);
    const int n_out = Hq * kHeadDim;
    const int o_lo = n_out * jj / cr, o_hi = n_out * (jj + 1) / cr;
    const int h_lo = o_lo / kHeadDim, h_hi = (o_hi - 1) / kHeadDim;
    // per head in the slice: M = max m_j, weights w_j = 2^(m_j - M), L = sum l_j w_j
    float *w_s = reinterpret_cast<float *>(smem + kRingOff);              // [heads][cr]
    for (int h = h_lo; h <= h_hi && o_lo < o_hi; ++h) {
        float mx = -INFINITY;
        for (int j = tid; j < cr; j += kStepThreads) mx = fmaxf(mx, __ldcg(&parts[(size_t)j * stride + h]));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) reinterpret_cast<float *>(s_wsum)[warp] = mx;
        __syncthreads();
        float M = -INFINITY;
        for (int w = 0; w < kStepWarps; ++w) M = fmaxf(M, reinterpret_cast<float *>(s_wsum)[w]);
        __syncthreads();
        float lsum = 0.f;
        for (int j = tid; j < cr; j += kStepThreads) {
            const float mj = __ldcg(&parts[(size_t)j * stride + h]);
            const float wj = (mj == -INFINITY) ? 0.f : exp2f(mj - M);
            w_s[(h - h_lo) * cr + j] = wj;
            lsum = fmaf(__ldcg(&parts[(size_t)j * stride + Hq + h]), wj, lsum);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
        if (lane == 0) reinterpret_cast<float *>(s_wsum)[warp] = lsum;
        __syncthreads();
        if (tid == 0) {
            float L = 0.f;
            for (int w = 0; w < kStepWarps; ++w) L += reinterpret_cast<float *>(s_wsum)[w];
            s_m[h - h_lo] = M;
            s_l[h - h_lo] = L;
        }
        __syncthreads();
    }
    // outputs: `tpo` threads per output, each summing a strided subset of the partials
    const int n_my = o_hi - o_lo;
    int tpo = 1;
    while (tpo < 32 && (tpo * 2) * n_my <= kStepThreads) tpo *= 2;
    const int sub = tid % tpo;
    for (int o_base = 0; o_base < n_my; o_base += kStepThreads / tpo) {
        const int oi = o_base + tid / tpo;
        float s = 0.f;
        int o = 0, h = 0;
        if (oi < n_my) {
            o = o_lo + oi;
            h = o / kHeadDim;
            const int d = o % kHeadDim;
            const float *wv = w_s + (h - h_lo) * cr;
            for (int j = sub; j < cr; j += tpo) s = fmaf(__ldcg(&parts[(size_t)j * stride + 2 * Hq + h * kHeadDim + d]), wv[j], s);
        }
        for (int off = tpo >> 1; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (oi < n_my && sub == 0) {
            const float L = s_l[h - h_lo];
            a.out[(int64_t)row * n_out + o] = float_to_bf16_bits(s / L);
            if (a.lse != nullptr && (o % kHeadDim) == 0)
                a.lse[(int64_t)row * Hq + h] = (s_m[h - h_lo] + log2f(L)) * kLn2;
        }
    }
}

// ------------------------------------------------------------------------------ launcher

namespace {
int g_step_ctas[64][5];     // per device and per G (1,2,4,8,16): co-resident CTAs, 0 = unknown

int g_index(int G) { return G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : G == 8 ? 3 : 4; }

template <int G>
int step_ctas_g(int dev) {
    int &slot = g_step_ctas[dev][g_index(G)];
    if (slot == 0) {
        auto kern = decode_step_kernel<G>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStepSmem) != cudaSuccess)
            return 0;
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStepThreads, kStepSmem) != cudaSuccess)
            return 0;
        if (per_sm < 1) return 0;
        slot = min(sms * per_sm, kMaxStepCtas);
    }
    return slot;
}

template <int G>
cudaError_t launch_step_g(const StepArgs &a, int ctas, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = kStepSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_step_kernel<G>, a);
}
}  // namespace

size_t decode_step_ws_bytes(int B, int64_t max_blocks, int Hq) { return step_layout(B, max_blocks, Hq).total; }

int decode_step_max_keys() { return kMaxKeys; }

int decode_step_grid(int G) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    switch (G) {
        case 1: return step_ctas_g<1>(dev);
        case 2: return step_ctas_g<2>(dev);
        case 4: return step_ctas_g<4>(dev);
        case 8: return step_ctas_g<8>(dev);
        case 16: return step_ctas_g<16>(dev);
        default: return 0;
    }
}

cudaError_t launch_decode_step(StepArgs a, void *ws, cudaStream_t st) {
    const StepLayout L = step_layout(a.B, a.max_blocks, a.n_q_heads);
    char *w = static_cast<char *>(ws);
    a.hdr = reinterpret_cast<WsHeader *>(w);
    a.rows = reinterpret_cast<void *>(w + L.rows);
    a.hist = reinterpret_cast<uint32_t *>(w + L.hist);
    a.cands = reinterpret_cast<unsigned long long *>(w + L.cands);
    a.part = reinterpret_cast<float *>(w + L.part);
    const int G = a.n_q_heads / a.n_kv_heads;
    const int ctas = decode_step_grid(G);
    if (ctas < a.B || ctas == 0) return cudaErrorInvalidConfiguration;
    switch (G) {
        case 1: return launch_step_g<1>(a, ctas, st);
        case 2: return launch_step_g<2>(a, ctas, st);
        case 4: return launch_step_g<4>(a, ctas, st);
        case 8: return launch_step_g<8>(a, ctas, st);
        case 16: return launch_step_g<16>(a, ctas, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qsa
