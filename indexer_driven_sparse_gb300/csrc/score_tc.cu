// a2 for a prefill chunk — the indexer scores of many queries of ONE sequence against its
// pooled keys, as a GEMM on the 5th-generation tensor cores.
//
// "GLM-5.3 最適化 第2部" (the indexer part of prefill): scoring is quadratic in the prefill
// length and can cost more than the attention; "3090x3で 314 万コンテキスト", section
// "なぜ": every query scores every complete pooled block before it. Here the chunk's
// queries share one pooled-key history, so S = Q_idx * P^T is a dense contraction
// (K = 128) and runs as tcgen05 MMAs:
//   tile = 128 queries x 256 pooled blocks, fp32 accumulator in TMEM (two accumulators,
//   so the epilogue of one tile overlaps the MMAs of the next);
//   warp 0: TMA loads of the Q and pooled-key tiles (128B swizzle) into a 2-stage ring;
//   warp 1: one thread issues the 8 MMAs (K = 16 each) of a tile and commits them;
//   warps 2-5: read the accumulator (one row per thread), transpose 32x32 through shared
//   memory, and store rows with coalesced 128-byte writes, only columns b < nb(p_row).
// For the fused prefill selection the same GEMM runs with two other epilogues: per row the
// maximum of every 64 visible blocks, or every visible score at or above the row's floor as
// a 64-bit key in per-(row, half tile) slots (8 epilogue warps then, two per lane quarter).
// Each CTA takes a contiguous run of tiles, queries fastest, so a stage keeps its pooled-key
// tile while the query tiles change.
// Products of bf16 values are exact in fp32; the tensor core sums them in fp32 in its own
// order. Every wait is bounded; a timeout records QSA_ERR_DEVICE_TIMEOUT and the roles
// drain what they issued before TMEM is freed.
#include "qsa_internal.cuh"
#include "qsa_ptx.cuh"
#include "qsa_tc.cuh"

#include <cuda.h>

#include <algorithm>

namespace qsa {

constexpr int kStThreads = 320;                             // TMA warp, MMA warp, 8 epilogue warps
// (scores: 4 epilogue warps take whole tiles; selection passes: 8, two per TMEM lane quarter,
// each taking half of a tile's columns)
constexpr int kStM = 128, kStN = 256;
constexpr uint32_t kStABytes = kStM * kIdxDim * 2;          // 32 KiB: two 64-column swizzled halves
constexpr uint32_t kStBBytes = kStN * kIdxDim * 2;          // 64 KiB
constexpr uint32_t kStStage = kStABytes + kStBBytes;
constexpr int kStXStride = 36;                              // floats per transposed row (16-byte aligned)
constexpr uint32_t kStXpose = 2 * kStStage;                 // per epilogue warp: two 32 x 32-float boxes
constexpr uint32_t kStWarpBuf = 2 * 32 * 32 * 4;            // (or one 32 x 36-float transpose)
static_assert(32 * kStXStride * 4 <= kStWarpBuf, "transpose fits the warp's boxes");
constexpr uint32_t kStSmem = kStXpose + 4 * kStWarpBuf + 1024;
static_assert(kStSmem + 1024 <= 227 * 1024, "shared memory per CTA (dynamic + static)");

struct ScoreTcArgs {
    const int32_t *q_pos;
    int32_t Nq;
    const int32_t *blk_off;
    int64_t n_pooled;
    float *scores;
    int64_t ld;
    int32_t n_m, n_n;
    int32_t vec;              // rows 16-byte aligned (scores aligned, ld % 4 == 0): 16-byte stores
    int32_t tma_store;        // whole 32 x 32 slices leave through the tensor map of the scores
    WsHeader *hdr;
    int32_t mode;             // 0: store the scores; 1: maxima of 64 blocks; 2: candidates >= thr
    float *gmax;              // mode 1: [Nq][n_n * 4]
    const float *thr;         // mode 2: [Nq]
    uint64_t *slots;          // mode 2: [Nq][n_n][2][kSelSlots] (two halves of a tile)
    uint8_t *scnt;            // mode 2: [Nq][n_n][2]
    const int32_t *guard;     // non-null: the launch runs only when *guard != 0
};

__global__ void __launch_bounds__(kStThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_p,
                    const __grid_constant__ CUtensorMap tm_s, ScoreTcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(sm);
    __shared__ uint64_t full[2], empty[2], tfull[2], tempty[2];
    __shared__ uint32_t tmem_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (a.guard != nullptr && __ldcg(a.guard) == 0) return;   // nothing asked for this pass

    if (warp == 1) tmem_alloc(&tmem_s, 512);
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
            mbar_init(smem_u32(&tfull[s]), 1);
            mbar_init(smem_u32(&tempty[s]), (a.mode == 0 ? 4 : 8) * 32);
        }
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_p);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_s;
    const int64_t off = a.blk_off[0];                 // the sequence's first pooled block
    const bool off_ok = off >= 0 && off <= a.n_pooled;
    if (!off_ok && tid == 0) record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereScore, 0);
    const int n_tiles = off_ok ? a.n_m * a.n_n : 0;
    // a contiguous run of tiles per CTA, queries fastest: consecutive tiles share their pooled
    // block tile, which then stays in shared memory instead of being loaded again
    const int t_begin = (int)((int64_t)n_tiles * blockIdx.x / gridDim.x);
    const int t_end = (int)((int64_t)n_tiles * (blockIdx.x + 1) / gridDim.x);
    auto timeout = [&]() { record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereScore, blockIdx.x); };

    if (warp == 0) {
        if (lane == 0) {
            int i = 0;
            int stage_n[2] = {-1, -1};              // pooled tile held by each stage
            for (int t = t_begin; t < t_end; ++t, ++i) {
                const int s = i & 1;
                if (i >= 2 && !mbar_wait_bounded(smem_u32(&empty[s]), ((i >> 1) - 1) & 1, kWaitLimitNs)) {
                    timeout();
                    break;
                }
                const int m = t % a.n_m, n = t / a.n_m;
                const uint32_t bar = smem_u32(&full[s]);
                const uint32_t da = sbase + s * kStStage, db = da + kStABytes;
                const bool keep_p = stage_n[s] == n;    // this stage already holds the pooled tile
                mbar_arrive_expect_tx(bar, keep_p ? kStABytes : kStStage);
                tma_load_2d(da, &tm_q, 0, m * kStM, bar);
                tma_load_2d(da + kStABytes / 2, &tm_q, 64, m * kStM, bar);
                if (!keep_p) {
                    tma_load_2d(db, &tm_p, 0, (int32_t)(off + (int64_t)n * kStN), bar);
                    tma_load_2d(db + kStBBytes / 2, &tm_p, 64, (int32_t)(off + (int64_t)n * kStN), bar);
                    stage_n[s] = n;
                }
            }
            // no copy may still be writing shared memory when the CTA exits
            for (int j = std::max(0, i - 2); j < i; ++j)
                mbar_wait_bounded(smem_u32(&full[j & 1]), (j >> 1) & 1, kWaitLimitNs);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int i = 0;
            bool issued = false;
            for (int t = t_begin; t < t_end; ++t, ++i) {
                const int s = i & 1, acc = i & 1;
                if (!mbar_wait_bounded(smem_u32(&full[s]), (i >> 1) & 1, kWaitLimitNs) ||
                    (i >= 2 && !mbar_wait_bounded(smem_u32(&tempty[acc]), ((i >> 1) - 1) & 1, kWaitLimitNs))) {
                    timeout();
                    break;
                }
                tc_fence_after();
                const uint32_t aa = sbase + s * kStStage, ab = aa + kStABytes;
#pragma unroll
                for (int ks = 0; ks < kIdxDim / 16; ++ks) {
                    const uint64_t ad = tc_desc(aa + (ks >> 2) * (kStABytes / 2) + (ks & 3) * 32, 16, 1024);
                    const uint64_t bd = tc_desc(ab + (ks >> 2) * (kStBBytes / 2) + (ks & 3) * 32, 16, 1024);
                    tc_mma(tmem + acc * kStN, ad, bd, tc_idesc(kStM, kStN, 0), ks > 0);
                }
                tc_commit(smem_u32(&empty[s]));
                tc_commit(smem_u32(&tfull[acc]));
                issued = true;
            }
            // the last commit covers every MMA issued: wait for it before TMEM is freed
            if (issued) mbar_wait_bounded(smem_u32(&tfull[(i - 1) & 1]), ((i - 1) >> 1) & 1, kWaitLimitNs);
        }
    } else if (warp - 2 < (a.mode == 0 ? 4 : 8)) {
        const int ew = warp - 2;                      // epilogue warp
        const int q4 = warp & 3;                      // the TMEM lane quarter this warp may access
        const int half = ew >> 2;                     // selection passes: slices [4 half, 4 half + 4)
        float *xp = reinterpret_cast<float *>(sm + kStXpose + (ew & 3) * kStWarpBuf);
        const uint32_t box0 = sbase + kStXpose + (ew & 3) * kStWarpBuf;   // two 4 KiB boxes
        float *xs = reinterpret_cast<float *>(sm + kStXpose) + ew * 1024;  // selection: 32 x 32, swizzled
        int nbox = 0;                                 // boxes stored by this warp so far
        // the row's position (and floor) are read one tile ahead, off the tile's critical path
        auto row_of = [&](int t) { return (t % a.n_m) * kStM + q4 * 32 + lane; };
        int p_nx = 0;
        float T_nx = 0.f;
        auto fetch = [&](int t) {
            const int r = row_of(t);
            p_nx = r < a.Nq ? __ldg(a.q_pos + r) : 0;
            T_nx = (a.mode == 2 && r < a.Nq) ? __ldg(a.thr + r) : 0.f;
        };
        if (t_begin < t_end) fetch(t_begin);
        int i = 0;
        for (int t = t_begin; t < t_end; ++t, ++i) {
            const int acc = i & 1;
            const int m = t % a.n_m, n = t / a.n_m;
            const int p_row = p_nx;
            const float T_row = T_nx;
            if (t + 1 < t_end) fetch(t + 1);
            const bool got = mbar_wait_bounded(smem_u32(&tfull[acc]), (i >> 1) & 1, kWaitLimitNs);
            if (!__all_sync(0xffffffffu, got)) {      // TMEM loads below are warp-collective
                if (lane == 0) timeout();
                break;
            }
            tc_fence_after();
            const int row = m * kStM + q4 * 32 + lane;
            int nb = 0;
            if (row < a.Nq) {
                const int p = p_row;
                const int64_t want = p >= 0 ? (p >> 2) : -1;
                if (want < 0 || want > a.ld || off + want > a.n_pooled) {
                    if (n == 0) record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereScore, row);
                } else {
                    nb = (int)want;
                }
            }
            const int64_t col0 = (int64_t)n * kStN;
            const int row0 = m * kStM + q4 * 32;
            const int nb_max = __reduce_max_sync(0xffffffffu, (unsigned)nb);
            // rows past the queries are clipped by the tensor map; they do not limit the slices
            const int nb_min = __reduce_min_sync(0xffffffffu, row < a.Nq ? (unsigned)nb : 0x7fffffffu);
            if (a.mode != 0) {
                // selection passes: the row's 64-block maxima, or its scores at or above the floor
                // as 64-bit keys (score key, then the lower block id first) in the tile's slots
                const float T = T_row;
                uint64_t *slot = a.mode == 2 ? a.slots + (((size_t)row * a.n_n + n) * 2 + half) * kSelSlots : nullptr;
                float gm = -INFINITY;
                uint32_t k = 0;
                auto process = [&](const float (&v)[32], int c) {
                    const int64_t cb = col0 + c * 32;
                    const int lim = (int)(nb - cb < 0 ? 0 : (nb - cb > 32 ? 32 : nb - cb));   // visible columns
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                    if (lim == 32) {                        // the common case: the whole slice is visible
#pragma unroll
                        for (int j = 0; j < 32; ++j) m4[j & 3] = fmaxf(m4[j & 3], v[j]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) m4[j & 3] = fmaxf(m4[j & 3], j < lim ? v[j] : -INFINITY);
                    }
                    const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                    if (a.mode == 1) {
                        gm = (c & 1) ? fmaxf(gm, mx) : mx;
                        if ((c & 1) && row < a.Nq) a.gmax[(size_t)row * (a.n_n * 4) + n * 4 + (c >> 1)] = gm;
                        return;
                    }
                    uint32_t msk = 0;
                    if (mx >= T) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) msk |= v[j] >= T ? (1u << j) : 0u;
                        if (lim < 32) msk &= (1u << lim) - 1u;   // lim < 32 here: the visible columns only
                    }
                    if (msk != 0u) {
                        // this row's values through its own row of shared memory (16-byte granules
                        // XOR-swizzled by row), so the set bits pick them by index
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            *reinterpret_cast<float4 *>(xs + lane * 32 + 4 * (q ^ (lane & 7))) =
                                make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                        for (; msk != 0u; msk &= msk - 1u) {
                            const int jj = __ffs(msk) - 1;
                            if (k < (uint32_t)kSelSlots)
                                slot[k] = ((uint64_t)score_key(xs[lane * 32 + 4 * ((jj >> 2) ^ (lane & 7)) + (jj & 3)])
                                           << 32) |
                                          (uint64_t)(0xFFFFFFFFu - (uint32_t)(cb + jj));
                            ++k;
                        }
                    }
                };
                // slices two at a time: the next slice's TMEM load is in flight while one is processed
                const uint32_t t_base = tmem + acc * kStN + ((uint32_t)(q4 * 32) << 16);
                const int c_lo = half * 4, c_hi = c_lo + 4;
                float va[32], vb[32];
                tmem_ld32_async(t_base + c_lo * 32, va);
                tmem_wait_ld(va);
#pragma unroll 1
                for (int c = c_lo; c < c_hi; c += 2) {
                    tmem_ld32_async(t_base + (c + 1) * 32, vb);
                    process(va, c);
                    tmem_wait_ld(vb);
                    if (c + 2 < c_hi) tmem_ld32_async(t_base + (c + 2) * 32, va);
                    process(vb, c + 1);
                    tmem_wait_ld(va);
                }
                if (a.mode == 2 && row < a.Nq) a.scnt[((size_t)row * a.n_n + n) * 2 + half] = (uint8_t)min(k, 255u);
                tc_fence_before();
                mbar_arrive(smem_u32(&tempty[acc]));
                continue;
            }
            // store passes: 4 rows x 32 columns per instruction, lane -> (row, 4 columns)
            const int sub_r = lane >> 3, sub_c = (lane & 7) * 4;
#pragma unroll 1
            for (int c = 0; c < kStN / 32; ++c) {
                float v[32];
                tmem_ld32(tmem + acc * kStN + ((uint32_t)(q4 * 32) << 16) + c * 32, v);
                if (col0 + c * 32 >= nb_max) continue;   // warp-uniform: nothing of this slice is kept
                if (a.tma_store && col0 + c * 32 + 32 <= nb_min) {
                    // the whole slice is kept: a 128B-swizzled 32 x 32 box, stored by the TMA engine
                    const uint32_t box = box0 + (uint32_t)(nbox & 1) * 4096u;
                    if (lane == 0 && nbox >= 2) bulk_wait_read<1>();   // this box's previous store has read it
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(box + lane * 128 + ((q ^ (lane & 7)) << 4)),
                                     "f"(v[4 * q]), "f"(v[4 * q + 1]), "f"(v[4 * q + 2]), "f"(v[4 * q + 3])
                                     : "memory");
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tm_s, (int32_t)(col0 + c * 32), row0, box);
                        bulk_commit_group();
                    }
                    ++nbox;
                    continue;
                }
                if (nbox > 0) {                          // the transpose overwrites both boxes
                    if (lane == 0) bulk_wait_read<0>();
                    __syncwarp();
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<float4 *>(xp + lane * kStXStride + 4 * q) =
                        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                __syncwarp();
                const int64_t col = col0 + c * 32 + sub_c;
#pragma unroll
                for (int pass = 0; pass < 8; ++pass) {
                    const int rl = pass * 4 + sub_r;
                    const int nb_r = __shfl_sync(0xffffffffu, nb, rl);
                    const float4 val = *reinterpret_cast<const float4 *>(xp + rl * kStXStride + sub_c);
                    float *dst = a.scores + (int64_t)(row0 + rl) * a.ld + col;
                    if (a.vec && col + 4 <= nb_r) {
                        *reinterpret_cast<float4 *>(dst) = val;
                    } else {
                        if (col < nb_r) dst[0] = val.x;
                        if (col + 1 < nb_r) dst[1] = val.y;
                        if (col + 2 < nb_r) dst[2] = val.z;
                        if (col + 3 < nb_r) dst[3] = val.w;
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&tempty[acc]));
        }
        if (lane == 0 && nbox > 0) bulk_wait_all();   // no store may still read shared memory at exit
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ----------------------------------------------------------------------------- host side

// 2-D tensor maps (rows of `inner` elements, `row_bytes` apart), 128B swizzle
static bool encode_tmap_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t rows,
                           uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
    using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                       const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                       CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                       CUtensorMapFloatOOBfill);
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    if (fn == nullptr || rows == 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_bf16_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                         uint32_t box_inner, uint32_t box_rows) {
    return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, inner, rows, row_bytes, box_inner, box_rows);
}

bool encode_tmap_f32_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                        uint32_t box_inner, uint32_t box_rows) {
    return encode_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, inner, rows, row_bytes, box_inner, box_rows);
}

bool score_tc_supported(int Nq, int64_t n_pooled) {
    return Nq >= kStM && n_pooled >= kStN && n_pooled < ((int64_t)1 << 31) - kStN;
}

// One CTA per row: the floor T = the 512th largest of the row's 64-block maxima (radix
// select on the order-preserving keys, 8 bits a pass). At least 512 visible scores reach T.
// Rows with fewer than 512 groups get -inf: every visible score is a candidate.
__global__ void __launch_bounds__(256) select_floor_kernel(const float *__restrict__ gmax, int gstride,
                                                           const int32_t *__restrict__ q_pos, int64_t ld,
                                                           float *__restrict__ thr) {
    __shared__ uint32_t keys[kSelMaxTiles * 4];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_prefix, s_need;
    const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
    const int p = q_pos[row];
    const int64_t nb = p >= 0 ? min((int64_t)(p >> 2), ld) : 0;
    const int64_t ng_all = (nb + kSelGroup - 1) / kSelGroup;
    const int ng = (int)(ng_all < (int64_t)gstride ? ng_all : (int64_t)gstride);
    if (ng < kBlockTopK) {
        if (tid == 0) thr[row] = -INFINITY;
        return;
    }
    for (int g = tid; g < ng; g += blockDim.x) keys[g] = score_key(__ldcg(gmax + (size_t)row * gstride + g));
    if (tid == 0) {
        s_prefix = 0u;
        s_need = kBlockTopK;
    }
    for (int shift = 24; shift >= 0; shift -= 8) {
        hist[tid] = 0u;
        __syncthreads();
        const uint32_t prefix = s_prefix, mask = shift == 24 ? 0u : ~0u << (shift + 8);
        for (int g = tid; g < ng; g += blockDim.x) {
            const uint32_t key = keys[g];
            if ((key & mask) == (prefix & mask)) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 32) {                         // the digit holding the need-th largest, from the top
            uint32_t c[8], sum = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                c[k] = hist[255 - (lane * 8 + k)];
                sum += c[k];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t need = s_need;
            uint32_t above = incl - sum;       // keys in higher digits than this lane's first
            const bool here = above < need && incl >= need;
            const unsigned who = __ballot_sync(0xffffffffu, here);
            if (lane == __ffs(who) - 1) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (above + c[k] >= need) {
                        s_prefix = prefix | ((uint32_t)(255 - (lane * 8 + k)) << shift);
                        s_need = need - above;
                        break;
                    }
                    above += c[k];
                }
            }
        }
        __syncthreads();
    }
    if (tid == 0) {
        const uint32_t k = s_prefix;             // the key of the 512th largest maximum
        thr[row] = k == 0u ? __int_as_float(0x7fc00000) : __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
    }
}

static cudaError_t launch_score_tc_mode(const uint16_t *q_idx, const int32_t *q_pos, int Nq, const uint16_t *pooled,
                                        int64_t n_pooled, const int32_t *blk_off, float *scores, int64_t ld,
                                        WsHeader *hdr, const ScoreTcArgs &mode_args, cudaStream_t st) {
    CUtensorMap tq, tp;
    if (!encode_tmap_bf16_2d(&tq, q_idx, kIdxDim, Nq, kIdxDim * 2, 64, kStM) ||
        !encode_tmap_bf16_2d(&tp, pooled, kIdxDim, n_pooled, kIdxDim * 2, 64, kStN))
        return cudaErrorInvalidValue;
    ScoreTcArgs a = mode_args;
    a.q_pos = q_pos;
    a.Nq = Nq;
    a.blk_off = blk_off;
    a.n_pooled = n_pooled;
    a.scores = scores;
    a.ld = ld;
    a.n_m = (Nq + kStM - 1) / kStM;
    a.n_n = (int)((ld + kStN - 1) / kStN);
    a.vec = (scores != nullptr && (uintptr_t)scores % 16 == 0 && ld % 4 == 0) ? 1 : 0;
    // the scores as [Nq rows of ld floats] in 32 x 32 boxes (needs 16-byte rows)
    CUtensorMap ts;
    memset(&ts, 0, sizeof(ts));
    a.tma_store = a.mode == 0 && a.vec &&
                          encode_tmap_f32_2d(&ts, scores, (uint64_t)ld, (uint64_t)Nq, (uint64_t)ld * 4, 32, 32)
                      ? 1
                      : 0;
    a.hdr = hdr;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t n_tiles = (int64_t)a.n_m * a.n_n;
    if (n_tiles > INT32_MAX) return cudaErrorInvalidValue;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, n_tiles));
    e = cudaFuncSetAttribute(score_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStSmem);
    if (e != cudaSuccess) return e;
    score_tc_kernel<<<grid, kStThreads, kStSmem, st>>>(tq, tp, ts, a);
    return cudaGetLastError();
}

cudaError_t launch_score_tc(const uint16_t *q_idx, const int32_t *q_pos, int Nq, const uint16_t *pooled,
                            int64_t n_pooled, const int32_t *blk_off, float *scores, int64_t ld, WsHeader *hdr,
                            cudaStream_t st) {
    return launch_score_tc_mode(q_idx, q_pos, Nq, pooled, n_pooled, blk_off, scores, ld, hdr, ScoreTcArgs{}, st);
}

static size_t al256(size_t b) { return (b + 255) / 256 * 256; }

// scratch: maxima [Nq][4 n_n] f32, floors [Nq] f32, slots [Nq][2 n_n][kSelSlots] u64,
// counts [Nq][2 n_n] u8, fallback rows [Nq] i32, fallback flag
size_t prefill_select_scratch_bytes(int Nq, int64_t ld) {
    const size_t n_n = (size_t)((ld + kStN - 1) / kStN);
    return al256((size_t)Nq * n_n * 4 * 4) + al256((size_t)Nq * 4) + al256((size_t)Nq * n_n * 2 * kSelSlots * 8) +
           al256((size_t)Nq * n_n * 2) + al256((size_t)Nq * 4) + 256;
}

bool prefill_select_supported(int Nq, int64_t n_pooled, int64_t ld) {
    return score_tc_supported(Nq, n_pooled) && (ld + kStN - 1) / kStN <= kSelMaxTiles;
}

cudaError_t launch_prefill_select(const uint16_t *q_idx, const int32_t *q_pos, int Nq, const uint16_t *pooled,
                                  int64_t n_pooled, const int32_t *blk_off, float *scores, int64_t ld, int32_t *blocks,
                                  int32_t *count, WsHeader *hdr, void *scratch, size_t scratch_bytes, cudaStream_t st) {
    if (Nq == 0) return cudaSuccess;
    if (scratch_bytes < prefill_select_scratch_bytes(Nq, ld)) return cudaErrorInvalidValue;
    const int n_n = (int)((ld + kStN - 1) / kStN);
    char *w = static_cast<char *>(scratch);
    float *gmax = reinterpret_cast<float *>(w);
    w += al256((size_t)Nq * n_n * 4 * 4);
    float *thr = reinterpret_cast<float *>(w);
    w += al256((size_t)Nq * 4);
    uint64_t *slots = reinterpret_cast<uint64_t *>(w);
    w += al256((size_t)Nq * n_n * 2 * kSelSlots * 8);
    uint8_t *scnt = reinterpret_cast<uint8_t *>(w);
    w += al256((size_t)Nq * n_n * 2);
    int32_t *fb_rows = reinterpret_cast<int32_t *>(w);
    w += al256((size_t)Nq * 4);
    int32_t *fb_any = reinterpret_cast<int32_t *>(w);
    cudaError_t e = cudaMemsetAsync(fb_rows, 0, al256((size_t)Nq * 4) + 4, st);
    if (e != cudaSuccess) return e;
    ScoreTcArgs m{};
    m.mode = 1;
    m.gmax = gmax;
    e = launch_score_tc_mode(q_idx, q_pos, Nq, pooled, n_pooled, blk_off, nullptr, ld, hdr, m, st);
    if (e != cudaSuccess) return e;
    select_floor_kernel<<<Nq, 256, 0, st>>>(gmax, n_n * 4, q_pos, ld, thr);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    m = ScoreTcArgs{};
    m.mode = 2;
    m.thr = thr;
    m.slots = slots;
    m.scnt = scnt;
    e = launch_score_tc_mode(q_idx, q_pos, Nq, pooled, n_pooled, blk_off, nullptr, ld, hdr, m, st);
    if (e != cudaSuccess) return e;
    TopkCandidates tc;
    tc.slots = slots;
    tc.scnt = scnt;
    tc.n_segs = 2 * n_n;
    tc.fb_rows = fb_rows;
    tc.fb_any = fb_any;
    e = launch_topk_with(nullptr, ld, q_pos, Nq, blocks, count, hdr, tc, st);
    if (e != cudaSuccess) return e;
    // the exact path for the rows left over (both launches return at once when there are none)
    m = ScoreTcArgs{};
    m.guard = fb_any;
    e = launch_score_tc_mode(q_idx, q_pos, Nq, pooled, n_pooled, blk_off, scores, ld, hdr, m, st);
    if (e != cudaSuccess) return e;
    TopkCandidates fb;
    fb.fb_rows = fb_rows;
    fb.fallback_only = 1;
    return launch_topk_with(scores, ld, q_pos, Nq, blocks, count, hdr, fb, st);
}

}  // namespace qsa
