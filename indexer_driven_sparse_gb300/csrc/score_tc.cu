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
// Products of bf16 values are exact in fp32; the tensor core sums them in fp32 in its own
// order. Every wait is bounded; a timeout records QSA_ERR_DEVICE_TIMEOUT and the roles
// drain what they issued before TMEM is freed.
#include "qsa_internal.cuh"
#include "qsa_ptx.cuh"
#include "qsa_tc.cuh"

#include <cuda.h>

#include <algorithm>

namespace qsa {

constexpr int kStThreads = 192;                             // TMA warp, MMA warp, 4 epilogue warps
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

    if (warp == 1) tmem_alloc(&tmem_s, 512);
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
            mbar_init(smem_u32(&tfull[s]), 1);
            mbar_init(smem_u32(&tempty[s]), 128);
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
    auto timeout = [&]() { record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereScore, blockIdx.x); };

    if (warp == 0) {
        if (lane == 0) {
            int i = 0;
            for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
                const int s = i & 1;
                if (i >= 2 && !mbar_wait_bounded(smem_u32(&empty[s]), ((i >> 1) - 1) & 1, kWaitLimitNs)) {
                    timeout();
                    break;
                }
                const int m = t % a.n_m, n = t / a.n_m;
                const uint32_t bar = smem_u32(&full[s]);
                const uint32_t da = sbase + s * kStStage, db = da + kStABytes;
                mbar_arrive_expect_tx(bar, kStStage);
                tma_load_2d(da, &tm_q, 0, m * kStM, bar);
                tma_load_2d(da + kStABytes / 2, &tm_q, 64, m * kStM, bar);
                tma_load_2d(db, &tm_p, 0, (int32_t)(off + (int64_t)n * kStN), bar);
                tma_load_2d(db + kStBBytes / 2, &tm_p, 64, (int32_t)(off + (int64_t)n * kStN), bar);
            }
            // no copy may still be writing shared memory when the CTA exits
            for (int j = std::max(0, i - 2); j < i; ++j)
                mbar_wait_bounded(smem_u32(&full[j & 1]), (j >> 1) & 1, kWaitLimitNs);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int i = 0;
            bool issued = false;
            for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
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
    } else {
        const int q4 = warp & 3;                      // the TMEM lane quarter this warp may access
        float *xp = reinterpret_cast<float *>(sm + kStXpose + (warp - 2) * kStWarpBuf);
        const uint32_t box0 = sbase + kStXpose + (warp - 2) * kStWarpBuf;   // two 4 KiB boxes
        int nbox = 0;                                 // boxes stored by this warp so far
        int i = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++i) {
            const int acc = i & 1;
            const int m = t % a.n_m, n = t / a.n_m;
            const bool got = mbar_wait_bounded(smem_u32(&tfull[acc]), (i >> 1) & 1, kWaitLimitNs);
            if (!__all_sync(0xffffffffu, got)) {      // TMEM loads below are warp-collective
                if (lane == 0) timeout();
                break;
            }
            tc_fence_after();
            const int row = m * kStM + q4 * 32 + lane;
            int nb = 0;
            if (row < a.Nq) {
                const int p = a.q_pos[row];
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

cudaError_t launch_score_tc(const uint16_t *q_idx, const int32_t *q_pos, int Nq, const uint16_t *pooled,
                            int64_t n_pooled, const int32_t *blk_off, float *scores, int64_t ld, WsHeader *hdr,
                            cudaStream_t st) {
    CUtensorMap tq, tp;
    if (!encode_tmap_bf16_2d(&tq, q_idx, kIdxDim, Nq, kIdxDim * 2, 64, kStM) ||
        !encode_tmap_bf16_2d(&tp, pooled, kIdxDim, n_pooled, kIdxDim * 2, 64, kStN))
        return cudaErrorInvalidValue;
    ScoreTcArgs a{};
    a.q_pos = q_pos;
    a.Nq = Nq;
    a.blk_off = blk_off;
    a.n_pooled = n_pooled;
    a.scores = scores;
    a.ld = ld;
    a.n_m = (Nq + kStM - 1) / kStM;
    a.n_n = (int)((ld + kStN - 1) / kStN);
    a.vec = ((uintptr_t)scores % 16 == 0 && ld % 4 == 0) ? 1 : 0;
    // the scores as [Nq rows of ld floats] in 32 x 32 boxes (needs 16-byte rows)
    CUtensorMap ts;
    memset(&ts, 0, sizeof(ts));
    a.tma_store = a.vec && encode_tmap_f32_2d(&ts, scores, (uint64_t)ld, (uint64_t)Nq, (uint64_t)ld * 4, 32, 32) ? 1 : 0;
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

}  // namespace qsa
