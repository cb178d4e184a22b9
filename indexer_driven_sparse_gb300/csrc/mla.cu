// Sparse MLA decode in its MQA form on the tensor cores ("GLM-5.3 最適化 第2部：16基のH200上
// でのPCP、DCP、およびHybrid HiSparse", footnote 1: a query reads 2,048 selected 656-byte FP8
// rows; QK runs over 576 dims and PV over 512; one row serves every head, which is what
// makes the contraction dense enough for tensor cores in decode).
//
// Row layout (656 B): the 512-dim latent as E4M3 codes, four fp32 scales (one per 128
// latent dims), the 64 rotary dims as bf16. Head h of a query attends its selected rows j:
//   logit = scale * (q_h[:512] . latent_j + q_h[512:] . rope_j),  out_h = sum_j softmax_j latent_j.
//
// mla_tile_kernel: one CTA per (tile of 64 selected rows, half of the latent dims, query).
//   - all warps gather the tile's rows: codes x scale -> bf16 (one rounding) and the bf16 rope
//     into a 128B-swizzled K-major tile [9 column blocks][64 rows][64 dims]; the query's heads
//     (up to 128 MMA rows, the rest zero) into a K-major tile of the same layout;
//   - warp 4 issues S = Q K^T (M 128, N 64, K 576) into tensor memory;
//   - warps 0-3 (one head row per thread) take the tile's softmax partial (max and sum in
//     log2 units) and write P (bf16 pairs) to tensor memory;
//   - warp 4 issues O = P V (M 128, N 256, K 64) with V = this CTA's 256 latent dims of the
//     same K tile read MN-major, A = P from tensor memory;
//   - warps 0-3 store the unnormalised O rows and (m, l) to the workspace.
// mla_merge_kernel: per (head, query), the tiles' partials merged by log-sum-exp (the LSE merge
// of "GLM-5.3 最適化 第2部", section DCP).
// Every mbarrier wait is bounded; a wait that gives up records QSA_ERR_DEVICE_TIMEOUT.
#include "qsa_internal.cuh"
#include "qsa_ptx.cuh"
#include "qsa_tc.cuh"

namespace qsa {

constexpr int kMlaRows = 128;                        // MMA M: head rows (H <= 128; the rest zero)
constexpr int kMlaTok = 64;                          // selected rows per tile: N of QK, K of PV
constexpr int kMlaLat = 512, kMlaRope = 64, kMlaDim = kMlaLat + kMlaRope;
constexpr int kMlaBlocks = kMlaDim / 64;             // 9 column blocks of 64 dims (128 B)
constexpr int kMlaRowBytes = 656;
constexpr int kMlaScaleOff = kMlaLat, kMlaRopeOff = kMlaLat + 16;
constexpr int kMlaThreads = 160;                     // warps 0-3 softmax / epilogue, warp 4 MMA
constexpr uint32_t kMlaQ = 0;                                           // 9 x 128 x 128 B
constexpr uint32_t kMlaK = kMlaBlocks * kMlaRows * 128;                 // 9 x 64 x 128 B
constexpr uint32_t kMlaSmem = kMlaK + kMlaBlocks * kMlaTok * 128 + 1024;   // + alignment slack
constexpr uint32_t kMlaTmS = 0, kMlaTmP = 64, kMlaTmO = 256;            // TMEM columns
constexpr int kWhereMla = 8;

struct MlaArgs {
    const uint16_t *q;        // [B][H][576]
    const uint8_t *kv;        // [n_tok][656]
    int64_t n_tok;
    const int32_t *rows;      // [B][max_rows]
    const int32_t *n_rows;    // [B]
    int32_t max_rows, H, B, n_tiles;
    float scale_log2;
    float *part_acc;          // [B][n_tiles][2][H][256]
    float *part_ml;           // [B][n_tiles][H][2]  (max and sum, log2 units)
    uint16_t *out;            // [B][H][512]
    float *lse;               // [B][H] or nullptr
    WsHeader *hdr;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ int mla_rows_of(const MlaArgs &a, int b) {
    const int n = a.n_rows[b];
    return n < 0 ? 0 : (n > a.max_rows ? a.max_rows : n);
}

__global__ void __launch_bounds__(kMlaThreads, 1) mla_tile_kernel(MlaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(sm);
    __shared__ uint64_t s_full, p_full, o_full;
    __shared__ uint32_t tmem_s;
    __shared__ float s_scale[kMlaTok][4];
    __shared__ int32_t s_row[kMlaTok];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t = blockIdx.x, hf = blockIdx.y, b = blockIdx.z;
    const int H = a.H;
    if (tid == 0 && a.n_rows[b] > a.max_rows && t == 0 && hf == 0)
        record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereMla, b);
    const int nr = mla_rows_of(a, b);
    const int j0 = t * kMlaTok;
    const int nv = nr - j0 < kMlaTok ? nr - j0 : kMlaTok;   // valid rows of this tile
    if (nv <= 0) return;                                      // the merge reads no partial of it

    if (warp == 4) tmem_alloc(&tmem_s, 512);
    if (tid == 0) {
        mbar_init(smem_u32(&s_full), 1);
        mbar_init(smem_u32(&p_full), kMlaRows);
        mbar_init(smem_u32(&o_full), 1);
        fence_mbar_init();
    }
    if (tid < kMlaTok) {
        int id = -1;
        if (tid < nv) {
            id = a.rows[(int64_t)b * a.max_rows + j0 + tid];
            if (id < 0 || id >= a.n_tok) {               // skip the row, record the error
                record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereMla, b);
                id = -1;
            }
        }
        s_row[tid] = id;
        float4 sc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (id >= 0) {
            const uint4 u = ldg_nc_v4(a.kv + (int64_t)id * kMlaRowBytes + kMlaScaleOff);
            sc = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
        }
        s_scale[tid][0] = sc.x;
        s_scale[tid][1] = sc.y;
        s_scale[tid][2] = sc.z;
        s_scale[tid][3] = sc.w;
    }
    // the query's heads, rows H..127 zero
    for (int i = tid; i < kMlaRows * kMlaBlocks * 8; i += kMlaThreads) {
        const int h = i / (kMlaBlocks * 8), rem = i - h * (kMlaBlocks * 8), blk = rem >> 3, g = rem & 7;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (h < H) v = ldg_nc_v4(a.q + ((int64_t)b * H + h) * kMlaDim + blk * 64 + g * 8);
        st_shared_v4(sbase + kMlaQ + blk * (kMlaRows * 128) + swz(h, g), v);
    }
    __syncthreads();                                           // s_row, s_scale
    // latent: 32 granules of 16 codes per row -> 2 bf16 granules each; padding rows zero
    for (int i = tid; i < kMlaTok * 32; i += kMlaThreads) {
        const int j = i >> 5, gi = i & 31;
        const int id = s_row[j];
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = 0u;
        if (id >= 0) {
            float f[16];
            e4m3x16_to_f32(ldg_nc_v4(a.kv + (int64_t)id * kMlaRowBytes + gi * 16), f);
            const float sc = s_scale[j][gi >> 3];
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(f[2 * e] * sc, f[2 * e + 1] * sc);
        }
        const uint32_t base = sbase + kMlaK + (gi >> 2) * (kMlaTok * 128);
        const int g0 = (gi & 3) * 2;
        st_shared_v4(base + swz(j, g0), make_uint4(w[0], w[1], w[2], w[3]));
        st_shared_v4(base + swz(j, g0 + 1), make_uint4(w[4], w[5], w[6], w[7]));
    }
    // rotary dims: column block 8, copied as they are
    for (int i = tid; i < kMlaTok * 8; i += kMlaThreads) {
        const int j = i >> 3, g = i & 7;
        const int id = s_row[j];
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (id >= 0) v = ldg_nc_v4(a.kv + (int64_t)id * kMlaRowBytes + kMlaRopeOff + g * 16);
        st_shared_v4(sbase + kMlaK + 8 * (kMlaTok * 128) + swz(j, g), v);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_s;

    if (warp == 4) {
        // ================================================================ MMA issue
        if (lane == 0) {
            const uint32_t qa = sbase + kMlaQ, kb = sbase + kMlaK;
#pragma unroll 1
            for (int ks = 0; ks < kMlaDim / 16; ++ks) {
                const uint64_t ad = tc_desc(qa + (ks >> 2) * (kMlaRows * 128) + (ks & 3) * 32, 16, 1024);
                const uint64_t bd = tc_desc(kb + (ks >> 2) * (kMlaTok * 128) + (ks & 3) * 32, 16, 1024);
                tc_mma(tmem + kMlaTmS, ad, bd, tc_idesc(kMlaRows, kMlaTok, 0), ks > 0);
            }
            tc_commit(smem_u32(&s_full));
            if (mbar_wait_bounded(smem_u32(&p_full), 0, kWaitLimitNs)) {
                tc_fence_after();
                // V: this CTA's four column blocks of the latent, read MN-major (16 rows per k-step)
                const uint32_t vb = kb + (uint32_t)(hf * 4) * (kMlaTok * 128);
#pragma unroll
                for (int ks = 0; ks < kMlaTok / 16; ++ks) {
                    const uint64_t bd = tc_desc(vb + ks * 2048, kMlaTok * 128, 1024);
                    tc_mma_ta(tmem + kMlaTmO, tmem + kMlaTmP + ks * 8, bd, tc_idesc(kMlaRows, 256, 1), ks > 0);
                }
                tc_commit(smem_u32(&o_full));
                mbar_wait_bounded(smem_u32(&o_full), 0, kWaitLimitNs);   // every MMA done before TMEM is freed
            } else {
                record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, b);
                mbar_wait_bounded(smem_u32(&s_full), 0, kWaitLimitNs);
            }
        }
        __syncwarp();
    } else {
        // ================================================================ softmax, epilogue
        const int row = tid;                                   // MMA row = TMEM lane = head
        const uint32_t t_row = tmem + ((uint32_t)(32 * warp) << 16);
        const bool got_s = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&s_full), 0, kWaitLimitNs));
        float m2 = -INFINITY, l = 0.f;
        if (got_s) {
            tc_fence_after();
            float s0[32], s1[32];
            tmem_ld32_async(t_row + kMlaTmS, s0);
            tmem_ld32_async(t_row + kMlaTmS + 32, s1);
            tmem_wait_ld(s0);
            tmem_wait_ld(s1);
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j < nv) mx = fmaxf(mx, s0[j]);
                if (j + 32 < nv) mx = fmaxf(mx, s1[j]);
            }
            m2 = mx * a.scale_log2;                            // nv >= 1: finite
            uint32_t pk[32];
            float ps = 0.f;
#pragma unroll
            for (int j = 0; j < 64; j += 2) {
                const float x0 = j < 32 ? s0[j] : s1[j - 32], x1 = j < 32 ? s0[j + 1] : s1[j - 31];
                const float e0 = j < nv ? ex2_approx(fmaf(x0, a.scale_log2, -m2)) : 0.f;
                const float e1 = j + 1 < nv ? ex2_approx(fmaf(x1, a.scale_log2, -m2)) : 0.f;
                ps += e0 + e1;
                pk[j >> 1] = pack_bf16x2(e0, e1);
            }
            l = ps;
            tmem_st32(t_row + kMlaTmP, pk);
        } else if (lane == 0) {
            record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, b);
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&p_full));
        const bool got_o = got_s && __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&o_full), 0, kWaitLimitNs));
        if (got_o) {
            tc_fence_after();
            float *acc = a.part_acc + ((((int64_t)b * a.n_tiles + t) * 2 + hf) * H + row) * 256;
#pragma unroll 1
            for (int c0 = 0; c0 < 256; c0 += 32) {
                float ov[32];
                tmem_ld32(t_row + kMlaTmO + c0, ov);           // warp-collective
                if (row < H) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<float4 *>(acc + c0 + 4 * k) =
                            make_float4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]);
                }
            }
            if (hf == 0 && row < H) {
                float *ml = a.part_ml + (((int64_t)b * a.n_tiles + t) * H + row) * 2;
                ml[0] = m2;
                ml[1] = l;
            }
        } else if (lane == 0 && got_s) {
            record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, b);
        }
        tc_fence_before();
    }
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Per (head, query): the tiles' partials merged by log-sum-exp; 256 threads, two dims each.
__global__ void __launch_bounds__(256) mla_merge_kernel(MlaArgs a) {
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int H = a.H;
    const int nt = (mla_rows_of(a, b) + kMlaTok - 1) / kMlaTok;
    const float *ml = a.part_ml + ((int64_t)b * a.n_tiles * H + h) * 2;
    float M = -INFINITY;
    for (int t = 0; t < nt; ++t) M = fmaxf(M, ml[(int64_t)t * H * 2]);
    float L = 0.f, o0 = 0.f, o1 = 0.f;
    for (int t = 0; t < nt; ++t) {
        const float m = ml[(int64_t)t * H * 2], lt = ml[(int64_t)t * H * 2 + 1];
        if (m == -INFINITY) continue;
        const float w = exp2f(m - M);
        L += lt * w;
        const float *acc = a.part_acc + (((int64_t)b * a.n_tiles + t) * 2 * H + h) * 256;
        o0 += w * acc[tid];
        o1 += w * acc[(int64_t)H * 256 + tid];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint16_t *dst = a.out + ((int64_t)b * H + h) * kMlaLat;
    dst[tid] = float_to_bf16_bits(o0 * inv);
    dst[256 + tid] = float_to_bf16_bits(o1 * inv);
    if (tid == 0 && a.lse != nullptr) a.lse[(int64_t)b * H + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

size_t mla_scratch_bytes(int H, int B, int max_rows) {
    const int64_t nt = (max_rows + kMlaTok - 1) / kMlaTok;
    return (size_t)B * nt * 2 * H * 256 * 4 + (size_t)B * nt * H * 2 * 4 + 256;
}

namespace {
bool g_mla_attr[64];
}

cudaError_t launch_sparse_mla(const uint16_t *q, int H, const uint8_t *kv, int64_t n_tok, const int32_t *rows,
                              const int32_t *n_rows, int max_rows, int B, float scale, uint16_t *out, float *lse,
                              WsHeader *hdr, void *scratch, cudaStream_t st) {
    if (B == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!g_mla_attr[dev]) {
        e = cudaFuncSetAttribute(mla_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMlaSmem);
        if (e != cudaSuccess) return e;
        g_mla_attr[dev] = true;
    }
    MlaArgs a{};
    a.q = q;
    a.kv = kv;
    a.n_tok = n_tok;
    a.rows = rows;
    a.n_rows = n_rows;
    a.max_rows = max_rows;
    a.H = H;
    a.B = B;
    a.n_tiles = (max_rows + kMlaTok - 1) / kMlaTok;
    a.scale_log2 = scale * kLog2e;
    a.part_acc = static_cast<float *>(scratch);
    a.part_ml = a.part_acc + (size_t)B * a.n_tiles * 2 * H * 256;
    a.out = out;
    a.lse = lse;
    a.hdr = hdr;
    if (a.n_tiles > 0) {
        mla_tile_kernel<<<dim3(a.n_tiles, 2, B), kMlaThreads, kMlaSmem, st>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    mla_merge_kernel<<<dim3(H, B), 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa
