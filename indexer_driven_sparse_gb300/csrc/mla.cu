// Sparse MLA decode in its MQA form on the tensor cores ("GLM-5.3 最適化 第2部：16基のH200上
// でのPCP、DCP、およびHybrid HiSparse", footnote 1: a query reads 2,048 selected 656-byte FP8
// rows; QK runs over 576 dims and PV over 512; one row serves every head, which is what
// makes the contraction dense enough for tensor cores in decode).
//
// Row layout (656 B): the 512-dim latent as E4M3 codes, four fp32 scales (one per 128
// latent dims), the 64 rotary dims as bf16. Head h of a query attends its selected rows j:
//   logit = scale * (q_h[:512] . latent_j + q_h[512:] . rope_j),  out_h = sum_j softmax_j latent_j.
//
// mla_tile_kernel, persistent: the work is every (query, latent half, tile of 64 selected rows)
// in that order; CTA c takes the contiguous run [W c / G, W (c + 1) / G) of it, so the CTAs
// carry equal shares. Within a run, the tiles of one (query, half) form a segment whose output
// accumulates in tensor memory with an online softmax; a segment ends with one partial
// (unnormalised O rows and their (max, sum)) for the merge.
// Per tile:
//   - all 8 warps store the tile's rows, loaded into registers while the previous tile was
//     computed, into a 128B-swizzled K-major tile [9 column blocks][64 rows][64 dims]: codes x
//     scale rounded once to bf16, the rotary dims as they are; rows past the query's count or
//     with an id outside the cache are zero and masked. Then they issue the next tile's loads
//     (row ids one tile further ahead) before the tile is computed;
//   - warp 4 issues S = Q K^T (M 128: the heads, the rest zero; N 64; K 576) into tensor memory;
//   - warps 0-3 (one head row per thread) take the tile's softmax in log2 units against the
//     segment's running max, which is raised (and O rescaled) only when a tile's max exceeds it
//     by more than 2^8, and write P as bf16 pairs to tensor memory;
//   - warp 4 issues O += P V (M 128, N 256, K 64): V is this half's 256 latent dims of the same
//     tile read MN-major, A = P from tensor memory.
// mla_merge_kernel: per (head, query), each half's segment partials merged by log-sum-exp (the
// LSE merge of "GLM-5.3 最適化 第2部", section DCP).
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
constexpr int kMlaThreads = 256;                     // warps 0-3 softmax / epilogue, warp 4 MMA; all gather
constexpr int kMlaWarps = kMlaThreads / 32;
constexpr int kMlaLatItems = kMlaTok * 32 / kMlaThreads;     // 16-code granules per thread per tile (8)
constexpr int kMlaRopeItems = kMlaTok * 8 / kMlaThreads;     // rotary granules per thread per tile (2)
constexpr uint32_t kMlaQ = 0;                                           // 9 x 128 x 128 B
constexpr uint32_t kMlaK = kMlaBlocks * kMlaRows * 128;                 // 9 x 64 x 128 B
constexpr uint32_t kMlaSmem = kMlaK + kMlaBlocks * kMlaTok * 128 + 1024;   // + alignment slack
constexpr uint32_t kMlaTmS = 0, kMlaTmP = 64, kMlaTmO = 256;            // TMEM columns
constexpr int kMlaMaxCtas = 256;                     // persistent grid bound (sizes the partials)
constexpr float kMlaRescale = 8.f;                   // raise the running max past 2^8 growth
constexpr int kWhereMla = 8;

struct MlaArgs {
    const uint16_t *q;        // [B][H][576]
    const uint8_t *kv;        // [n_tok][656]
    int64_t n_tok;
    const int32_t *rows;      // [B][max_rows]
    const int32_t *n_rows;    // [B]
    int32_t max_rows, H, B, n_tiles, grid;
    float scale_log2;
    float *part_acc;          // [grid + 2B][H][256] unnormalised O rows of a segment
    float *part_ml;           // [grid + 2B][H][2]   (max, sum) in log2 units
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

// First work item >= w (below w_hi) whose tile holds rows of its query; else w_hi.
__device__ __forceinline__ int64_t mla_next_item(const MlaArgs &a, int64_t w, int64_t w_hi) {
    while (w < w_hi) {
        const int64_t P = w / a.n_tiles;
        const int t = (int)(w - P * a.n_tiles);
        if (t * kMlaTok < mla_rows_of(a, (int)(P >> 1))) return w;
        w = (P + 1) * a.n_tiles;
    }
    return w_hi;
}

// Work range of CTA c: [W c / G, W (c + 1) / G) with W = B x 2 x n_tiles.
__device__ __forceinline__ int64_t mla_range_lo(const MlaArgs &a, int c) {
    return (int64_t)a.B * 2 * a.n_tiles * c / a.grid;
}

constexpr int kMlaNoRow = INT32_MIN;                 // tile row past the query's rows

// The raw row id of tile row j of item (b, t) (no check yet), or kMlaNoRow past the query's rows.
__device__ __forceinline__ int mla_raw_id(const MlaArgs &a, int b, int t, int j, int nr) {
    const int r = t * kMlaTok + j;
    return r < nr ? __ldg(a.rows + (int64_t)b * a.max_rows + r) : kMlaNoRow;
}

// The id a tile row reads, or -1: past the query's rows, or an id outside the cache (then the
// error is recorded and the row is skipped).
__device__ __forceinline__ int mla_checked_id(const MlaArgs &a, int id, int b) {
    if (id == kMlaNoRow) return -1;
    if (id < 0 || id >= a.n_tok) {
        record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereMla, b);
        return -1;
    }
    return id;
}

__global__ void __launch_bounds__(kMlaThreads, 1) mla_tile_kernel(MlaArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(sm);
    __shared__ uint64_t s_full, p_full, o_full;
    __shared__ uint32_t tmem_s;
    __shared__ float s_scale[kMlaTok][4];
    __shared__ uint32_t s_valid[2];                  // valid rows of the tile being computed

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, c = blockIdx.x;
    const int64_t w_lo = mla_range_lo(a, c), w_hi = mla_range_lo(a, c + 1);
    if (w_lo >= w_hi) return;

    if (warp == 4) tmem_alloc(&tmem_s, 512);
    if (tid == 0) {
        mbar_init(smem_u32(&s_full), 1);
        mbar_init(smem_u32(&p_full), kMlaRows);
        mbar_init(smem_u32(&o_full), 1);
        fence_mbar_init();
        for (int b = 0; b < a.B && c == 0; ++b)
            if (a.n_rows[b] > a.max_rows) record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereMla, b);
    }
    // every (query, half) the run touches starts as an empty partial (max -inf); a segment
    // with rows overwrites its own later
    if (tid < H) {
        for (int64_t P = w_lo / a.n_tiles; P <= (w_hi - 1) / a.n_tiles; ++P) {
            float *ml = a.part_ml + ((size_t)(c + P) * H + tid) * 2;
            ml[0] = -INFINITY;
            ml[1] = 0.f;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_s;

    // registers of the next tile: its raw row ids (one tile further ahead, loaded without a
    // check so that the loads overlap) and its row data (loaded while the previous tile computes)
    int id_lat[kMlaLatItems], id_rope[kMlaRopeItems], id_sc = kMlaNoRow, id_b = 0;
    uint4 d_lat[kMlaLatItems], d_rope[kMlaRopeItems], d_sc = make_uint4(0, 0, 0, 0);
    bool d_valid = false;                            // the data's row (threads < 64) is attended
    auto load_ids = [&](int64_t w) {
        const int64_t P = w / a.n_tiles;
        const int b = (int)(P >> 1), t = (int)(w - P * a.n_tiles), nr = mla_rows_of(a, b);
        id_b = b;
#pragma unroll
        for (int k = 0; k < kMlaLatItems; ++k) id_lat[k] = mla_raw_id(a, b, t, warp + kMlaWarps * k, nr);
#pragma unroll
        for (int k = 0; k < kMlaRopeItems; ++k) id_rope[k] = mla_raw_id(a, b, t, (tid + kMlaThreads * k) >> 3, nr);
        id_sc = tid < kMlaTok ? mla_raw_id(a, b, t, tid, nr) : kMlaNoRow;
    };
    auto load_data = [&]() {
#pragma unroll
        for (int k = 0; k < kMlaLatItems; ++k) {
            const int id = mla_checked_id(a, id_lat[k], id_b);
            d_lat[k] = id >= 0 ? ldg_nc_v4(a.kv + (int64_t)id * kMlaRowBytes + lane * 16) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < kMlaRopeItems; ++k) {
            const int id = mla_checked_id(a, id_rope[k], id_b);
            d_rope[k] = id >= 0 ? ldg_nc_v4(a.kv + (int64_t)id * kMlaRowBytes + kMlaRopeOff + (tid & 7) * 16)
                                : make_uint4(0, 0, 0, 0);
        }
        const int id = mla_checked_id(a, id_sc, id_b);
        d_sc = id >= 0 ? ldg_nc_v4(a.kv + (int64_t)id * kMlaRowBytes + kMlaScaleOff) : make_uint4(0, 0, 0, 0);
        d_valid = id >= 0;
    };

    int64_t w = mla_next_item(a, w_lo, w_hi);
    if (w < w_hi) {
        load_ids(w);
        load_data();
    }
    int64_t w_next = w < w_hi ? mla_next_item(a, w + 1, w_hi) : w_hi;
    if (w_next < w_hi) load_ids(w_next);

    int q_b = -1;                                   // query whose heads the Q tile holds
    int64_t seg = -1;                               // (query, half) of the open segment
    bool o_has = false;                             // O holds this segment's earlier tiles
    float m_run = -INFINITY, l_run = 0.f;           // softmax threads: the row's running max, sum
    bool ok = true;
    uint32_t k = 0;                                 // tiles computed (mbarrier phases)
    while (w < w_hi && ok) {
        const int64_t P = w / a.n_tiles;
        const int b = (int)(P >> 1), hf = (int)(P & 1);
        // ---- (a) the previous tile's MMAs are done: K, Q and O may be rewritten
        if (k > 0) ok = __syncthreads_and(mbar_wait_bounded(smem_u32(&o_full), (k - 1) & 1, kWaitLimitNs));
        if (!ok) break;
        tc_fence_after();
        if (P != seg) {
            seg = P;
            o_has = false;
            m_run = -INFINITY;
            l_run = 0.f;
            if (b != q_b) {                          // the query's heads; rows H..127 zero
                q_b = b;
                for (int i = tid; i < kMlaRows * kMlaBlocks * 8; i += kMlaThreads) {
                    const int h = i / (kMlaBlocks * 8), rem = i - h * (kMlaBlocks * 8), blk = rem >> 3, g = rem & 7;
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (h < H) v = ldg_nc_v4(a.q + ((int64_t)b * H + h) * kMlaDim + blk * 64 + g * 8);
                    st_shared_v4(sbase + kMlaQ + blk * (kMlaRows * 128) + swz(h, g), v);
                }
            }
        }
        // ---- (b) the tile's rows into the swizzled K tile
        if (tid < kMlaTok) {
            s_scale[tid][0] = __uint_as_float(d_sc.x);
            s_scale[tid][1] = __uint_as_float(d_sc.y);
            s_scale[tid][2] = __uint_as_float(d_sc.z);
            s_scale[tid][3] = __uint_as_float(d_sc.w);
        }
        if (warp < 2) {
            const unsigned bal = __ballot_sync(0xffffffffu, d_valid);
            if (lane == 0) s_valid[warp] = bal;
        }
        __syncthreads();
#pragma unroll
        for (int q = 0; q < kMlaLatItems; ++q) {
            const int j = warp + kMlaWarps * q;
            float f[16];
            e4m3x16_to_f32(d_lat[q], f);
            const float sc = s_scale[j][lane >> 3];
            uint32_t u[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) u[e] = pack_bf16x2(f[2 * e] * sc, f[2 * e + 1] * sc);
            const uint32_t base = sbase + kMlaK + (lane >> 2) * (kMlaTok * 128);
            const int g0 = (lane & 3) * 2;
            st_shared_v4(base + swz(j, g0), make_uint4(u[0], u[1], u[2], u[3]));
            st_shared_v4(base + swz(j, g0 + 1), make_uint4(u[4], u[5], u[6], u[7]));
        }
#pragma unroll
        for (int q = 0; q < kMlaRopeItems; ++q) {
            const int i = tid + kMlaThreads * q;
            st_shared_v4(sbase + kMlaK + 8 * (kMlaTok * 128) + swz(i >> 3, i & 7), d_rope[q]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t qa = sbase + kMlaQ, kb = sbase + kMlaK;
        if (warp == 4 && lane == 0) {                // S = Q K^T runs while the warps issue loads
#pragma unroll 1
            for (int ks = 0; ks < kMlaDim / 16; ++ks) {
                const uint64_t ad = tc_desc(qa + (ks >> 2) * (kMlaRows * 128) + (ks & 3) * 32, 16, 1024);
                const uint64_t bd = tc_desc(kb + (ks >> 2) * (kMlaTok * 128) + (ks & 3) * 32, 16, 1024);
                tc_mma(tmem + kMlaTmS, ad, bd, tc_idesc(kMlaRows, kMlaTok, 0), ks > 0);
            }
            tc_commit(smem_u32(&s_full));
        }
        // ---- (c) the next tile's rows in flight while this one is computed (ids one further)
        const int64_t w2 = w_next;
        if (w2 < w_hi) {
            load_data();
            w_next = mla_next_item(a, w2 + 1, w_hi);
            if (w_next < w_hi) load_ids(w_next);
        }
        const bool seg_end = w2 >= w_hi || w2 / a.n_tiles != P;
        const uint32_t ph = k & 1;
        // ---- (d) roles
        if (warp == 4) {
            if (lane == 0) {
                if (mbar_wait_bounded(smem_u32(&p_full), ph, kWaitLimitNs)) {
                    tc_fence_after();
                    // V: this half's four column blocks of the latent, read MN-major (16 rows per k-step)
                    const uint32_t vb = kb + (uint32_t)(hf * 4) * (kMlaTok * 128);
#pragma unroll
                    for (int ks = 0; ks < kMlaTok / 16; ++ks) {
                        const uint64_t bd = tc_desc(vb + ks * 2048, kMlaTok * 128, 1024);
                        tc_mma_ta(tmem + kMlaTmO, tmem + kMlaTmP + ks * 8, bd, tc_idesc(kMlaRows, 256, 1),
                                  o_has || ks > 0);
                    }
                } else {
                    record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, b);
                }
                tc_commit(smem_u32(&o_full));        // also after a timeout: the next wait ends
            }
            __syncwarp();
        } else if (warp < 4) {
            const uint32_t t_row = tmem + ((uint32_t)(32 * warp) << 16);
            const bool got_s = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&s_full), ph, kWaitLimitNs));
            if (got_s) {
                tc_fence_after();
                float s0[32], s1[32];
                tmem_ld32_async(t_row + kMlaTmS, s0);
                tmem_ld32_async(t_row + kMlaTmS + 32, s1);
                tmem_wait_ld(s0);
                tmem_wait_ld(s1);
                const uint32_t v0 = s_valid[0], v1 = s_valid[1];
                float mx = -INFINITY;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    if ((v0 >> j) & 1u) mx = fmaxf(mx, s0[j]);
                    if ((v1 >> j) & 1u) mx = fmaxf(mx, s1[j]);
                }
                const float m_t = mx * a.scale_log2;
                // raise the running max (and rescale O) only when this tile's max passes it by 2^8
                const bool raise = m_t > m_run + kMlaRescale;
                const float alpha = raise && m_run != -INFINITY ? ex2_approx(m_run - m_t) : 1.f;
                if (raise) {
                    m_run = m_t;
                    l_run *= alpha;
                }
                if (o_has && __any_sync(0xffffffffu, alpha != 1.f)) {
                    // warp-collective: every lane loads and stores its row, scaled by its alpha
#pragma unroll 1
                    for (int c0 = 0; c0 < 256; c0 += 32) {
                        float ov[32];
                        tmem_ld32(t_row + kMlaTmO + c0, ov);
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] *= alpha;
                        tmem_st32(t_row + kMlaTmO + c0, ov);
                    }
                }
                uint32_t pk[32];
                float ps = 0.f;
#pragma unroll
                for (int j = 0; j < 64; j += 2) {
                    const float x0 = j < 32 ? s0[j] : s1[j - 32], x1 = j < 32 ? s0[j + 1] : s1[j - 31];
                    const uint32_t vm = j < 32 ? v0 : v1;
                    const int jb = j & 31;
                    const float e0 = (vm >> jb) & 1u ? ex2_approx(fmaf(x0, a.scale_log2, -m_run)) : 0.f;
                    const float e1 = (vm >> (jb + 1)) & 1u ? ex2_approx(fmaf(x1, a.scale_log2, -m_run)) : 0.f;
                    ps += e0 + e1;
                    pk[j >> 1] = pack_bf16x2(e0, e1);
                }
                l_run += ps;
                tmem_st32(t_row + kMlaTmP, pk);
            } else if (lane == 0) {
                record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, b);
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&p_full));
            if (seg_end) {
                // ---- the segment's partial: unnormalised O rows and (max, sum)
                const bool got_o =
                    got_s && __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&o_full), ph, kWaitLimitNs));
                const int row = tid;                         // MMA row = TMEM lane = head
                if (got_o) {
                    tc_fence_after();
                    float *acc = a.part_acc + ((size_t)(c + P) * H + row) * 256;
#pragma unroll 1
                    for (int c0 = 0; c0 < 256; c0 += 32) {
                        float ov[32];
                        tmem_ld32(t_row + kMlaTmO + c0, ov);     // warp-collective
                        if (row < H) {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                *reinterpret_cast<float4 *>(acc + c0 + 4 * e) =
                                    make_float4(ov[4 * e], ov[4 * e + 1], ov[4 * e + 2], ov[4 * e + 3]);
                        }
                    }
                    if (row < H) {
                        float *ml = a.part_ml + ((size_t)(c + P) * H + row) * 2;
                        ml[0] = m_run;
                        ml[1] = l_run;
                    }
                } else if (lane == 0 && got_s) {
                    record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, b);
                }
                tc_fence_before();
            }
        }
        o_has = true;
        ++k;
        w = w2;
    }
    // every MMA has completed before the columns are freed
    if (k > 0 && tid == 0 && !mbar_wait_bounded(smem_u32(&o_full), (k - 1) & 1, kWaitLimitNs))
        record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, 0);
    if (!ok && tid == 0) record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, 0);
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Per (head, query): each half's segment partials merged by log-sum-exp; 256 threads, one
// latent dim of each half each. The CTAs whose runs touch (query, half) P are the partials
// c + P for c in [c_lo, c_hi].
__global__ void __launch_bounds__(256) mla_merge_kernel(MlaArgs a) {
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int H = a.H;
    const int64_t W = (int64_t)a.B * 2 * a.n_tiles;
    float L0 = 0.f, M0 = -INFINITY;
    for (int hf = 0; hf < 2 && W == 0; ++hf)          // no tiles at all: zeros, lse -inf
        a.out[((int64_t)b * H + h) * kMlaLat + hf * 256 + tid] = 0;
    for (int hf = 0; hf < 2 && W > 0; ++hf) {
        const int64_t P = 2 * (int64_t)b + hf, p_lo = P * a.n_tiles, p_hi = p_lo + a.n_tiles;
        int c_lo = (int)(p_lo * a.grid / W);
        c_lo = c_lo > 0 ? c_lo - 1 : 0;
        while (c_lo + 1 < a.grid && mla_range_lo(a, c_lo + 1) <= p_lo) ++c_lo;
        float M = -INFINITY;
        for (int c = c_lo; c < a.grid && mla_range_lo(a, c) < p_hi; ++c)
            M = fmaxf(M, a.part_ml[((size_t)(c + P) * H + h) * 2]);
        float L = 0.f, o = 0.f;
        for (int c = c_lo; c < a.grid && mla_range_lo(a, c) < p_hi; ++c) {
            const float *ml = a.part_ml + ((size_t)(c + P) * H + h) * 2;
            if (ml[0] == -INFINITY) continue;
            const float wgt = exp2f(ml[0] - M);
            L += ml[1] * wgt;
            o += wgt * a.part_acc[((size_t)(c + P) * H + h) * 256 + tid];
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        a.out[((int64_t)b * H + h) * kMlaLat + hf * 256 + tid] = float_to_bf16_bits(o * inv);
        if (hf == 0) {
            L0 = L;
            M0 = M;
        }
    }
    if (tid == 0 && a.lse != nullptr) a.lse[(int64_t)b * H + h] = L0 > 0.f ? (M0 + log2f(L0)) * kLn2 : -INFINITY;
}

size_t mla_scratch_bytes(int H, int B, int max_rows) {
    (void)max_rows;
    const size_t n_part = (size_t)kMlaMaxCtas + 2 * (size_t)B;
    return n_part * H * 256 * 4 + n_part * H * 2 * 4 + 256;
}

namespace {
bool g_mla_attr[64];
int g_mla_sms[64];
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
        e = cudaDeviceGetAttribute(&g_mla_sms[dev], cudaDevAttrMultiProcessorCount, dev);
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
    const int64_t W = (int64_t)B * 2 * a.n_tiles;
    int sms = g_mla_sms[dev] < kMlaMaxCtas ? g_mla_sms[dev] : kMlaMaxCtas;
    a.grid = (int)(W < sms ? W : sms);
    a.scale_log2 = scale * kLog2e;
    a.part_acc = static_cast<float *>(scratch);
    a.part_ml = a.part_acc + ((size_t)kMlaMaxCtas + 2 * (size_t)B) * H * 256;
    a.out = out;
    a.lse = lse;
    a.hdr = hdr;
    if (a.grid > 0) {
        mla_tile_kernel<<<a.grid, kMlaThreads, kMlaSmem, st>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    } else {
        a.grid = 1;                                  // no rows anywhere: the merge writes zeros
    }
    mla_merge_kernel<<<dim3(H, B), 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa
