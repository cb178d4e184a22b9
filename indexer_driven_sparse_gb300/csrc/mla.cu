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
    int32_t halves;           // segments per query: 2 (latent halves, mla_tile_kernel) or 1
    float scale_log2;
    float *part_acc;          // [grid + halves B][H][512 / halves] unnormalised O rows of a segment
    float *part_ml;           // [grid + halves B][H][2]   (max, sum) in log2 units
    uint16_t *out;            // [B][H][512]
    float *lse;               // [B][H] or nullptr
    WsHeader *hdr;
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Row counts of the queries a CTA's run touches, read once into shared memory (the run
// walks them in order; a count read from global memory at each step would put a dependent
// round trip in front of every tile's loads). Queries past the cached window are read from
// global memory.
constexpr int kMlaCountCache = 128;
struct MlaCounts {
    const int *s;   // shared: counts of queries b0 .. b0 + kMlaCountCache - 1
    int b0;
};

__device__ __forceinline__ int mla_clamp_rows(const MlaArgs &a, int n) {
    return n < 0 ? 0 : (n > a.max_rows ? a.max_rows : n);
}

__device__ __forceinline__ int mla_rows_of(const MlaArgs &a, const MlaCounts &cnt, int b) {
    const unsigned i = (unsigned)(b - cnt.b0);
    return i < (unsigned)kMlaCountCache ? cnt.s[i] : mla_clamp_rows(a, a.n_rows[b]);
}

// First work item >= w (below w_hi) whose tile holds rows of its query; else w_hi.
__device__ __forceinline__ int64_t mla_next_item(const MlaArgs &a, const MlaCounts &cnt, int64_t w, int64_t w_hi) {
    while (w < w_hi) {
        const int64_t P = w / a.n_tiles;
        const int t = (int)(w - P * a.n_tiles);
        if (t * kMlaTok < mla_rows_of(a, cnt, (int)(P / a.halves))) return w;
        w = (P + 1) * a.n_tiles;
    }
    return w_hi;
}

// Work range of CTA c: [W c / G, W (c + 1) / G) with W = B x 2 x n_tiles.
__device__ __forceinline__ int64_t mla_range_lo(const MlaArgs &a, int c) {
    return (int64_t)a.B * a.halves * a.n_tiles * c / a.grid;
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
    __shared__ int s_count[kMlaCountCache];

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
    const MlaCounts cnt{s_count, (int)(w_lo / (2 * (int64_t)a.n_tiles))};
    for (int i = tid; i < kMlaCountCache; i += kMlaThreads)
        s_count[i] = cnt.b0 + i < a.B ? mla_clamp_rows(a, a.n_rows[cnt.b0 + i]) : 0;
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
        const int b = (int)(P >> 1), t = (int)(w - P * a.n_tiles), nr = mla_rows_of(a, cnt, b);
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

    int64_t w = mla_next_item(a, cnt, w_lo, w_hi);
    if (w < w_hi) {
        load_ids(w);
        load_data();
    }
    int64_t w_next = w < w_hi ? mla_next_item(a, cnt, w + 1, w_hi) : w_hi;
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
            w_next = mla_next_item(a, cnt, w2 + 1, w_hi);
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

// The CTA whose run holds work item x: the last c with mla_range_lo(c) <= x.
__device__ __forceinline__ int mla_cta_of(const MlaArgs &a, int64_t x, int64_t W) {
    int c = (int)(x * a.grid / W);
    c = c > 0 ? c - 1 : 0;
    while (c + 1 < a.grid && mla_range_lo(a, c + 1) <= x) ++c;
    return c;
}

// Per (head, query): each half's segment partials merged by log-sum-exp. The CTAs whose
// runs touch (query, half) P form the range [c_lo, c_hi]; their partials are c + P. Warp hf
// finds the range of half hf and turns the partials' (max, sum) into weights in shared
// memory once; then every thread merges one latent dim of each half (256 threads).
__global__ void __launch_bounds__(256) mla_merge_kernel(MlaArgs a) {
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.H;
    const int64_t W = (int64_t)a.B * 2 * a.n_tiles;
    __shared__ float s_w[2][kMlaMaxCtas];
    __shared__ int s_c0[2], s_n[2];
    __shared__ float s_M[2], s_L[2];
    if (W == 0) {                                    // no tiles at all: zeros, lse -inf
        for (int hf = 0; hf < 2; ++hf) a.out[((int64_t)b * H + h) * kMlaLat + hf * 256 + tid] = 0;
        if (tid == 0 && a.lse != nullptr) a.lse[(int64_t)b * H + h] = -INFINITY;
        return;
    }
    if (warp < 2) {
        const int hf = warp;
        const int64_t P = 2 * (int64_t)b + hf, p_lo = P * a.n_tiles;
        const int c_lo = mla_cta_of(a, p_lo, W), c_hi = mla_cta_of(a, p_lo + a.n_tiles - 1, W);
        const int n = c_hi - c_lo + 1;
        float M = -INFINITY;
        for (int k = lane; k < n; k += 32) M = fmaxf(M, a.part_ml[((size_t)(c_lo + k + P) * H + h) * 2]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.f;
        for (int k = lane; k < n; k += 32) {
            const float *ml = a.part_ml + ((size_t)(c_lo + k + P) * H + h) * 2;
            const float wgt = ml[0] == -INFINITY ? 0.f : exp2f(ml[0] - M);
            s_w[hf][k] = wgt;
            L = fmaf(ml[1], wgt, L);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (lane == 0) {
            s_c0[hf] = c_lo;
            s_n[hf] = n;
            s_M[hf] = M;
            s_L[hf] = L;
        }
    }
    __syncthreads();
    for (int hf = 0; hf < 2; ++hf) {
        const int64_t P = 2 * (int64_t)b + hf;
        const int c0 = s_c0[hf], n = s_n[hf];
        float o = 0.f;
        for (int k = 0; k < n; ++k)
            if (s_w[hf][k] != 0.f) o = fmaf(s_w[hf][k], a.part_acc[((size_t)(c0 + k + P) * H + h) * 256 + tid], o);
        const float L = s_L[hf];
        a.out[((int64_t)b * H + h) * kMlaLat + hf * 256 + tid] = float_to_bf16_bits(L > 0.f ? o * (1.f / L) : 0.f);
    }
    if (tid == 0 && a.lse != nullptr) a.lse[(int64_t)b * H + h] = s_L[0] > 0.f ? (s_M[0] + log2f(s_L[0])) * kLn2 : -INFINITY;
}

// ------------------------------------------------------------------ transposed kernel, H <= 64
// mla_tr_kernel computes each 64-row tile once for all 512 latent dims, with the roles of the
// operands exchanged so that the 64 heads are the N dimension of every MMA:
//   S^T(t) = K(t) Q^T        M 64 (the tile's rows), N 64 heads, K 576; an M = 64 result
//                            holds row 16 q + l in lane l < 16 of tensor-memory lane quarter q;
//   O^T   += V(t)^T P(t)^T   per 128 latent dims: M 128 dims (V read MN-major from the same
//                            K tile), N 64 heads, K 64 rows; P^T (bf16, one 128-byte row of 64
//                            heads per tile row) is written to shared memory by the softmax.
// O^T (512 dims x 64 heads, fp32) takes 256 tensor-memory columns and the two S^T buffers 128,
// so one CTA holds a query's whole output and no latent half is computed twice. Roles:
//   - warps 9-15 (224 converters): the next tile's rows in registers (row ids one tile further
//     ahead), stored as bf16 into one of two K tiles; the query's heads reloaded when it changes;
//   - warp 8 (one thread): S^T(t) as soon as K(t) is stored, then O^T += V(t-1)^T P(t-1)^T once
//     the softmax of the previous tile is done;
//   - warps 0-7 (softmax group): lanes 0-15 of warp w hold tile row 16 (w mod 4) + lane for
//     heads 0-31 (warps 0-3) or 32-63 (4-7); per head, the tile maximum and
//     sum are reduced over the rows by warp reduce-scatter and shared memory, the running maximum
//     (raised, with O rescaled, only past 2^8 growth) kept by one lane per head. All eight warps
//     rescale O^T and write the segment's partial (each warp one lane quarter, 32 heads).
// Work items are (query, tile) pairs; a CTA's run is a contiguous range of them and each query
// it touches yields one partial, merged by mla_merge_tr_kernel. Every wait is bounded; a wait
// that gives up records QSA_ERR_DEVICE_TIMEOUT and sets a CTA-wide abort flag after which every
// wait returns at once, while every thread still passes the same named barriers.
constexpr int kTrThreads = 512;                                 // 16 warps: 4 per scheduler, 128 registers
constexpr int kTrSoft = 256;                                    // softmax group: warps 0-7
constexpr int kTrMmaWarp = 8;
constexpr int kTrConv0 = 9;                                     // converters: warps 9-15
constexpr int kTrConvWarps = 7, kTrConv = 32 * kTrConvWarps;
constexpr int kTrLatItems = (kMlaTok + kTrConvWarps - 1) / kTrConvWarps;   // rows cw + 7k (10; the last partial)
constexpr int kTrRopeItems = (kMlaTok * 8 + kTrConv - 1) / kTrConv;       // rotary granules ct + 224k (3)
constexpr uint32_t kTrBlk = kMlaTok * 128;                      // a column block of a 64-row tile
constexpr uint32_t kTrTile = kMlaBlocks * kTrBlk;               // 73,728 B
constexpr uint32_t kTrQ = 0, kTrK0 = kTrTile, kTrP = 3 * kTrTile;   // Q, K tiles 0 and 1, P^T
constexpr uint32_t kTrMisc = kTrP + kMlaTok * 128;              // small state after the tiles
constexpr int kTrCount = 32;                                    // cached row counts
struct TrMisc {
    uint64_t kfull[2], kfree[2], sfull[2], pfull, ofull, ofree, done;
    uint32_t tmem, abort, resc, pad;
    uint32_t valid[2][2];
    float red[4][kMlaTok];        // per lane quarter: head maxima
    float sum[4][kMlaTok];        // per lane quarter: head sums
    float mref[kMlaTok], alpha[kMlaTok];
    int count[kTrCount];
};
constexpr uint32_t kTrSmem = kTrMisc + (uint32_t)sizeof(TrMisc);
constexpr uint32_t kTrTmS = 0, kTrTmO = 128;                    // S^T x2 (64 cols each), O^T 4 x 64
constexpr int kTrBarSoft = 1;

__device__ __forceinline__ void named_bar(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// kind::f16 instruction descriptor with both operand majors: fp32 accumulate, bf16 A and B
__device__ __forceinline__ uint32_t tr_idesc(int M, int N, int a_mn, int b_mn) {
    return tc_idesc(M, N, b_mn) | ((uint32_t)a_mn << 15);
}

// Bounded wait that also gives up at once when the CTA has aborted; a timeout sets the flag.
__device__ __forceinline__ bool tr_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            return false;
        }
    }
    return true;
}

// Warp reduce-scatter of 32 values per lane: afterwards lane l holds op over the 32 lanes of
// value l (max or sum).
template <bool MAX>
__device__ __forceinline__ float tr_reduce_scatter(float (&v)[32], int lane) {
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
        const bool up = (lane & d) != 0;
#pragma unroll
        for (int i = 0; i < d; ++i) {
            const float send = up ? v[i] : v[i + d];
            const float keep = up ? v[i + d] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, d);
            v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
        }
    }
    return v[0];
}

// The walk over a CTA's run, identical in every role.
struct TrWalk {
    int64_t w, w_next, w_hi;
    int b, b_prev, seg;                              // query; segments (queries) opened so far - 1
    bool first, last;
    __device__ void settle(const MlaArgs &a) {
        if (w >= w_hi) return;
        b = (int)(w / a.n_tiles);
        first = b != b_prev;
        if (first) ++seg;
        last = w_next >= w_hi || (int)(w_next / a.n_tiles) != b;
    }
    __device__ void init(const MlaArgs &a, const MlaCounts &cnt, int64_t w_lo, int64_t hi) {
        w_hi = hi;
        b_prev = -1;
        seg = -1;
        w = mla_next_item(a, cnt, w_lo, w_hi);
        w_next = w < w_hi ? mla_next_item(a, cnt, w + 1, w_hi) : w_hi;
        settle(a);
    }
    __device__ void advance(const MlaArgs &a, const MlaCounts &cnt) {
        b_prev = b;
        w = w_next;
        w_next = w < w_hi ? mla_next_item(a, cnt, w + 1, w_hi) : w_hi;
        settle(a);
    }
};

__global__ void __launch_bounds__(kTrThreads, 1) mla_tr_kernel(MlaArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_u32(smem);
    TrMisc &m = *reinterpret_cast<TrMisc *>(smem + kTrMisc);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H, c = blockIdx.x;
    const int64_t w_lo = mla_range_lo(a, c), w_hi = mla_range_lo(a, c + 1);
    if (w_lo >= w_hi) return;
    if (sbase & 1023) {                              // the swizzled tiles need 1024-byte alignment
        if (tid == 0) record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereMla, -1);
        return;
    }
    volatile uint32_t *abort = &m.abort;
    const uint32_t qa = sbase + kTrQ, kt0 = sbase + kTrK0, pt = sbase + kTrP;

    if (warp == kTrMmaWarp) tmem_alloc(&m.tmem, 512);
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&m.kfull[i]), kTrConv);
            mbar_init(smem_u32(&m.kfree[i]), 1);
            mbar_init(smem_u32(&m.sfull[i]), 1);
        }
        mbar_init(smem_u32(&m.pfull), kTrSoft);
        mbar_init(smem_u32(&m.ofull), 1);
        mbar_init(smem_u32(&m.ofree), kTrSoft);
        mbar_init(smem_u32(&m.done), 1);
        fence_mbar_init();
        m.abort = 0;
        m.resc = 0;
        for (int b = 0; b < a.B && c == 0; ++b)
            if (a.n_rows[b] > a.max_rows) record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereMla, b);
    }
    if (tid < H) {                                   // empty partials of every query touched
        for (int64_t b = w_lo / a.n_tiles; b <= (w_hi - 1) / a.n_tiles; ++b) {
            float *ml = a.part_ml + ((size_t)(c + b) * H + tid) * 2;
            ml[0] = -INFINITY;
            ml[1] = 0.f;
        }
    }
    const MlaCounts cnt{m.count, (int)(w_lo / a.n_tiles)};
    for (int i = tid; i < kTrCount; i += kTrThreads)
        m.count[i] = cnt.b0 + i < a.B ? mla_clamp_rows(a, a.n_rows[cnt.b0 + i]) : 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = m.tmem;

    TrWalk wk;
    wk.init(a, cnt, w_lo, w_hi);

    if (warp >= kTrConv0) {
        // ------------------------------------------------------------ converters
        const int cw = warp - kTrConv0, ct = cw * 32 + lane;
        int id_lat[kTrLatItems], id_rope[kTrRopeItems], id_v = kMlaNoRow, id_b = 0;
        uint4 d_lat[kTrLatItems], d_rope[kTrRopeItems];
        float d_scl[kTrLatItems];
        bool d_valid = false;
        auto load_ids = [&](int64_t w) {
            const int b = (int)(w / a.n_tiles), t = (int)(w - (int64_t)b * a.n_tiles), nr = mla_rows_of(a, cnt, b);
            id_b = b;
#pragma unroll
            for (int k = 0; k < kTrLatItems; ++k) {
                const int j = cw + kTrConvWarps * k;
                id_lat[k] = j < kMlaTok ? mla_raw_id(a, b, t, j, nr) : kMlaNoRow;
            }
#pragma unroll
            for (int k = 0; k < kTrRopeItems; ++k) {
                const int i = ct + kTrConv * k;
                id_rope[k] = i < kMlaTok * 8 ? mla_raw_id(a, b, t, i >> 3, nr) : kMlaNoRow;
            }
            id_v = ct < kMlaTok ? mla_raw_id(a, b, t, ct, nr) : kMlaNoRow;
        };
        auto load_data = [&]() {
#pragma unroll
            for (int k = 0; k < kTrLatItems; ++k) {
                const int id = mla_checked_id(a, id_lat[k], id_b);
                const uint8_t *row = a.kv + (int64_t)(id >= 0 ? id : 0) * kMlaRowBytes;
                d_lat[k] = id >= 0 ? ldg_nc_v4(row + lane * 16) : make_uint4(0, 0, 0, 0);
                d_scl[k] = id >= 0 ? __ldg(reinterpret_cast<const float *>(row + kMlaScaleOff) + (lane >> 3)) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < kTrRopeItems; ++k) {
                const int id = mla_checked_id(a, id_rope[k], id_b);
                d_rope[k] = id >= 0 ? ldg_nc_v4(a.kv + (int64_t)id * kMlaRowBytes + kMlaRopeOff + (ct & 7) * 16)
                                    : make_uint4(0, 0, 0, 0);
            }
            d_valid = mla_checked_id(a, id_v, id_b) >= 0;
        };
        if (wk.w < w_hi) {
            load_ids(wk.w);
            load_data();
            if (wk.w_next < w_hi) load_ids(wk.w_next);
        }
        int q_b = -1;
        for (uint32_t t = 0; wk.w < w_hi; ++t) {
            const int buf = t & 1, b = wk.b;
            const uint32_t kb = kt0 + buf * kTrTile;
            if (t >= 2 && !tr_wait(smem_u32(&m.kfree[buf]), ((t - 2) >> 1) & 1, abort) && ct == 0)
                record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, b);
            if (b != q_b) {                          // the query's heads (rows H..63 zero)
                if (t >= 1 && !tr_wait(smem_u32(&m.sfull[(t - 1) & 1]), ((t - 1) >> 1) & 1, abort) && ct == 0)
                    record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, b);
                q_b = b;
                // 64 heads x 72 granules over 224 threads: 21 per thread (the last partial), seven
                // loaded at a time before they are stored
                constexpr int kQGran = kMlaTok * kMlaBlocks * 8;
                constexpr int kQItems = (kQGran + kTrConv - 1) / kTrConv, kQBatch = 7;
                static_assert(kQItems % kQBatch == 0, "whole batches");
#pragma unroll
                for (int i0 = 0; i0 < kQItems; i0 += kQBatch) {
                    uint4 v[kQBatch];
#pragma unroll
                    for (int k = 0; k < kQBatch; ++k) {
                        const int i = ct + kTrConv * (i0 + k), h = i / (kMlaBlocks * 8), rem = i - h * (kMlaBlocks * 8);
                        v[k] = i < kQGran && h < H
                                   ? ldg_nc_v4(a.q + ((int64_t)b * H + h) * kMlaDim + (rem >> 3) * 64 + (rem & 7) * 8)
                                   : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                    for (int k = 0; k < kQBatch; ++k) {
                        const int i = ct + kTrConv * (i0 + k), h = i / (kMlaBlocks * 8), rem = i - h * (kMlaBlocks * 8);
                        if (i < kQGran) st_shared_v4(qa + (rem >> 3) * kTrBlk + swz(h, rem & 7), v[k]);
                    }
                }
            }
            if (cw < 2) {
                const unsigned bal = __ballot_sync(0xffffffffu, d_valid);
                if (lane == 0) m.valid[buf][cw] = bal;
            }
#pragma unroll
            for (int q = 0; q < kTrLatItems; ++q) {
                const int j = cw + kTrConvWarps * q;
                if (j >= kMlaTok) break;
                float f[16];
                e4m3x16_to_f32(d_lat[q], f);
                const float sc = d_scl[q];
                uint32_t u[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) u[e] = pack_bf16x2(f[2 * e] * sc, f[2 * e + 1] * sc);
                const uint32_t base = kb + (lane >> 2) * kTrBlk;
                const int g0 = (lane & 3) * 2;
                st_shared_v4(base + swz(j, g0), make_uint4(u[0], u[1], u[2], u[3]));
                st_shared_v4(base + swz(j, g0 + 1), make_uint4(u[4], u[5], u[6], u[7]));
            }
#pragma unroll
            for (int q = 0; q < kTrRopeItems; ++q) {
                const int i = ct + kTrConv * q;
                if (i < kMlaTok * 8) st_shared_v4(kb + 8 * kTrBlk + swz(i >> 3, i & 7), d_rope[q]);
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&m.kfull[buf]));
            if (wk.w_next < w_hi) {                  // the next tile's rows in flight (ids one further)
                load_data();
                const int64_t w3 = mla_next_item(a, cnt, wk.w_next + 1, w_hi);
                if (w3 < w_hi) load_ids(w3);
            }
            wk.advance(a, cnt);
        }
    } else if (warp == kTrMmaWarp) {
        // ------------------------------------------------------------ MMA issue (one thread)
        if (lane == 0) {
            bool pv_first = false;
            int pv_seg = 0, pv_b = 0;
            auto pv = [&](uint32_t u) {              // O^T += V(u)^T P(u)^T, per 128 latent dims
                bool go = tr_wait(smem_u32(&m.pfull), u & 1, abort);
                if (go && pv_first && pv_seg > 0) go = tr_wait(smem_u32(&m.ofree), (pv_seg - 1) & 1, abort);
                if (go) {
                    tc_fence_after();
                    const uint32_t kb = kt0 + (u & 1) * kTrTile;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
#pragma unroll
                        for (int ks = 0; ks < kMlaTok / 16; ++ks) {
                            const uint64_t ad = tc_desc(kb + (2 * i) * kTrBlk + ks * 2048, kTrBlk, 1024);
                            const uint64_t bd = tc_desc(pt + ks * 2048, kTrBlk, 1024);
                            tc_mma(tmem + kTrTmO + 64 * i, ad, bd, tr_idesc(128, kMlaTok, 1, 1), !pv_first || ks > 0);
                        }
                    }
                } else {
                    record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, pv_b);
                }
                tc_commit(smem_u32(&m.kfree[u & 1]));   // also after a timeout: the phases advance
                tc_commit(smem_u32(&m.ofull));
            };
            uint32_t t = 0;
            for (; wk.w < w_hi; ++t) {
                const int buf = t & 1;
                if (tr_wait(smem_u32(&m.kfull[buf]), (t >> 1) & 1, abort)) {
                    tc_fence_after();
                    const uint32_t kb = kt0 + buf * kTrTile;
#pragma unroll 1
                    for (int ks = 0; ks < kMlaDim / 16; ++ks) {
                        const uint64_t ad = tc_desc(kb + (ks >> 2) * kTrBlk + (ks & 3) * 32, 16, 1024);
                        const uint64_t bd = tc_desc(qa + (ks >> 2) * kTrBlk + (ks & 3) * 32, 16, 1024);
                        tc_mma(tmem + kTrTmS + buf * 64, ad, bd, tr_idesc(kMlaTok, kMlaTok, 0, 0), ks > 0);
                    }
                } else {
                    record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, wk.b);
                }
                tc_commit(smem_u32(&m.sfull[buf]));
                if (t > 0) pv(t - 1);
                pv_first = wk.first;
                pv_seg = wk.seg;
                pv_b = wk.b;
                wk.advance(a, cnt);
            }
            if (t > 0) pv(t - 1);
            tc_commit(smem_u32(&m.done));            // every MMA of this CTA has completed
            if (!tr_wait(smem_u32(&m.done), 0, abort)) record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax group, epilogue
        // S^T is an M = 64 MMA: tile row 16 q + l sits in lane l < 16 of TMEM lane quarter q
        const int quad = warp & 3, hg = warp >> 2;    // TMEM lane quarter; head group (32 heads)
        const int row = 16 * quad + (lane & 15);      // the tile row of lanes 0-15
        const bool owner = quad == 0;                 // lane l of warps 0 / 4 keeps head 32 hg + l
        const int oh = 32 * hg + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(32 * quad) << 16);
        float m_run = -INFINITY, l_run = 0.f;         // owners: the head's running max and sum
        for (uint32_t t = 0; wk.w < w_hi; ++t) {
            const int buf = t & 1, b = wk.b;
            bool ok = tr_wait(smem_u32(&m.kfull[buf]), (t >> 1) & 1, abort);   // the tile's valid rows
            ok = tr_wait(smem_u32(&m.sfull[buf]), (t >> 1) & 1, abort) && ok;
            tc_fence_after();
            float s[32], v[32];
            tmem_ld32_async(t_lane + kTrTmS + buf * 64 + 32 * hg, s);
            tmem_wait_ld(s);
            const bool valid = lane < 16 && ((m.valid[buf][row >> 5] >> (row & 31)) & 1u);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = valid ? s[j] : -INFINITY;
            m.red[quad][oh] = tr_reduce_scatter<true>(v, lane);
            named_bar(kTrBarSoft, kTrSoft);
            if (owner) {
                // the previous tile's sums, then this tile's maximum against the running one
                if (!wk.first) l_run += (m.sum[0][oh] + m.sum[1][oh]) + (m.sum[2][oh] + m.sum[3][oh]);
                const float m_t = fmaxf(fmaxf(m.red[0][oh], m.red[1][oh]), fmaxf(m.red[2][oh], m.red[3][oh])) * a.scale_log2;
                if (wk.first) {
                    m_run = -INFINITY;
                    l_run = 0.f;
                }
                const bool raise = m_t > m_run + kMlaRescale;
                const float alpha = raise && m_run != -INFINITY ? ex2_approx(m_run - m_t) : 1.f;
                if (raise) {
                    m_run = m_t;
                    l_run *= alpha;
                }
                m.mref[oh] = m_run;
                m.alpha[oh] = alpha;
                if (alpha != 1.f && !wk.first) m.resc = 1;
            }
            // PV of the previous tile has completed: P^T may be rewritten and O^T rescaled
            if (t > 0) ok = tr_wait(smem_u32(&m.ofull), (t - 1) & 1, abort) && ok;
            named_bar(kTrBarSoft, kTrSoft);
            tc_fence_after();
            {
                uint32_t pk[16];
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float e0 = valid ? ex2_approx(fmaf(s[j], a.scale_log2, -m.mref[32 * hg + j])) : 0.f;
                    const float e1 = valid ? ex2_approx(fmaf(s[j + 1], a.scale_log2, -m.mref[32 * hg + j + 1])) : 0.f;
                    v[j] = e0;
                    v[j + 1] = e1;
                    pk[j >> 1] = pack_bf16x2(e0, e1);
                }
                if (lane < 16) {
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        st_shared_v4(pt + swz(row, 4 * hg + g),
                                     make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]));
                }
                m.sum[quad][oh] = tr_reduce_scatter<false>(v, lane);
            }
            if (m.resc) {                            // warp-uniform: every lane reads the flag
#pragma unroll 1
                for (int i = 0; i < 4; ++i) {
                    float ov[32];
                    tmem_ld32(t_lane + kTrTmO + 64 * i + 32 * hg, ov);
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] *= m.alpha[32 * hg + e];
                    tmem_st32(t_lane + kTrTmO + 64 * i + 32 * hg, ov);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(&m.pfull));
            named_bar(kTrBarSoft, kTrSoft);          // the flag is read by all before it is cleared
            if (tid == 0) m.resc = 0;
            if (!ok && lane == 0) record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, b);
            if (wk.last) {
                // ---- the query's partial from this run: O^T columns and (max, sum) per head
                const bool got_o = tr_wait(smem_u32(&m.ofull), t & 1, abort);
                tc_fence_after();
                if (owner && oh < H) {
                    float *ml = a.part_ml + ((size_t)(c + b) * H + oh) * 2;
                    ml[0] = m_run;
                    ml[1] = l_run + ((m.sum[0][oh] + m.sum[1][oh]) + (m.sum[2][oh] + m.sum[3][oh]));
                }
#pragma unroll 1
                for (int i = 0; i < 4; ++i) {
                    float ov[32];
                    tmem_ld32(t_lane + kTrTmO + 64 * i + 32 * hg, ov);     // warp-collective
                    const int d = 128 * i + 32 * quad + lane;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int h = 32 * hg + e;
                        if (h < H && got_o) a.part_acc[((size_t)(c + b) * H + h) * kMlaLat + d] = ov[e];
                    }
                }
                if (!got_o && lane == 0) record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereMla, b);
                tc_fence_before();
                mbar_arrive(smem_u32(&m.ofree));
            }
            wk.advance(a, cnt);
        }
    }
    // warp 8 saw every MMA complete (or gave up) before the columns are freed
    tc_fence_before();
    __syncthreads();
    if (warp == kTrMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Per (head, query) of mla_tr_kernel: the query's partials (one per CTA whose run touches it)
// merged by log-sum-exp; 256 threads, two latent dims each.
__global__ void __launch_bounds__(256) mla_merge_tr_kernel(MlaArgs a) {
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.H;
    const int64_t W = (int64_t)a.B * a.n_tiles;
    __shared__ float s_w[kMlaMaxCtas];
    __shared__ int s_c0, s_n;
    __shared__ float s_M, s_L;
    if (W == 0) {
        a.out[((int64_t)b * H + h) * kMlaLat + tid] = 0;
        a.out[((int64_t)b * H + h) * kMlaLat + 256 + tid] = 0;
        if (tid == 0 && a.lse != nullptr) a.lse[(int64_t)b * H + h] = -INFINITY;
        return;
    }
    if (warp == 0) {
        const int64_t p_lo = (int64_t)b * a.n_tiles;
        const int c_lo = mla_cta_of(a, p_lo, W), c_hi = mla_cta_of(a, p_lo + a.n_tiles - 1, W);
        const int n = c_hi - c_lo + 1;
        float M = -INFINITY;
        for (int k = lane; k < n; k += 32) M = fmaxf(M, a.part_ml[((size_t)(c_lo + k + b) * H + h) * 2]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.f;
        for (int k = lane; k < n; k += 32) {
            const float *ml = a.part_ml + ((size_t)(c_lo + k + b) * H + h) * 2;
            const float wgt = ml[0] == -INFINITY ? 0.f : exp2f(ml[0] - M);
            s_w[k] = wgt;
            L = fmaf(ml[1], wgt, L);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (lane == 0) {
            s_c0 = c_lo;
            s_n = n;
            s_M = M;
            s_L = L;
        }
    }
    __syncthreads();
    const int c0 = s_c0, n = s_n;
    float o0 = 0.f, o1 = 0.f;
    for (int k = 0; k < n; ++k) {
        const float wk = s_w[k];
        if (wk == 0.f) continue;
        const float *acc = a.part_acc + ((size_t)(c0 + k + b) * H + h) * kMlaLat;
        o0 = fmaf(wk, acc[tid], o0);
        o1 = fmaf(wk, acc[256 + tid], o1);
    }
    const float L = s_L, inv = L > 0.f ? 1.f / L : 0.f;
    a.out[((int64_t)b * H + h) * kMlaLat + tid] = float_to_bf16_bits(o0 * inv);
    a.out[((int64_t)b * H + h) * kMlaLat + 256 + tid] = float_to_bf16_bits(o1 * inv);
    if (tid == 0 && a.lse != nullptr) a.lse[(int64_t)b * H + h] = L > 0.f ? (s_M + log2f(L)) * kLn2 : -INFINITY;
}

size_t mla_scratch_bytes(int H, int B, int max_rows) {
    (void)max_rows;
    // partial rows: (grid + B) x H x 512 floats for mla_tr_kernel, (grid + 2B) x H x 256 for
    // mla_tile_kernel (no more); (max, sum) pairs for up to grid + 2B segments
    const size_t n_acc = (size_t)kMlaMaxCtas + (size_t)B, n_ml = (size_t)kMlaMaxCtas + 2 * (size_t)B;
    return n_acc * H * kMlaLat * 4 + n_ml * H * 2 * 4 + 256;
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
        e = cudaFuncSetAttribute(mla_tr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTrSmem);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&g_mla_sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_mla_attr[dev] = true;
    }
    const bool tr = H <= kMlaTok;                    // up to 64 heads: the transposed kernel
    MlaArgs a{};
    a.q = q;
    a.kv = kv;
    a.n_tok = n_tok;
    a.rows = rows;
    a.n_rows = n_rows;
    a.max_rows = max_rows;
    a.H = H;
    a.B = B;
    a.halves = tr ? 1 : 2;
    a.n_tiles = (max_rows + kMlaTok - 1) / kMlaTok;
    const int64_t W = (int64_t)B * a.halves * a.n_tiles;
    int sms = g_mla_sms[dev] < kMlaMaxCtas ? g_mla_sms[dev] : kMlaMaxCtas;
    a.grid = (int)(W < sms ? W : sms);
    a.scale_log2 = scale * kLog2e;
    a.part_acc = static_cast<float *>(scratch);
    a.part_ml = a.part_acc + ((size_t)kMlaMaxCtas + (size_t)B) * H * kMlaLat;
    a.out = out;
    a.lse = lse;
    a.hdr = hdr;
    if (a.grid > 0) {
        if (tr)
            mla_tr_kernel<<<a.grid, kTrThreads, kTrSmem, st>>>(a);
        else
            mla_tile_kernel<<<a.grid, kMlaThreads, kMlaSmem, st>>>(a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    } else {
        a.grid = 1;                                  // no rows anywhere: the merge writes zeros
    }
    if (tr)
        mla_merge_tr_kernel<<<dim3(H, B), 256, 0, st>>>(a);
    else
        mla_merge_kernel<<<dim3(H, B), 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa
