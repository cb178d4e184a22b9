// a6 — prefill chunk on the 5th-generation tensor cores (tcgen05, accumulators in TMEM).
//
// "3090x3で 314 万コンテキスト", section "ちなみにこの欠点": each chunk token selects its own
// 2048 tokens, so together they touch nearly the whole history; the fix is to walk the
// history in fixed intervals (outer loop) with all chunk tokens inside (inner loop),
// merging softmax partials as the walk proceeds.
//
// Work unit: a tile of QT consecutive chunk queries x G query heads of one KV head
// (QT x G = 128 rows, the MMA's M). The tile walks the history interval by interval. In
// each interval it marks, per pooled block, which of its queries selected the block (and
// which queries own it as their current, partial block), and compacts the marked blocks
// into a union. The union's tokens go through the tensor cores 64 at a time:
//   S = Q K^T         (M=128, N=64,  K=256)   into TMEM columns [0, 64)
//   softmax rows      one thread per row: each row keeps only the tokens its query may
//                     see (its own selection, or its own block up to itself), online
//                     max/sum in base 2 with a lazy rescale of O (only when the running
//                     max grows by more than 2^8)
//   O += P V          (M=128, N=256, K=64)   into TMEM columns [256, 512)
// Operands sit in shared memory in the 128-byte-swizzled layouts the MMA reads directly:
// Q, K and P K-major, V MN-major. K/V rows are gathered with 16-byte cp.async into two
// buffers whose completion is tracked by mbarriers; MMAs complete onto mbarriers via
// tcgen05.commit. Every wait is bounded (250 ms): a timeout records
// QSA_ERR_DEVICE_TIMEOUT, drains what is in flight (bounded), frees TMEM and returns.
#include "qsa_internal.cuh"
#include "qsa_ptx.cuh"
#include "qsa_tc.cuh"

#include <algorithm>

namespace qsa {

constexpr int kTcThreads = 128;
constexpr int kTcRows = 128;                 // MMA M
constexpr int kTcChunk = 64;                 // tokens per MMA step (N of QK, K of PV)
constexpr int kTcMaxBpi = 2048;              // blocks per sub-interval (8192 tokens)
constexpr int kTcMaxIntervals = 256;
static_assert((int64_t)kTcMaxBpi * kTcMaxIntervals == kPrefillTcMaxBlocks, "tile table limits");
constexpr int kTcMaxQt = 16;                 // queries per tile (G = 8)

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kTcQ = 0;                              // 128 x 256 bf16, K-major   64 KiB
constexpr uint32_t kTcK0 = 65536;                          // 2 x (64 x 256) K-major    2 x 32 KiB
constexpr uint32_t kTcV0 = kTcK0 + 2 * 32768;              // 2 x (64 x 256) MN-major   2 x 32 KiB
constexpr uint32_t kTcP = kTcV0 + 2 * 32768;               // 128 x 64 bf16, K-major     16 KiB
constexpr uint32_t kTcSel = kTcP + 16384;                  // per-block query bits       4 KiB (uint16 x 2048)
constexpr uint32_t kTcUnion = kTcSel + 2 * kTcMaxBpi;      // union block offsets        4 KiB (uint16)
constexpr uint32_t kTcEtab = kTcUnion + 2 * kTcMaxBpi;     // [QT][intervals] list ends  (uint16)
constexpr uint32_t kTcSmem = kTcEtab + 2 * 16 * kTcMaxIntervals + 1024;   // + alignment slack

// OR `bits` into the 16-bit entry i of a shared array (32-bit atomic on the containing word)
__device__ __forceinline__ void sel_or(uint16_t *sel, int i, uint32_t bits) {
    uint32_t *w = reinterpret_cast<uint32_t *>(sel) + (i >> 1);
    atomicOr(w, (bits & 0xFFFFu) << ((i & 1) * 16));
}

struct TcArgs {
    const uint16_t *q;        // [Nc, Hq, 256]
    const uint16_t *k_cache;  // [p0+Nc, Hkv, 256]
    const uint16_t *v_cache;
    const int32_t *blocks;    // [Nc, 512]
    const int32_t *count;     // [Nc]
    uint16_t *out;            // [Nc, Hq, 256]
    float *lse;               // [Nc, Hq] or nullptr
    int32_t p0, Nc, Hq, Hkv;
    int32_t bpi;              // blocks per sub-interval
    int32_t n_iv;             // sub-intervals
    float scale_log2;
    WsHeader *hdr;
};

template <int G>
__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(TcArgs a) {
    constexpr int QT = kTcRows / G;                      // queries per tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(sm);
    uint16_t *sel = reinterpret_cast<uint16_t *>(sm + kTcSel);
    uint16_t *uni = reinterpret_cast<uint16_t *>(sm + kTcUnion);
    uint16_t *etab = reinterpret_cast<uint16_t *>(sm + kTcEtab);

    __shared__ uint64_t bar_s, bar_o, bar_kv[2];
    __shared__ uint32_t tmem_s;
    __shared__ int s_wc[kTcThreads / 32];
    __shared__ uint32_t s_allow[kTcChunk];
    __shared__ int32_t s_cnt[kTcMaxQt];

    const int tid = threadIdx.x, warp = tid >> 5;
    if (warp == 0) tmem_alloc(&tmem_s, 512);
    if (tid == 0) {
        mbar_init(smem_u32(&bar_s), 1);
        mbar_init(smem_u32(&bar_o), 1);
        mbar_init(smem_u32(&bar_kv[0]), kTcThreads);
        mbar_init(smem_u32(&bar_kv[1]), kTcThreads);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_s;
    const uint32_t t_s = tmem + ((uint32_t)(32 * warp) << 16);          // this warp's lanes, S columns
    const uint32_t t_o = t_s + 256;                                      // O columns
    uint32_t n_s = 0, n_o = 0, n_kv[2] = {0, 0};                         // completed phases per barrier
    // A wait that gives up clears `ok` in its thread only; the CTA acts on it at the next
    // __syncthreads_or, so every thread leaves the loops at the same barrier.
    bool ok = true;

    auto wait_bar = [&](uint64_t *bar, uint32_t phase) -> bool {
        if (!mbar_wait_bounded(smem_u32(bar), phase & 1u, kWaitLimitNs)) {
            record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWherePrefill, blockIdx.x);
            return false;
        }
        return true;
    };

    const int n_qt = (a.Nc + QT - 1) / QT;
    const int n_tiles = n_qt * a.Hkv;
    const int row = tid;                         // this thread's MMA row (= TMEM lane)
    const int q_loc = row / G, h_loc = row % G;
    const int64_t last_tok = (int64_t)a.p0 + a.Nc - 1;

    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int qt = tile / a.Hkv, g = tile % a.Hkv;
        const int i0 = qt * QT;
        const int nq = min(QT, a.Nc - i0);
        // ---- tile set-up: query positions, selection counts, Q rows (K-major, swizzled)
        if (tid < QT) {
            int c = tid < nq ? a.count[i0 + tid] : 0;
            const int nbq = tid < nq ? (a.p0 + i0 + tid) >> 2 : 0;
            if (c < 0 || c > kBlockTopK || c > nbq) {
                record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWherePrefill, i0 + tid);
                c = 0;
            }
            s_cnt[tid] = c;
        }
        for (int gi = tid; gi < kTcRows * 32; gi += kTcThreads) {
            const int r = gi >> 5, gg = gi & 31;
            const int qq = r / G, hh = r % G;
            const uint32_t dst = sbase + kTcQ + (gg >> 3) * (kTcRows * 128) + swz(r, gg & 7);
            if (qq < nq) {
                cp_async16(dst, a.q + ((int64_t)(i0 + qq) * a.Hq + g * G + hh) * kHeadDim + gg * 8);
            } else {
                asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0) : "memory");
            }
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        // ---- list ends per (query, sub-interval): etab[q][v] = first list index in interval > v
        for (int i = tid; i < QT * a.n_iv; i += kTcThreads) etab[i] = 0xFFFFu;
        __syncthreads();
        // (the lists must be strictly ascending below the query's own block: anything else
        // is recorded as a bounds error, so no entry is dropped silently)
        for (int qq = 0; qq < nq; ++qq) {
            const int32_t *lst = a.blocks + (int64_t)(i0 + qq) * kBlockTopK;
            const int c = s_cnt[qq];
            const int nbq = (a.p0 + i0 + qq) >> 2;
            for (int i = tid; i < c; i += kTcThreads) {
                const int b = lst[i];
                const int bn = i + 1 < c ? lst[i + 1] : nbq;
                if (b < 0 || bn <= b || bn > nbq) {
                    record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWherePrefill, i0 + qq);
                    continue;
                }
                const int v = b / a.bpi;
                if (i + 1 == c || bn / a.bpi != v) etab[qq * a.n_iv + v] = (uint16_t)(i + 1);
            }
        }
        __syncthreads();
        if (tid < QT) {                          // intervals without entries end where the previous one did
            uint16_t run = 0;
            for (int v = 0; v < a.n_iv; ++v) {
                const uint16_t e = etab[tid * a.n_iv + v];
                if (e != 0xFFFFu) run = e;
                etab[tid * a.n_iv + v] = run;
            }
        }
        __syncthreads();

        // per-row softmax state (rows of queries past the chunk end stay fully masked)
        float m_ref = -INFINITY, l_sum = 0.f;
        bool o_init = false;
        const int nb_last = (a.p0 + i0 + nq - 1) >> 2;           // the tile's highest own block
        const int n_iv_tile = min(a.n_iv, nb_last / a.bpi + 1);

        for (int v = 0; v < n_iv_tile && ok; ++v) {
            const int b_lo = v * a.bpi;
            const int b_hi = min(b_lo + a.bpi, nb_last + 1);
            // ---- mark the blocks of this interval each query selected or owns
            for (int i = tid; i < a.bpi; i += kTcThreads) sel[i] = 0;
            __syncthreads();
            for (int qq = 0; qq < nq; ++qq) {
                const int32_t *lst = a.blocks + (int64_t)(i0 + qq) * kBlockTopK;
                const int e0 = v == 0 ? 0 : etab[qq * a.n_iv + v - 1];
                const int e1 = etab[qq * a.n_iv + v];
                const int nbq = (a.p0 + i0 + qq) >> 2;
                for (int i = e0 + tid; i < e1; i += kTcThreads) {
                    const int b = lst[i];
                    if (b < 0 || b >= nbq || b < b_lo || b >= b_hi) {
                        record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWherePrefill, i0 + qq);
                        continue;
                    }
                    sel_or(sel, b - b_lo, 1u << qq);
                }
                if (tid == 0 && nbq >= b_lo && nbq < b_hi) sel_or(sel, nbq - b_lo, 1u << qq);   // own block
            }
            __syncthreads();
            // ---- compact the marked blocks into the union, ascending (ballot + warp-count scan)
            int nu = 0;
            for (int base_i = 0; base_i < b_hi - b_lo; base_i += kTcThreads) {
                const int i = base_i + tid;
                const bool m = i < b_hi - b_lo && sel[i] != 0;
                const unsigned bal = __ballot_sync(0xffffffffu, m);
                if ((tid & 31) == 0) s_wc[warp] = __popc(bal);
                __syncthreads();
                int before = nu, total = 0;
#pragma unroll
                for (int w = 0; w < kTcThreads / 32; ++w) {
                    if (w < warp) before += s_wc[w];
                    total += s_wc[w];
                }
                if (m) uni[before + __popc(bal & ((1u << (tid & 31)) - 1u))] = (uint16_t)i;
                nu += total;
                __syncthreads();
            }
            const int n_ch = (nu + kTcChunk / kRatio - 1) / (kTcChunk / kRatio);

            // ---- gather of chunk c's K and V rows into buffer c & 1 (64 tokens x 256 dims each)
            auto gather = [&](int c) {
                const int buf = c & 1;
                const int ub0 = c * (kTcChunk / kRatio);
                for (int gi = tid; gi < kTcChunk * 64; gi += kTcThreads) {
                    const int j = gi >> 6;                 // token within the chunk
                    const int rem = gi & 63;
                    const int is_v = rem >> 5, gg = rem & 31;
                    int ui = ub0 + (j >> 2);
                    if (ui >= nu) ui = ub0;                // padding column: any valid token (masked)
                    // the newest block may extend past the last token; its tail is masked
                    const int64_t tok = min((int64_t)(b_lo + uni[ui]) * kRatio + (j & 3), last_tok);
                    const uint16_t *src = (is_v ? a.v_cache : a.k_cache) + (tok * a.Hkv + g) * kHeadDim + gg * 8;
                    const uint32_t dst = sbase + (is_v ? kTcV0 : kTcK0) + buf * 32768 + (gg >> 3) * (kTcChunk * 128) +
                                         swz(j, gg & 7);
                    cp_async16(dst, src);
                }
                cp_async_arrive(smem_u32(&bar_kv[buf]));
            };
            if (n_ch > 0) {
                // the previous chunk's PV may still read the buffer gather(0) refills
                if (o_init && !wait_bar(&bar_o, n_o - 1)) ok = false;
                gather(0);
            }

            for (int c = 0; c < n_ch; ++c) {
                const int buf = c & 1;
                // the other buffer is free once the previous chunk's PV finished
                if (c + 1 < n_ch) {
                    if (o_init && !wait_bar(&bar_o, n_o - 1)) ok = false;
                    gather(c + 1);
                }
                // column info: token ids and which queries may see them
                if (tid < kTcChunk) {
                    const int j = tid;
                    const int ui = c * (kTcChunk / kRatio) + (j >> 2);
                    uint32_t allow = 0u;
                    if (ui < nu) {
                        const int blk = b_lo + uni[ui];
                        const int tok = blk * kRatio + (j & 3);
                        allow = sel[uni[ui]];
                        // an owner sees its own block only up to itself
                        for (int qq = 0; qq < nq; ++qq) {
                            const int pq = a.p0 + i0 + qq;
                            if ((pq >> 2) == blk && tok > pq) allow &= ~(1u << qq);
                        }
                    }
                    s_allow[j] = allow;
                }
                if (!wait_bar(&bar_kv[buf], n_kv[buf])) ok = false;
                ++n_kv[buf];
                fence_proxy_async_smem();
                tc_fence_before();
                if (__syncthreads_or(!ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (tid == 0) {               // S = Q K^T
                    const uint32_t qa = sbase + kTcQ, kb = sbase + kTcK0 + buf * 32768;
#pragma unroll
                    for (int s = 0; s < kHeadDim / 16; ++s) {
                        const uint64_t ad = tc_desc(qa + (s >> 2) * (kTcRows * 128) + (s & 3) * 32, 16, 1024);
                        const uint64_t bd = tc_desc(kb + (s >> 2) * (kTcChunk * 128) + (s & 3) * 32, 16, 1024);
                        tc_mma(tmem, ad, bd, tc_idesc(kTcRows, kTcChunk, 0), s > 0);
                    }
                    tc_commit(smem_u32(&bar_s));
                }
                if (!wait_bar(&bar_s, n_s)) ok = false;
                ++n_s;
                // the previous PV must be done before P is rewritten or O rescaled
                if (o_init && !wait_bar(&bar_o, n_o - 1)) ok = false;
                tc_fence_after();
                // ---- softmax of this thread's row
                float x[kTcChunk];
                {
                    float t0[32], t1[32];
                    tmem_ld32(t_s, t0);
                    tmem_ld32(t_s + 32, t1);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        x[j] = (s_allow[j] >> q_loc) & 1u ? t0[j] * a.scale_log2 : -INFINITY;
                        x[j + 32] = (s_allow[j + 32] >> q_loc) & 1u ? t1[j] * a.scale_log2 : -INFINITY;
                    }
                }
                float cmax = -INFINITY;
#pragma unroll
                for (int j = 0; j < kTcChunk; ++j) cmax = fmaxf(cmax, x[j]);
                // lazy rescale: move the reference only when the row max grew by more than 2^8
                float f = 1.f;
                if (cmax > m_ref + 8.f) {
                    if (m_ref != -INFINITY) f = exp2f(m_ref - cmax);
                    m_ref = cmax;
                }
                l_sum *= f;
                // TMEM loads and stores are warp-collective: the warp rescales together
                if (o_init && __any_sync(0xffffffffu, f != 1.f)) {
#pragma unroll 1
                    for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
                        float ov[32];
                        tmem_ld32(t_o + c0, ov);
#pragma unroll
                        for (int j = 0; j < 32; ++j) ov[j] *= f;
                        tmem_st32(t_o + c0, ov);
                    }
                }
                float psum = 0.f;
                uint32_t pk[kTcChunk / 2];
#pragma unroll
                for (int j = 0; j < kTcChunk; j += 2) {
                    const float e0 = x[j] == -INFINITY ? 0.f : exp2f(x[j] - m_ref);
                    const float e1 = x[j + 1] == -INFINITY ? 0.f : exp2f(x[j + 1] - m_ref);
                    const uint16_t b0 = float_to_bf16_bits(e0), b1 = float_to_bf16_bits(e1);
                    psum += e0 + e1;          // fp32 row sum: the LSE stays exact to fp32 rounding
                    pk[j / 2] = (uint32_t)b0 | ((uint32_t)b1 << 16);
                }
                l_sum += psum;
#pragma unroll
                for (int gg = 0; gg < 8; ++gg) {
                    const uint32_t dst = sbase + kTcP + swz(row, gg);
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(pk[gg * 4]),
                                 "r"(pk[gg * 4 + 1]), "r"(pk[gg * 4 + 2]), "r"(pk[gg * 4 + 3])
                                 : "memory");
                }
                fence_proxy_async_smem();
                tc_fence_before();
                if (__syncthreads_or(!ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (tid == 0) {               // O += P V
                    const uint32_t pa = sbase + kTcP, vb = sbase + kTcV0 + buf * 32768;
#pragma unroll
                    for (int s = 0; s < kTcChunk / 16; ++s) {
                        const uint64_t ad = tc_desc(pa + s * 32, 16, 1024);
                        const uint64_t bd = tc_desc(vb + s * 2048, kTcChunk * 128, 1024);
                        tc_mma(tmem + 256, ad, bd, tc_idesc(kTcRows, kHeadDim, 1), o_init || s > 0);
                    }
                    tc_commit(smem_u32(&bar_o));
                }
                ++n_o;
                o_init = true;
            }
        }
        if (!ok) break;
        // ---- finish the tile: O / l -> bf16, lse
        if (o_init && !wait_bar(&bar_o, n_o - 1)) ok = false;
        if (__syncthreads_or(!ok)) {
            ok = false;
            break;
        }
        tc_fence_after();
        if (o_init) {                            // every valid row saw at least its own token
            const bool store = q_loc < nq && l_sum > 0.f;
            const float inv = store ? 1.f / l_sum : 0.f;
            uint16_t *dst = a.out + ((int64_t)(i0 + q_loc) * a.Hq + g * G + h_loc) * kHeadDim;
#pragma unroll 1
            for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
                float ov[32];
                tmem_ld32(t_o + c0, ov);          // warp-collective: every lane loads
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    w[j] = (uint32_t)float_to_bf16_bits(ov[2 * j] * inv) |
                           ((uint32_t)float_to_bf16_bits(ov[2 * j + 1] * inv) << 16);
                if (store) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<uint4 *>(dst + c0 + 8 * j) =
                            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                }
            }
            if (store && a.lse != nullptr)
                a.lse[(int64_t)(i0 + q_loc) * a.Hq + g * G + h_loc] = (m_ref + log2f(l_sum)) * kLn2;
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    if (!ok) {
        // drain: the last commits may still be in flight (bounded waits), then free TMEM
        if (n_s > 0) mbar_wait_bounded(smem_u32(&bar_s), (n_s - 1) & 1u, kWaitLimitNs);
        if (n_o > 0) mbar_wait_bounded(smem_u32(&bar_o), (n_o - 1) & 1u, kWaitLimitNs);
        asm volatile("cp.async.wait_all;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

bool prefill_tc_supported(int Hq, int Hkv) {
    const int G = Hkv > 0 ? Hq / Hkv : 0;
    return G == 8 || G == 16;
}

cudaError_t launch_prefill_tc(const AttnArgs &a, int interval_tokens, WsHeader *hdr, cudaStream_t st) {
    TcArgs t{};
    t.q = a.q;
    t.k_cache = a.k_cache;
    t.v_cache = a.v_cache;
    t.blocks = a.blocks;
    t.count = a.count;
    t.out = a.out;
    t.lse = a.lse;
    t.p0 = a.p0;
    t.Nc = a.rows;
    t.Hq = a.n_q_heads;
    t.Hkv = a.n_kv_heads;
    t.scale_log2 = a.scale_log2;
    t.hdr = hdr;
    const int64_t n_blocks = ((int64_t)a.p0 + a.rows) / kRatio + 1;
    // the interval sets the evaluation order only; it is clamped to what the on-chip tables hold
    int64_t bpi = std::min<int64_t>(interval_tokens / kRatio, kTcMaxBpi);
    bpi = std::max<int64_t>(bpi, (n_blocks + kTcMaxIntervals - 1) / kTcMaxIntervals);
    if (bpi > kTcMaxBpi) return cudaErrorInvalidValue;
    t.bpi = (int)bpi;
    t.n_iv = (int)((n_blocks + bpi - 1) / bpi);
    const int G = a.n_q_heads / a.n_kv_heads;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int n_tiles = ((a.rows + kTcRows / G - 1) / (kTcRows / G)) * a.n_kv_heads;
    const int grid = std::max(1, std::min(sms, n_tiles));
    switch (G) {
        case 8:
            e = cudaFuncSetAttribute(prefill_tc_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
            if (e != cudaSuccess) return e;
            prefill_tc_kernel<8><<<grid, kTcThreads, kTcSmem, st>>>(t);
            break;
        case 16:
            e = cudaFuncSetAttribute(prefill_tc_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
            if (e != cudaSuccess) return e;
            prefill_tc_kernel<16><<<grid, kTcThreads, kTcSmem, st>>>(t);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace qsa
