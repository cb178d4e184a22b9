// a6 — prefill chunk on the 5th-generation tensor cores (tcgen05, accumulators in TMEM).
//
// "3090x3で 314 万コンテキスト", section "ちなみにこの欠点": each chunk token selects its own
// 2048 tokens, so together they touch nearly the whole history; the fix is to walk the
// history in fixed intervals (outer loop) with all chunk tokens inside (inner loop),
// merging softmax partials as the walk proceeds.
//
// Work unit: a tile of QT consecutive chunk queries x G query heads of one KV head
// (QT x G = 128 rows, the MMA's M). Two kernels:
//
// 1. Plan (one CTA per query tile, shared by its KV heads). Walking the history interval
//    by interval, it marks per pooled block which of the tile's queries selected it (or
//    own it as their current, partial block), and places the marked blocks of every interval
//    in the tile's ascending union, cut into chunks of 16 blocks (64 tokens; a chunk may
//    straddle two intervals, so only the tile's last chunk is partial). Each chunk record
//    holds the 16 block ids and,
//    per query, a 64-bit word of the tokens it may see (its own selection; its own block
//    only up to itself).
//
// 2. Attention (one CTA per SM, persistent over tiles), per chunk g:
//      S = Q K^T         (M=128, N=64,  K=256)   into TMEM columns [64 (g%2), +64)
//      softmax rows      one thread per row, online max/sum in base 2 with a lazy rescale
//                        of O (only when the running max grows by more than 2^8)
//      O += P V          (M=128, N=256, K=64)    into TMEM columns [256, 512)
//    Roles (512 threads):
//      warps 0-3   softmax: one row per thread; at a tile's end, O / l -> bf16 and the LSE;
//      warps 4-9   K producers: the leading thread bulk-copies chunk records two ahead; the
//                  six warps load each new tile's Q rows and every chunk's K rows (64 tokens
//                  x 512 bytes) as 16-byte cp.async into 128-byte-swizzled shared memory,
//                  two stages;
//      warps 10-14 V producers: the V rows the same way into their own two stages. Each
//                  producer warp follows the mbarriers on its own, so a slow warp holds back
//                  no other; many issuing warps make rows arrive faster, since one warp's
//                  cp.async issue stalls on the memory system;
//      warp 15     one thread issues the MMAs: QK of chunk g+1 before PV of chunk g, so the
//                  tensor core computes the next scores while the softmax runs.
//    Hand-offs are mbarriers (cp.async arrivals, tcgen05.commit, thread arrivals).
// Every wait is bounded (250 ms): a timeout records QSA_ERR_DEVICE_TIMEOUT and raises a CTA
// flag; each role leaves its loops where all its threads agree, drains what it issued
// (bounded), and TMEM is freed after a final barrier.
#include "qsa_internal.cuh"
#include "qsa_ptx.cuh"
#include "qsa_tc.cuh"

#include <algorithm>

namespace qsa {

constexpr int kTcRows = 128;                 // MMA M
constexpr int kTcChunk = 64;                 // tokens per chunk (N of QK, K of PV)
constexpr int kTcBlocksPerChunk = kTcChunk / kRatio;
constexpr int kTcMaxBpi = 2048;              // blocks per sub-interval (8192 tokens)
constexpr int kTcMaxIntervals = 256;
static_assert((int64_t)kTcMaxBpi * kTcMaxIntervals == kPrefillTcMaxBlocks, "tile table limits");
constexpr int kTcMaxQt = 16;                 // queries per tile (G = 8)

// ----------------------------------------------------------------------------- plan

struct ChunkRec {                            // 256 bytes
    int32_t blk[kTcBlocksPerChunk];          // block ids (-1: padding)
    uint32_t vis[kTcMaxQt][2];               // per query: tokens it may see (bit j = token j), lo/hi
    int32_t first, last;                     // first / last chunk of the tile
    int32_t pad[14];
};
static_assert(sizeof(ChunkRec) == 256, "chunk record size");
constexpr int kRecCopyBytes = 208;           // blk, vis, flags
// chunks per tile: the union has at most QT * (512 + 1) blocks (the bound keeps a chunk of slack per interval)
constexpr int kPlanCap = (kTcMaxQt * (kBlockTopK + 1) + kTcBlocksPerChunk - 1) / kTcBlocksPerChunk + kTcMaxIntervals;
constexpr int kPlanThreads = 384;                // 12 warps: two CTAs fit an SM
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kStartStride = kTcMaxIntervals + 8;

// dynamic shared memory of the plan kernel
constexpr uint32_t kPlLists = 0;                                           // int32 [QT][512]
constexpr uint32_t kPlStart = kPlLists + 4 * kTcMaxQt * kBlockTopK;        // uint16 [QT][intervals + 1]
constexpr uint32_t kPlCounts = kPlStart + 2 * kTcMaxQt * kStartStride;     // int32 [intervals + 1]
constexpr uint32_t kPlMasks = kPlCounts + 4 * (kTcMaxIntervals + 8);       // uint16 [warp][2048]
constexpr uint32_t kPlBits = kPlMasks + 2 * kTcMaxBpi * kPlanWarps;         // uint32 [warp][64]: marked blocks
constexpr uint32_t kPlSmem = kPlBits + 4 * (kTcMaxBpi / 32) * kPlanWarps;

static size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// plan layout: chunk counts [n_qt], the dealt tile order [< 2 * n_tiles], chunk records [n_qt][kPlanCap]
size_t prefill_tc_plan_bytes(int Nc, int Hq, int Hkv) {
    if (!prefill_tc_supported(Hq, Hkv) || Nc <= 0) return 0;
    const int QT = kTcRows / (Hq / Hkv);
    const size_t n_qt = (size_t)(Nc + QT - 1) / QT;
    return round256(n_qt * 4) + round256(n_qt * Hkv * 2 * 4) + n_qt * kPlanCap * sizeof(ChunkRec);
}

// One CTA: query tiles sorted by chunk count, largest first (counting sort), and their (tile, KV
// head) work items dealt to the CTAs in snake order: round r goes left to right when r is even,
// right to left when odd, so every CTA's summed load stays close to the mean.
constexpr int kOrderThreads = 1024;
__global__ void __launch_bounds__(kOrderThreads) prefill_order_kernel(const int32_t *n_chunks, int n_qt, int Hkv,
                                                                      int grid, int n_rounds, int32_t *order) {
    __shared__ int base[kPlanCap + 1];
    for (int i = threadIdx.x; i <= kPlanCap; i += blockDim.x) base[i] = 0;
    __syncthreads();
    for (int q = threadIdx.x; q < n_qt; q += blockDim.x) atomicAdd(&base[min(max(n_chunks[q], 0), kPlanCap)], 1);
    __syncthreads();
    if (threadIdx.x < 32) {      // base[s] = query tiles with more than s chunks (one warp, sizes descending)
        const int lane = threadIdx.x;
        constexpr int kPer = (kPlanCap + 1 + 31) / 32;
        int v[kPer], sum = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int s = kPlanCap - (lane * kPer + j);
            v[j] = s >= 0 ? base[s] : 0;
            sum += v[j];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int run = incl - sum;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int s = kPlanCap - (lane * kPer + j);
            if (s >= 0) base[s] = run;
            run += v[j];
        }
    }
    __syncthreads();
    auto slot = [&](int k) -> int {      // position of sorted work item k in the [round][CTA] table
        const int r = k / grid, c = k - r * grid;
        return r * grid + ((r & 1) ? grid - 1 - c : c);
    };
    for (int q = threadIdx.x; q < n_qt; q += blockDim.x) {
        const int rank = atomicAdd(&base[min(max(n_chunks[q], 0), kPlanCap)], 1);
        for (int h = 0; h < Hkv; ++h) order[slot(rank * Hkv + h)] = q * Hkv + h;
    }
    for (int k = n_qt * Hkv + threadIdx.x; k < n_rounds * grid; k += blockDim.x) order[slot(k)] = -1;
}

struct PlanArgs {
    const int32_t *blocks;    // [Nc, 512]
    const int32_t *count;     // [Nc]
    int32_t p0, Nc, QT, bpi, n_iv;
    int32_t *n_chunks;        // [n_qt]
    ChunkRec *recs;           // [n_qt][kPlanCap]
    WsHeader *hdr;
};

__device__ __forceinline__ void sel_or(uint16_t *sel, int i, uint32_t bits) {
    uint32_t *w = reinterpret_cast<uint32_t *>(sel) + (i >> 1);
    atomicOr(w, (bits & 0xFFFFu) << ((i & 1) * 16));
}

// One CTA per query tile; warps take intervals v = warp, warp + 8, ... in two passes
// (chunk counts, then records at the scanned offsets).
__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(PlanArgs a) {
    extern __shared__ __align__(16) uint8_t psm[];
    int32_t *lists = reinterpret_cast<int32_t *>(psm + kPlLists);
    uint16_t *start = reinterpret_cast<uint16_t *>(psm + kPlStart);
    int32_t *counts = reinterpret_cast<int32_t *>(psm + kPlCounts);
    __shared__ int32_t s_cnt[kTcMaxQt], s_p[kTcMaxQt];
    __shared__ int s_bad, s_total;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint16_t *m = reinterpret_cast<uint16_t *>(psm + kPlMasks) + warp * kTcMaxBpi;
    uint32_t *bits = reinterpret_cast<uint32_t *>(psm + kPlBits) + warp * (kTcMaxBpi / 32);
    const int qt = blockIdx.x, QT = a.QT;
    const int i0 = qt * QT, nq = min(QT, a.Nc - i0);
    const int nb_last = (a.p0 + i0 + nq - 1) >> 2;
    const int n_iv_tile = min(a.n_iv, nb_last / a.bpi + 1);
    if (tid < QT) {
        int c = 0;
        const int p = a.p0 + i0 + tid;
        if (tid < nq) {
            c = a.count[i0 + tid];
            if (c < 0 || c > kBlockTopK || c > (p >> 2)) {
                record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWherePrefill, i0 + tid);
                c = 0;
            }
        }
        s_cnt[tid] = c;
        s_p[tid] = tid < nq ? p : -1;
    }
    if (tid == 0) s_bad = 0;
    __syncthreads();
    // ---- the tile's lists; each must be strictly ascending below the query's own block
    // (16-byte asynchronous copies, all in flight at once; entries past a count are unused)
    for (int e = tid; e < QT * kBlockTopK / 4; e += kPlanThreads) {
        const int qq = (4 * e) / kBlockTopK;
        if (qq < nq) cp_async16(smem_u32(lists + 4 * e), a.blocks + (int64_t)(i0 + qq) * kBlockTopK + (4 * e) % kBlockTopK);
    }
    cp_async_wait_all();
    __syncthreads();
    for (int e = tid; e < QT * kBlockTopK; e += kPlanThreads) {
        const int qq = e / kBlockTopK, i = e % kBlockTopK;
        const int c = s_cnt[qq];
        if (i < c) {
            const int b = lists[e];
            const int bn = i + 1 < c ? lists[e + 1] : (s_p[qq] >> 2);
            if (b < 0 || bn <= b) {
                record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWherePrefill, i0 + qq);
                s_bad = 1;
            }
        }
    }
    __syncthreads();
    if (s_bad) {                               // nothing is attended for this tile
        if (tid == 0) a.n_chunks[qt] = 0;
        return;
    }
    // ---- start[q][v]: first list index with block >= v * bpi (binary search)
    for (int e = tid; e < QT * (n_iv_tile + 1); e += kPlanThreads) {
        const int qq = e / (n_iv_tile + 1), v = e % (n_iv_tile + 1);
        const int32_t *l = lists + qq * kBlockTopK;
        int lo = 0, hi = s_cnt[qq];
        const int key = v * a.bpi;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (l[mid] < key) lo = mid + 1;
            else hi = mid;
        }
        start[qq * kStartStride + v] = (uint16_t)lo;
    }
    __syncthreads();

    // marks of interval v in this warp's mask array; returns how many blocks are marked
    auto mark = [&](int v) -> int {
        const int b_lo = v * a.bpi;
        const int span = min(b_lo + a.bpi, nb_last + 1) - b_lo;
        uint4 *m4 = reinterpret_cast<uint4 *>(m);
        for (int i = lane; i < kTcMaxBpi / 8; i += 32) m4[i] = make_uint4(0, 0, 0, 0);
        bits[lane] = 0u;
        bits[lane + 32] = 0u;
        __syncwarp();
        // per block: which of the tile's queries take it (mask), and that it is marked (bit)
        auto mark_one = [&](int i, uint32_t q_bit) {
            sel_or(m, i, q_bit);
            atomicOr(&bits[i >> 5], 1u << (i & 31));
        };
        for (int qq = 0; qq < nq; ++qq) {
            const int e0 = start[qq * kStartStride + v], e1 = start[qq * kStartStride + v + 1];
            for (int i = e0 + lane; i < e1; i += 32) mark_one(lists[qq * kBlockTopK + i] - b_lo, 1u << qq);
        }
        if (lane < nq) {
            const int nbq = s_p[lane] >> 2;
            if (nbq >= b_lo && nbq - b_lo < span) mark_one(nbq - b_lo, 1u << lane);   // own block
        }
        __syncwarp();
        return (int)__reduce_add_sync(0xffffffffu, (unsigned)(__popc(bits[lane]) + __popc(bits[lane + 32])));
    };

    // ---- pass 1: union blocks per interval
    for (int v = warp; v < n_iv_tile; v += kPlanWarps) {
        const int nu = mark(v);
        if (lane == 0) counts[v] = nu;
    }
    __syncthreads();
    if (warp == 0) {                           // exclusive scan over the intervals
        constexpr int per = (kTcMaxIntervals + 31) / 32;
        int loc[per], sum = 0;
#pragma unroll
        for (int k = 0; k < per; ++k) {
            const int v = lane * per + k;
            loc[k] = v < n_iv_tile ? counts[v] : 0;
            sum += loc[k];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        __syncwarp();
        int run = incl - sum;
#pragma unroll
        for (int k = 0; k < per; ++k) {
            const int v = lane * per + k;
            if (v < n_iv_tile) counts[v] = run;
            run += loc[k];
        }
        if (lane == 31) s_total = incl;
    }
    __syncthreads();
    // the tile's union in ascending block order, cut into chunks of 16 blocks: a chunk may
    // straddle two intervals (the intervals set the walk's order, not the chunking)
    const int total = (s_total + kTcBlocksPerChunk - 1) / kTcBlocksPerChunk;
    if (total > kPlanCap) {                    // cannot happen for valid lists; stop cleanly
        if (tid == 0) {
            record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWherePrefill, i0);
            a.n_chunks[qt] = 0;
        }
        return;
    }
    // ---- the records start as blk = -1, visibility 0, with the tile's first / last flags
    ChunkRec *out = a.recs + (size_t)qt * kPlanCap;
    for (int e = tid; e < total * (int)(sizeof(ChunkRec) / 16); e += kPlanThreads) {
        const int c = e / (int)(sizeof(ChunkRec) / 16), w = e % (int)(sizeof(ChunkRec) / 16);
        uint4 val = make_uint4(0, 0, 0, 0);
        if (w < kTcBlocksPerChunk / 4) val = make_uint4(~0u, ~0u, ~0u, ~0u);
        if (w == (int)(offsetof(ChunkRec, first) / 16))
            reinterpret_cast<int32_t *>(&val)[(offsetof(ChunkRec, first) % 16) / 4] = c == 0;
        if (w == (int)(offsetof(ChunkRec, last) / 16))
            reinterpret_cast<int32_t *>(&val)[(offsetof(ChunkRec, last) % 16) / 4] = c == total - 1;
        reinterpret_cast<uint4 *>(out + c)[w] = val;
    }
    __syncthreads();
    // ---- pass 2: every marked block at its position in the tile's union
    for (int v = warp; v < n_iv_tile; v += kPlanWarps) {
        const int b_lo = v * a.bpi;
        mark(v);
        const int off = counts[v];             // union blocks of the earlier intervals
        // the marked blocks in ascending order: lane l takes the bit words 2 l and 2 l + 1
        // (blocks [64 l, 64 l + 64) of the interval); a warp scan of their counts places each
        const uint32_t w0 = bits[2 * lane], w1 = bits[2 * lane + 1];
        const int cnt = __popc(w0) + __popc(w1);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int pos = off + incl - cnt;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            for (uint32_t bb = h ? w1 : w0; bb != 0u; bb &= bb - 1u) {
                const int i = 64 * lane + 32 * h + __ffs(bb) - 1;
                const uint32_t mk = m[i];
                ChunkRec *r = out + pos / kTcBlocksPerChunk;
                const int slot = pos % kTcBlocksPerChunk, b = b_lo + i;
                r->blk[slot] = b;
                for (uint32_t mm = mk; mm != 0; mm &= mm - 1u) {
                    const int qq = __ffs(mm) - 1;
                    uint32_t vbits = 0xFu;
                    const int p = s_p[qq];
                    if ((p >> 2) == b) vbits = (1u << ((p & 3) + 1)) - 1u;   // its own block: up to itself
                    atomicOr(&r->vis[qq][slot >> 3], vbits << ((slot & 7) * 4));
                }
                ++pos;
            }
        }
    }
    if (tid == 0) a.n_chunks[qt] = total;
}

// ----------------------------------------------------------------------------- attention

constexpr int kTcSoftmaxThreads = 128;
constexpr int kTcKWarps = 6, kTcVWarps = 5;  // producer warps for K (and Q, records) and for V
constexpr int kTcProducerWarps = kTcKWarps + kTcVWarps;
constexpr int kTcMmaWarp = 4 + kTcProducerWarps;
constexpr int kTcThreads = kTcSoftmaxThreads + kTcProducerWarps * 32 + 32;
constexpr int kTcRing = 4;                   // chunk records in flight

// shared memory layout (offsets from a 1024-byte aligned base)
constexpr uint32_t kTcQ = 0;                              // 128 x 256 bf16, K-major    64 KiB
constexpr int kTcKStages = 2, kTcVStages = 2;
constexpr uint32_t kTcK = 65536;                           // stages of 64 x 256, K-major    32 KiB each
constexpr uint32_t kTcV = kTcK + kTcKStages * 32768;       // stages of 64 x 256, MN-major   32 KiB each
constexpr uint32_t kTcRecs = kTcV + kTcVStages * 32768;    // ChunkRec [ring]
// tensor memory columns: S (2 x 64 fp32), P (2 x 64 bf16 = 2 x 32), O (256 fp32)
constexpr uint32_t kTcTmemS = 0, kTcTmemP = 128, kTcTmemO = 256;
constexpr uint32_t kTcSmem = kTcRecs + sizeof(ChunkRec) * kTcRing + 1024;   // + alignment slack
static_assert(kTcSmem + 1024 <= 227 * 1024, "shared memory per CTA (dynamic + static)");

struct TcArgs {
    const uint16_t *q;        // [Nc, Hq, 256]
    const uint16_t *k_cache;  // [p0+Nc, Hkv, 256]
    const uint16_t *v_cache;
    uint16_t *out;            // [Nc, Hq, 256]
    float *lse;               // [Nc, Hq] or nullptr
    const int32_t *n_chunks;  // [n_qt] (plan)
    const ChunkRec *recs;     // [n_qt][kPlanCap] (plan)
    const int32_t *order;     // [rounds][grid] tiles dealt to the CTAs (plan), -1 past the end
    int32_t p0, Nc, Hq, Hkv;
    float scale_log2;
    WsHeader *hdr;
};

// registers per thread: each of the 4 schedulers holds 16K registers for its share of the
// CTA's warps (one CTA per SM)
constexpr int kTcMaxRegs = (16384 / (((kTcThreads / 32 + 3) / 4) * 32)) & ~7;
static_assert(kTcThreads % 128 == 0, "whole warps on every scheduler");

template <int G>
__global__ void __maxnreg__(kTcMaxRegs) prefill_tc_kernel(TcArgs a) {
    constexpr int QT = kTcRows / G;                      // queries per tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(sm);
    ChunkRec *ring = reinterpret_cast<ChunkRec *>(sm + kTcRecs);

    __shared__ uint64_t k_full[kTcKStages], k_empty[kTcKStages], v_full[kTcVStages], v_empty[kTcVStages], s_full[2];
    __shared__ uint64_t r_full[kTcRing], r_empty[kTcRing];
    __shared__ uint64_t p_full[2], pv_done[2];
    __shared__ uint64_t q_full, q_free, o_free;
    __shared__ uint32_t tmem_s;
    __shared__ volatile int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (warp == kTcMmaWarp) tmem_alloc(&tmem_s, 512);
    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&s_full[s]), 1);
        }
        for (int s = 0; s < kTcKStages; ++s) {
            mbar_init(smem_u32(&k_full[s]), kTcKWarps * 32);           // cp.async arrivals
            mbar_init(smem_u32(&k_empty[s]), 1);
        }
        for (int s = 0; s < kTcVStages; ++s) {
            mbar_init(smem_u32(&v_full[s]), kTcVWarps * 32);
            mbar_init(smem_u32(&v_empty[s]), 1);
        }
        for (int s = 0; s < kTcRing; ++s) {
            mbar_init(smem_u32(&r_full[s]), 1);                        // bulk copy of the record
            mbar_init(smem_u32(&r_empty[s]), kTcSoftmaxThreads + kTcProducerWarps);   // readers
        }
        mbar_init(smem_u32(&q_full), 2 * kTcKWarps * 32);          // cp.async + thread arrivals
        mbar_init(smem_u32(&q_free), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&p_full[s]), kTcSoftmaxThreads);
            mbar_init(smem_u32(&pv_done[s]), 1);
        }
        mbar_init(smem_u32(&o_free), kTcSoftmaxThreads);
        fence_mbar_init();
        s_abort = 0;
    }
    // the K and V stages start as zeros: a chunk's padding columns are not loaded, so they
    // hold zeros or an earlier chunk's rows, finite either way (masked in S, P = 0 against V)
    for (uint32_t i = tid; i < (kTcKStages + kTcVStages) * 32768u / 16u; i += kTcThreads)
        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(sbase + kTcK + 16u * i), "r"(0) : "memory");
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_s;
    const int n_qt = (a.Nc + QT - 1) / QT;
    const int n_tiles = n_qt * a.Hkv;
    // this CTA's tiles: one per round of the dealt order (largest first), -1 past the end
    const int n_rounds = (n_tiles + (int)gridDim.x - 1) / (int)gridDim.x;
    auto tile_at = [&](int r) -> int { return r < n_rounds ? a.order[(size_t)r * gridDim.x + blockIdx.x] : -1; };
    auto size_at = [&](int t) -> int { return t >= 0 ? a.n_chunks[t / a.Hkv] : 0; };
    // to the next chunk of a stream (round r, tile t, chunk c of n), skipping tiles without chunks
    auto advance = [&](int &r, int &t, int &c, int &n) {
        ++c;
        while (r < n_rounds && c >= n) {
            ++r;
            t = tile_at(r);
            c = 0;
            n = size_at(t);
        }
    };

    auto wait = [&](uint64_t *bar, uint32_t phase) -> bool {
        if (mbar_wait_bounded(smem_u32(bar), phase & 1u, kWaitLimitNs)) return true;
        record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWherePrefill, blockIdx.x);
        s_abort = 1;
        return false;
    };

    // a warp's wait: every lane polls; the warp goes on only if all saw the phase and no role
    // has given up
    auto wait_warp = [&](uint64_t *bar, uint32_t phase) -> bool {
        const bool w = wait(bar, phase);
        return __all_sync(0xffffffffu, w) && !__any_sync(0xffffffffu, s_abort != 0);
    };

    if (warp >= 4 && warp < kTcMmaWarp) {
        // ================================================================ producers (cp.async)
        // K warps: records (bulk copies, two ahead), Q tiles, K rows; V warps: V rows. Each
        // warp follows the mbarriers on its own, so a slow warp holds back no other.
        const bool is_k = warp < 4 + kTcKWarps;
        const int nthr = is_k ? kTcKWarps * 32 : kTcVWarps * 32;
        const int pt = tid - kTcSoftmaxThreads - (is_k ? 0 : kTcKWarps * 32);
        const bool leader = is_k && pt == 0;
        const int64_t last_tok = (int64_t)a.p0 + a.Nc - 1;
        const uint16_t *cache = is_k ? a.k_cache : a.v_cache;
        const uint32_t stage0 = sbase + (is_k ? kTcK : kTcV);
        uint64_t *full = is_k ? k_full : v_full;
        uint64_t *empty = is_k ? k_empty : v_empty;
        const int n_stages = is_k ? kTcKStages : kTcVStages;
        // the CTA's chunk stream: its tile list in order, chunk by chunk; tiles without chunks
        // (invalid lists) are skipped
        int ri = 0, c_in = 0, tile = tile_at(0), n_ch = size_at(tile);
        if (n_rounds > 0 && n_ch == 0) {
            c_in = -1;
            advance(ri, tile, c_in, n_ch);
        }
        int pf_ri = ri, pf_tile = tile, pf_c = c_in, pf_n = n_ch, pf_g = 0;
        auto prefetch = [&]() -> bool {         // leader: record of chunk pf_g into ring slot pf_g % ring
            if (pf_ri >= n_rounds) return true;
            const int rs = pf_g % kTcRing;
            if (pf_g >= kTcRing && !wait(&r_empty[rs], pf_g / kTcRing - 1)) return false;
            const ChunkRec *src = a.recs + (size_t)(pf_tile / a.Hkv) * kPlanCap + pf_c;
            mbar_arrive_expect_tx(smem_u32(&r_full[rs]), kRecCopyBytes);
            bulk_g2s(sbase + kTcRecs + rs * (uint32_t)sizeof(ChunkRec), src, kRecCopyBytes, smem_u32(&r_full[rs]));
            ++pf_g;
            advance(pf_ri, pf_tile, pf_c, pf_n);
            return true;
        };
        bool ok = true;
        if (leader) ok = prefetch() && prefetch();
        ok = __all_sync(0xffffffffu, ok);
        int g = 0, t_loc = -1, cur_tile = -1;
        while (ok && ri < n_rounds) {
            const int gkv = tile % a.Hkv;
            if (is_k && tile != cur_tile) {
                // ---- a new tile: its Q rows once the previous tile's QK MMAs are done
                cur_tile = tile;
                ++t_loc;
                if (t_loc > 0 && !wait_warp(&q_free, t_loc - 1)) {
                    ok = false;
                    break;
                }
                const int i0 = (tile / a.Hkv) * QT, nq = min(QT, a.Nc - i0);
                for (int gi = pt; gi < kTcRows * 32; gi += nthr) {
                    const int r = gi >> 5, gg = gi & 31;
                    const int qq = r / G, hh = r % G;
                    const uint32_t dst = sbase + kTcQ + (gg >> 3) * (kTcRows * 128) + swz(r, gg & 7);
                    if (qq < nq)
                        cp_async16(dst, a.q + ((int64_t)(i0 + qq) * a.Hq + gkv * G + hh) * kHeadDim + gg * 8);
                    else
                        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0) : "memory");
                }
                cp_async_arrive(smem_u32(&q_full));
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&q_full));
            }
            if (leader && !prefetch()) ok = false;
            const int s = g % n_stages, rs = g % kTcRing;
            if (!__all_sync(0xffffffffu, ok) || !wait_warp(&r_full[rs], g / kTcRing) ||
                (g >= n_stages && !wait_warp(&empty[s], g / n_stages - 1))) {
                ok = false;
                break;
            }
            const ChunkRec &r = ring[rs];
            for (int gi = pt; gi < kTcChunk * 32; gi += nthr) {
                const int j = gi >> 5, gg = gi & 31;
                const int b = r.blk[j >> 2];
                if (b < 0) continue;                   // padding column: not loaded (masked)
                // the newest block may extend past the last token; its tail is masked
                const int64_t tok = min((int64_t)b * kRatio + (j & 3), last_tok);
                cp_async16(stage0 + s * 32768 + (gg >> 3) * (kTcChunk * 128) + swz(j, gg & 7),
                           cache + (tok * a.Hkv + gkv) * kHeadDim + gg * 8);
            }
            cp_async_arrive(smem_u32(&full[s]));
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&r_empty[rs]));   // this warp is done with the record
            ++g;
            advance(ri, tile, c_in, n_ch);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        // no record copy may still be writing shared memory when the CTA exits (bounded waits)
        if (leader)
            for (int j = max(g, pf_g - 2); j < pf_g; ++j)
                mbar_wait_bounded(smem_u32(&r_full[j % kTcRing]), (uint32_t)(j / kTcRing) & 1u, kWaitLimitNs);
    } else if (warp == kTcMmaWarp) {
        // ================================================================ MMA issue
        if (lane == 0) {
            int g = 0, n_q = 0, n_tile = -1;
            // this CTA's chunk stream: (tile, chunk) in order, tiles without chunks skipped
            int it_r = 0, it_c = -1;
            int it_n = size_at(tile_at(0));
            auto next_chunk = [&](int &f, int &l) -> bool {
                ++it_c;
                while (it_r < n_rounds && it_c >= it_n) {  // each pass moves to the next tile
                    ++it_r;
                    it_c = 0;
                    it_n = size_at(tile_at(it_r));
                }
                if (it_r >= n_rounds) return false;
                f = it_c == 0;
                l = it_c == it_n - 1;
                return true;
            };
            uint64_t *last_bar = nullptr;        // the barrier of the last commit, and its phase
            uint32_t last_phase = 0;
            int first = 0, last = 0;
            bool ok = next_chunk(first, last);
            auto issue_qk = [&](int gq, int f, int l) -> bool {
                const int s = gq & 1, sk = gq % kTcKStages;   // S buffer, K stage
                if (!wait(&k_full[sk], gq / kTcKStages)) return false;
                if (f) {
                    if (!wait(&q_full, n_q)) return false;
                    ++n_q;
                }
                fence_proxy_async_smem();
                tc_fence_after();
                const uint32_t qa = sbase + kTcQ, kb = sbase + kTcK + sk * 32768;
#pragma unroll
                for (int ks = 0; ks < kHeadDim / 16; ++ks) {
                    const uint64_t ad = tc_desc(qa + (ks >> 2) * (kTcRows * 128) + (ks & 3) * 32, 16, 1024);
                    const uint64_t bd = tc_desc(kb + (ks >> 2) * (kTcChunk * 128) + (ks & 3) * 32, 16, 1024);
                    tc_mma(tmem + kTcTmemS + s * kTcChunk, ad, bd, tc_idesc(kTcRows, kTcChunk, 0), ks > 0);
                }
                tc_commit(smem_u32(&s_full[s]));
                tc_commit(smem_u32(&k_empty[sk]));
                last_bar = &k_empty[sk];
                last_phase = (uint32_t)(gq / kTcKStages);
                if (l) tc_commit(smem_u32(&q_free));
                return true;
            };
            if (ok) ok = issue_qk(0, first, last);
            while (ok) {
                int f1 = 0, l1 = 0;
                const bool more = next_chunk(f1, l1);
                if (more && !issue_qk(g + 1, f1, l1)) break;
                // ---- O (+)= P V for chunk g
                const int s = g & 1, sv = g % kTcVStages;     // P buffer, V stage
                if (!wait(&p_full[s], g >> 1) || !wait(&v_full[sv], g / kTcVStages)) break;
                if (first) {
                    ++n_tile;
                    if (n_tile > 0 && !wait(&o_free, n_tile - 1)) break;   // the previous tile's O was read
                }
                fence_proxy_async_smem();
                tc_fence_after();
                // P from tensor memory (its 16-token k-steps are 8 columns apart), V from shared memory
                const uint32_t pa = tmem + kTcTmemP + s * (kTcChunk / 2), vb = sbase + kTcV + sv * 32768;
#pragma unroll
                for (int ks = 0; ks < kTcChunk / 16; ++ks) {
                    const uint64_t bd = tc_desc(vb + ks * 2048, kTcChunk * 128, 1024);
                    tc_mma_ta(tmem + kTcTmemO, pa + ks * 8, bd, tc_idesc(kTcRows, kHeadDim, 1), !first || ks > 0);
                }
                tc_commit(smem_u32(&v_empty[sv]));
                tc_commit(smem_u32(&pv_done[s]));
                last_bar = &pv_done[s];
                last_phase = (uint32_t)(g >> 1);
                if (!more) break;
                ++g;
                first = f1;
                last = l1;
            }
            // the last commit covers every MMA issued: wait for it before TMEM is freed
            if (last_bar != nullptr) mbar_wait_bounded(smem_u32(last_bar), last_phase & 1u, kWaitLimitNs);
        }
    } else {
        // ================================================================ softmax
        const int row = tid;                     // MMA row = TMEM lane
        const int q_loc = row / G, h_loc = row % G;
        const uint32_t t_row = tmem + ((uint32_t)(32 * warp) << 16);
        const uint32_t t_o = t_row + kTcTmemO;
        int g = 0;
        bool ok = true;
        for (int r = 0; r < n_rounds && ok; ++r) {
            const int tile = tile_at(r);
            const int n_ch = size_at(tile);
            if (n_ch == 0) continue;                     // no tile, or invalid lists: nothing attended
            const int i0 = (tile / a.Hkv) * QT, nq = min(QT, a.Nc - i0), gkv = tile % a.Hkv;
            float m_ref = -INFINITY, l_sum = 0.f;
            bool o_init = false;
            for (int c = 0; c < n_ch; ++c) {
                const int s = g & 1, rs = g % kTcRing;
                if (!wait_warp(&r_full[rs], g / kTcRing) || !wait_warp(&s_full[s], g >> 1)) {
                    ok = false;
                    break;
                }
                const uint32_t vlo = ring[rs].vis[q_loc][0], vhi = ring[rs].vis[q_loc][1];
                mbar_arrive(smem_u32(&r_empty[rs]));
                tc_fence_after();
                // masked row max over the chunk (raw scores; the scale is positive), 8 partial maxima
                float mx[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mx[k] = -INFINITY;
                {
                    float s0[32], s1[32];
                    tmem_ld32_async(t_row + s * kTcChunk, s0);
                    tmem_ld32_async(t_row + s * kTcChunk + 32, s1);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        mx[j & 7] = fmaxf(mx[j & 7], (vlo >> j) & 1u ? s0[j] : -INFINITY);
                        mx[j & 7] = fmaxf(mx[j & 7], (vhi >> j) & 1u ? s1[j] : -INFINITY);
                    }
                }
                const float cmax =
                    fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
                    a.scale_log2;
                // lazy rescale: move the reference only when the row max grew by more than 2^8
                float f = 1.f;
                if (cmax > m_ref + 8.f) {
                    if (m_ref != -INFINITY) f = ex2_approx(m_ref - cmax);
                    m_ref = cmax;
                }
                l_sum *= f;
                // p = 2^(s * scale - m_ref) on visible columns (m_ref is finite whenever one is);
                // the scores are read from TMEM again, 32 columns at a time, to keep registers low
                float ps[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) ps[k] = 0.f;
                uint32_t pk[kTcChunk / 2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float sv[32];
                    tmem_ld32(t_row + s * kTcChunk + h * 32, sv);
                    const uint32_t vb = h ? vhi : vlo;
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float e0 = (vb >> j) & 1u ? ex2_approx(fmaf(sv[j], a.scale_log2, -m_ref)) : 0.f;
                        const float e1 = (vb >> (j + 1)) & 1u ? ex2_approx(fmaf(sv[j + 1], a.scale_log2, -m_ref)) : 0.f;
                        ps[(j >> 1) & 7] += e0 + e1;   // fp32 row sum: the LSE stays exact to fp32 rounding
                        pk[h * 16 + j / 2] = pack_bf16x2(e0, e1);
                    }
                }
                l_sum += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
                // P's buffer is free once the PV two chunks back is done; a rescale of O waits for
                // the previous PV (TMEM loads and stores are warp-collective: the warp rescales together)
                const bool rescale = o_init && __any_sync(0xffffffffu, f != 1.f);
                if ((g >= 2 && !wait_warp(&pv_done[s], (g >> 1) - 1)) ||
                    (rescale && !wait_warp(&pv_done[s ^ 1], (g - 1) >> 1))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (rescale) {
#pragma unroll 1
                    for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
                        float ov[32];
                        tmem_ld32(t_o + c0, ov);
#pragma unroll
                        for (int j = 0; j < 32; ++j) ov[j] *= f;
                        tmem_st32(t_o + c0, ov);
                    }
                }
                tmem_st32(t_row + kTcTmemP + s * (kTcChunk / 2), pk);
                tc_fence_before();
                mbar_arrive(smem_u32(&p_full[s]));
                o_init = true;
                ++g;
            }
            if (!ok) break;
            // ---- finish the tile: O / l -> bf16, lse; then O may be overwritten
            if (!wait_warp(&pv_done[(g - 1) & 1], (g - 1) >> 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const bool store = q_loc < nq && l_sum > 0.f;   // every valid row saw its own token
            const float inv = store ? 1.f / l_sum : 0.f;
            uint16_t *dst = a.out + ((int64_t)(i0 + q_loc) * a.Hq + gkv * G + h_loc) * kHeadDim;
#pragma unroll 1
            for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
                float ov[32];
                tmem_ld32(t_o + c0, ov);          // warp-collective: every lane loads
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const __nv_bfloat162 h2 = __floats2bfloat162_rn(ov[2 * j] * inv, ov[2 * j + 1] * inv);
                    w[j] = *reinterpret_cast<const uint32_t *>(&h2);
                }
                if (store) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<uint4 *>(dst + c0 + 8 * j) =
                            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                }
            }
            if (store && a.lse != nullptr)
                a.lse[(int64_t)(i0 + q_loc) * a.Hq + gkv * G + h_loc] = (m_ref + log2f(l_sum)) * kLn2;
            tc_fence_before();
            mbar_arrive(smem_u32(&o_free));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp) tmem_dealloc(tmem, 512);
}

bool prefill_tc_supported(int Hq, int Hkv) {
    const int G = Hkv > 0 ? Hq / Hkv : 0;
    return G == 8 || G == 16;
}

cudaError_t launch_prefill_tc(const AttnArgs &a, int interval_tokens, WsHeader *hdr, void *scratch,
                              size_t scratch_bytes, cudaStream_t st) {
    const int G = a.n_q_heads / a.n_kv_heads;
    const int QT = kTcRows / G;
    const int n_qt = (a.rows + QT - 1) / QT;
    if (scratch_bytes < prefill_tc_plan_bytes(a.rows, a.n_q_heads, a.n_kv_heads)) return cudaErrorInvalidValue;
    const int n_tiles = n_qt * a.n_kv_heads;
    char *sp = static_cast<char *>(scratch);
    int32_t *n_chunks = reinterpret_cast<int32_t *>(sp);
    int32_t *order = reinterpret_cast<int32_t *>(sp + round256((size_t)n_qt * 4));
    ChunkRec *recs = reinterpret_cast<ChunkRec *>(sp + round256((size_t)n_qt * 4) + round256((size_t)n_tiles * 2 * 4));
    if (((uintptr_t)recs & 255) != 0) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int grid = std::max(1, std::min(sms, n_tiles));
    const int n_rounds = (n_tiles + grid - 1) / grid;    // n_rounds * grid < 2 * n_tiles

    const int64_t n_blocks = ((int64_t)a.p0 + a.rows) / kRatio + 1;
    // the interval sets the evaluation order only; it is clamped to what the on-chip tables hold
    int64_t bpi = std::min<int64_t>(interval_tokens / kRatio, kTcMaxBpi);
    bpi = std::max<int64_t>(bpi, (n_blocks + kTcMaxIntervals - 1) / kTcMaxIntervals);
    if (bpi > kTcMaxBpi) return cudaErrorInvalidValue;

    PlanArgs pa{};
    pa.blocks = a.blocks;
    pa.count = a.count;
    pa.p0 = a.p0;
    pa.Nc = a.rows;
    pa.QT = QT;
    pa.bpi = (int)bpi;
    pa.n_iv = (int)((n_blocks + bpi - 1) / bpi);
    pa.n_chunks = n_chunks;
    pa.recs = recs;
    pa.hdr = hdr;
    e = cudaFuncSetAttribute(prefill_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPlSmem);
    if (e != cudaSuccess) return e;
    prefill_plan_kernel<<<n_qt, kPlanThreads, kPlSmem, st>>>(pa);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    prefill_order_kernel<<<1, kOrderThreads, 0, st>>>(n_chunks, n_qt, a.n_kv_heads, grid, n_rounds, order);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    TcArgs t{};
    t.q = a.q;
    t.k_cache = a.k_cache;
    t.v_cache = a.v_cache;
    t.out = a.out;
    t.lse = a.lse;
    t.n_chunks = n_chunks;
    t.recs = recs;
    t.order = order;
    t.p0 = a.p0;
    t.Nc = a.rows;
    t.Hq = a.n_q_heads;
    t.Hkv = a.n_kv_heads;
    t.scale_log2 = a.scale_log2;
    t.hdr = hdr;
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
