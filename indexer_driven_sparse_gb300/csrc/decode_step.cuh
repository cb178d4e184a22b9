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
// Each sequence (row) owns a contiguous group of c CTAs (sized by its context); CTA j owns
// the block range [nb*j/c, nb*(j+1)/c). The design keeps the number of dependent global
// round trips after the bandwidth-bound scan small:
//   1. The CTA owning block nb-1 re-pools it from the raw keys (exact fp64 mean).
//   2. Each CTA streams its pooled rows through a 4-stage shared-memory ring filled by bulk
//      async copies (TMA engine), keeping the 32-bit order-preserving score keys of its
//      range on chip and histogramming their top 12 bits.
//   3. Each CTA publishes its exact local top-K keys (64-bit: score key << 32 | ~block),
//      K = 2 x 512 / c rounded up to a power of two in [16, 512].
//   4. One row barrier. Every CTA then reads all published keys and computes the same
//      exact 512th key T and every CTA's output offset. If some CTA might hold more than K
//      selected blocks (its K-th key >= T), all CTAs take the exact fallback instead: a
//      global histogram, a threshold bin and the bin's members resolved at two barriers.
//   5. Each CTA writes its selected ids (ascending) and attends its own selected tokens
//      (plus the query's own block, in the row's last CTA), producing an (m, l, acc) partial.
//   6. Row barrier; the CTAs of the row merge all partials by LSE, each a slice of the
//      outputs, loading everything they need in one round trip.
// Dense rows (nb <= 512) select everything and skip 2-4. Every wait is bounded (250 ms on
// the GPU clock): a barrier or mbarrier that gives up records QSA_ERR_DEVICE_TIMEOUT and
// the CTA returns.
//
// Template parameters: G query heads per KV head; F8, FP8 indexer keys (128 E4M3 codes +
// an fp32 scale per block) instead of bf16; KV8, FP8 K/V rows (per token and KV head, 256
// E4M3 codes in a codes plane and one fp32 scale per 128 dims in a scales plane) instead
// of bf16 rows; RC, a VRAM row cache in front of bf16 K/V rows that live in host memory
// ("125B MoE を 3090 3 枚で運用する vLLM 最適化編", section 5): a direct-mapped cache of whole
// token rows (K and V of every KV head), each sequence owning an equal share of the slots.
// A selected token whose slot holds it is read from the cache (its slot is marked as hit in
// this step's epoch), any other from host memory; a missed token claims its slot with an
// atomic max of (epoch << 32 | token). After the row's second barrier, when no CTA of the row
// reads the cache any more, the claim's winner writes the row and the tag, unless the slot
// was hit in this step. Only tokens of complete blocks are cached (the query's own block may
// still be written by the caller). The kernel template lives in this header; decode_step.cu instantiates the
// bf16-K/V kernels and decode_step_kv8.cu the FP8-K/V ones, so the two compile in parallel.
#pragma once
#include "qsa_internal.cuh"
#include "qsa_ptx.cuh"

#include <float.h>

namespace qsa {
// Everything up to the FP8-K/V launch declarations at the end is local to each translation
// unit that includes this header.
namespace {

constexpr int kStepThreads = 512;
constexpr int kStepWarps = kStepThreads / 32;
constexpr int kHistBins = 4096;                       // top 12 bits of the score key
constexpr int kHistShift = 20;
constexpr int kRingStages = 4;
constexpr int kChunkRows = 128;                       // 128 pooled rows = 32 KiB per stage
constexpr int kChunkBytes = kChunkRows * kIdxDim * 2;
constexpr int kRingBytes = kRingStages * kChunkBytes;
constexpr int kMaxKeys = 12288;                       // score keys per CTA kept on chip
constexpr int kAttnTok = 32;                          // tokens per attention step
constexpr int kAttnWeightBlocks = 16384;              // attention cost of a row, in scanned blocks
constexpr int kMaxPub = 512;                          // published keys per CTA (+1 flag slot)

constexpr size_t kRingOff = 0;
constexpr size_t kKeysOff = kRingOff + (size_t)kRingBytes;
constexpr size_t kHistOff = kKeysOff + (size_t)kMaxKeys * 4;
constexpr size_t kQOff = kHistOff + (size_t)kHistBins * 4;          // query, bf16 [Hq][256]
constexpr size_t kNewRowOff = kQOff + (size_t)2 * kMaxGroup * kHeadDim * 2;
constexpr size_t kRawOff = kNewRowOff + 256;                          // 4 raw key rows, bf16
constexpr size_t kMbarOff = kRawOff + (size_t)kRatio * kIdxDim * 2;
constexpr size_t kStepSmem = kMbarOff + 16 * kRingStages;      // ring full / empty mbarriers
// FP8 keys (128 one-byte codes + an fp32 scale per block): a stage holds 256 code rows, and
// its scales arrive on the same mbarrier as the 16-byte-aligned run of whole 4-scale groups
// that covers them (at most 260 floats), in a ring of their own after the mbarriers.
constexpr int kChunkRows8 = kChunkBytes / kIdxDim;
constexpr int kScaleStageBytes = (kChunkRows8 + 8) * 4;
constexpr size_t kScaleOff = kStepSmem;
constexpr size_t kStepSmem8 = kScaleOff + (size_t)kRingStages * kScaleStageBytes;
static_assert(kScaleOff % 16 == 0, "bulk copies need 16-byte aligned destinations");

template <bool F8>
constexpr size_t step_smem() { return F8 ? kStepSmem8 : kStepSmem; }

// First scale and byte count of the aligned run of 4-scale groups covering rows
// [first, first + rows) (the scale array is padded to a multiple of 4 entries).
__device__ __forceinline__ void scale_run(int64_t first, int rows, int64_t *s0, uint32_t *bytes) {
    const int64_t a = first & ~(int64_t)3;
    const int64_t e = (first + rows + 3) & ~(int64_t)3;
    *s0 = a;
    *bytes = (uint32_t)((e - a) * 4);
}

// FP8: quantise the newest pooled block exactly as pool_keys_fp8_kernel does. Threads
// 0..127 hold one bf16 dim each in v (when `active`); every thread of the CTA calls this.
// Writes the codes and the scale to global memory, the codes to row8 (shared) and the scale
// to s_amax[4].
__device__ void quantize_newest(const StepArgs &a, int64_t dst, bool active, uint16_t v, uint8_t *row8,
                                float *s_amax) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool mine = active && tid < kIdxDim;
    const float x = mine ? bf16_bits_to_float(v) : 0.f;
    float m = fabsf(x);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0 && warp < kIdxDim / 32) s_amax[warp] = m;
    __syncthreads();
    const float amax = fmaxf(fmaxf(s_amax[0], s_amax[1]), fmaxf(s_amax[2], s_amax[3]));
    const float scale = __fdiv_rn(amax, kE4m3Max);
    if (mine) {
        const uint8_t code = scale > 0.f ? (uint8_t)(e4m3x2_of(__fdiv_rn(x, scale), 0.f) & 0xFFu) : (uint8_t)0;
        row8[tid] = code;
        a.codes[dst * kIdxDim + tid] = code;
        if (tid == 0) a.scales[dst] = scale;
    }
    __syncthreads();
    if (tid == 0) s_amax[4] = scale;
    __syncthreads();
}

struct StepRowState {
    uint32_t gen;               // barrier generation, advanced once per completed barrier
    uint32_t pad0;
    uint32_t counts[4];         // arrival counters, indexed by (generation - 1) & 3
    int32_t t1;                 // fallback: threshold bin (top 12 key bits)
    int32_t need;               // fallback: members of the threshold bin still to take
    unsigned long long t64;     // fallback: exact 64-bit threshold key
    uint32_t cand_count;
    int32_t pad1;
    int32_t definite[kMaxStepCtas];
    int32_t offset[kMaxStepCtas];
};

constexpr size_t kRowStateBytes = (sizeof(StepRowState) + 255) / 256 * 256;
__host__ __device__ constexpr size_t step_row_state_bytes() { return kRowStateBytes; }

StepLayout step_layout_of(int B, int64_t max_blocks, int Hq) {
    StepLayout L;
    L.rows = kWsHeaderBytes;
    L.hist = L.rows + (size_t)B * step_row_state_bytes();
    L.cands = L.hist + (size_t)B * kHistBins * 4;
    L.part = L.cands + ((size_t)B * (size_t)max_blocks * 8 + 255) / 256 * 256;
    L.pub = L.part + (size_t)kMaxStepCtas * Hq * (kHeadDim + 2) * 4;
    L.trace = L.pub + (size_t)kMaxStepCtas * (kMaxPub + 1) * 8;
    L.total = L.trace + (size_t)kMaxStepCtas * kTraceSlots * 8;
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

// Row barrier over `n` CTAs. Barrier number k of a launch completes generation g0 + k + 1
// (g0: the generation when the launch started). Arrival is one acq_rel atomic; the last
// CTA to arrive gets 1 back, may do exclusive work, and must call bar_release, which
// re-arms the next barrier's counter and publishes the generation with one release store.
// Others poll the generation (bounded). Returns 1 (last), 0 (released) or -1 (timeout).
__device__ int bar_arrive(StepRowState *rs, uint32_t g0, int k, int n, WsHeader *hdr, int row, int *s_flag) {
    // A GPU-scope fence orders only the calling thread's writes: every thread that wrote
    // data for other CTAs fences before the CTA barrier that precedes the arrival.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t g = g0 + (uint32_t)k + 1u;
        const uint32_t old = atom_add_acq_rel_u32(&rs->counts[(g - 1u) & 3u], 1u);
        int res = 1;
        if (old + 1u != (uint32_t)n) {
            res = 0;
            const uint64_t t0 = globaltimer_ns();
            while ((int32_t)(ld_acquire_u32(&rs->gen) - g) < 0) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    record_error(hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereStep, row);
                    res = -1;
                    break;
                }
                __nanosleep(32);
            }
        }
        *s_flag = res;
    }
    __syncthreads();
    return *s_flag;
}

// Plain row barrier (no exclusive work by the last CTA): every CTA polls the arrival
// counter itself, so no release hop follows the last arrival. Every barrier g leaves the
// counter of barrier g + 2 cleared: here the last CTA clears it (it was last used by
// barrier g - 2, which every CTA has passed; no CTA reaches g + 2 before this CTA arrives
// at g + 1); bar_release clears g + 1 and g + 2 before its release. With publish_gen the
// last CTA also sets the generation to g (the launch's last barrier; the next launch
// starts from it). Returns 0, or -1 on a timeout.
__device__ int bar_sync_fast(StepRowState *rs, uint32_t g0, int k, int n, bool publish_gen, WsHeader *hdr, int row,
                             int *s_flag) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t g = g0 + (uint32_t)k + 1u;
        uint32_t *cnt = &rs->counts[(g - 1u) & 3u];
        const uint32_t old = atom_add_acq_rel_u32(cnt, 1u);
        int res = 0;
        if (old + 1u == (uint32_t)n) {
            rs->counts[(g + 1u) & 3u] = 0u;
            if (publish_gen) st_release_u32(&rs->gen, g);
        } else {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_u32(cnt) < (uint32_t)n) {
                if (globaltimer_ns() - t0 > kWaitLimitNs) {
                    record_error(hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereStep, row);
                    res = -1;
                    break;
                }
            }
        }
        *s_flag = res;
    }
    __syncthreads();
    return *s_flag;
}

__device__ void bar_release(StepRowState *rs, uint32_t g0, int k) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        // the counters of barriers g + 1 and g + 2: no CTA passes g before this release
        const uint32_t g = g0 + (uint32_t)k + 1u;
        rs->counts[g & 3u] = 0u;
        rs->counts[(g + 1u) & 3u] = 0u;
        st_release_u32(&rs->gen, g);
    }
}

// CTA-wide: in hist[0..nbins) (bins high = better, nbins a power of two >= 256), find the
// bin where the count from the top first reaches `need` (1 <= need <= total). Writes the
// bin to *s_d and the count strictly above it to *s_above; all threads return after a sync.
__device__ void block_find_bin(const uint32_t *hist, int nbins, uint32_t need, int *s_d, uint32_t *s_above,
                               uint32_t *s_wtot) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = nbins >= kStepThreads ? nbins / kStepThreads : 1;
    const int nact = nbins / per;
    uint32_t x = 0;
    if (tid < nact)
        for (int i = 0; i < per; ++i) x += hist[tid * per + i];
    uint32_t s = x;                               // suffix sum within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, s, o);
        if (lane + o < 32) s += v;
    }
    if (lane == 0) s_wtot[warp] = s;
    __syncthreads();
    // counts of the warps above this one: a suffix scan of the 16 warp totals in registers
    uint32_t t = lane < kStepWarps ? s_wtot[lane] : 0u;
#pragma unroll
    for (int o = 1; o < kStepWarps; o <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, t, o);
        if (lane + o < kStepWarps) t += v;
    }
    const uint32_t higher = __shfl_sync(0xffffffffu, t, (warp + 1) & 31) * (warp + 1 < kStepWarps ? 1u : 0u);
    const uint32_t S = s + higher;                // count in this thread's bins and above
    if (tid < nact && S >= need && S - x < need) {
        uint32_t run = S - x;
        int d = tid * per + per - 1;
        for (; d > tid * per; --d) {
            if (run + hist[d] >= need) break;
            run += hist[d];
        }
        *s_d = d;
        *s_above = run;
    }
    __syncthreads();
}

// CTA-wide: a threshold T such that exactly `need` of the nonzero 64-bit keys among
// keys[0..n) (shared or global memory; zero marks an empty slot) are >= T. T is the
// need-th largest key, or a value just above the next key down. The radix digits start
// below the prefix that every nonzero key shares (found from their min and max), so the
// histogram spreads instead of piling into a few hot bins; 11-bit passes stop as soon as
// the chosen bin holds exactly the keys still needed. With `scratch` (capacity `cap`), the
// first pass's chosen bin is compacted so later passes touch only its members.
// Requires need <= number of nonzero keys; returns ~0 when there is none.
__device__ unsigned long long select_kth_key64(const unsigned long long *keys, uint32_t n, uint32_t need,
                                               uint32_t *hist, int *s_d, uint32_t *s_above, uint32_t *s_wtot,
                                               unsigned long long *s_red, unsigned long long *scratch = nullptr,
                                               uint32_t cap = 0, uint32_t *s_cn = nullptr) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned long long mn = ~0ull, mx = 0ull;
    for (uint32_t i = tid; i < n; i += kStepThreads) {
        const unsigned long long k = keys[i];
        if (k != 0ull) {
            mn = k < mn ? k : mn;
            mx = k > mx ? k : mx;
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const unsigned long long a = __shfl_xor_sync(0xffffffffu, mn, o);
        const unsigned long long b = __shfl_xor_sync(0xffffffffu, mx, o);
        mn = a < mn ? a : mn;
        mx = b > mx ? b : mx;
    }
    if (lane == 0) {
        s_red[warp] = mn;
        s_red[kStepWarps + warp] = mx;
    }
    __syncthreads();
    mn = ~0ull;
    mx = 0ull;
    for (int w = 0; w < kStepWarps; ++w) {
        mn = s_red[w] < mn ? s_red[w] : mn;
        mx = s_red[kStepWarps + w] > mx ? s_red[kStepWarps + w] : mx;
    }
    if (mx == 0ull) return ~0ull;
    const unsigned long long diff = mn ^ mx;
    if (diff == 0ull) return mx;                      // a single distinct key
    int hi = 64 - __clzll((long long)diff);           // bits >= hi are shared by every nonzero key
    unsigned long long prefix = hi >= 64 ? 0ull : (mx >> hi) << hi;
    bool compacted = false;
    while (hi > 0) {
        const int width = hi >= 11 ? 11 : hi;
        const int shift = hi - width;
        const int nbins = 1 << width;
        for (int i = tid; i < 2048; i += kStepThreads) hist[i] = 0;
        __syncthreads();
        for (uint32_t i = tid; i < n; i += kStepThreads) {
            const unsigned long long k = keys[i];
            if (k != 0ull && (hi >= 64 || (k >> hi) == (prefix >> hi)))
                atomicAdd(&hist[(uint32_t)(k >> shift) & (nbins - 1)], 1u);
        }
        __syncthreads();
        block_find_bin(hist, nbins < 256 ? 256 : nbins, need, s_d, s_above, s_wtot);
        const int d = *s_d;
        const uint32_t in_bin = hist[d];
        prefix |= (unsigned long long)d << shift;
        need -= *s_above;
        __syncthreads();
        if (in_bin == need) return prefix;           // the whole bin is kept
        if (!compacted && scratch != nullptr && in_bin <= cap) {
            // later passes see only the members of the chosen bin
            if (tid == 0) *s_cn = 0;
            __syncthreads();
            for (uint32_t i = tid; i < n; i += kStepThreads) {
                const unsigned long long k = keys[i];
                if (k != 0ull && (k >> shift) == (prefix >> shift)) scratch[atomicAdd(s_cn, 1u)] = k;
            }
            __syncthreads();
            keys = scratch;
            n = *s_cn;
            compacted = true;
        }
        hi = shift;
    }
    return prefix;
}

// Register-resident variant of select_kth_key64 for n <= 8 x 512 keys: each thread keeps
// its (at most 8) keys in registers, so no pass reloads them and every loop unrolls.
__device__ unsigned long long select_kth_key64_reg(const unsigned long long *keys, uint32_t n, uint32_t need,
                                                   uint32_t *hist, int *s_d, uint32_t *s_above, uint32_t *s_wtot,
                                                   unsigned long long *s_red) {
    constexpr int R = 8;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned long long kr[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint32_t i = tid + r * kStepThreads;
        kr[r] = i < n ? keys[i] : 0ull;
    }
    unsigned long long mn = ~0ull, mx = 0ull;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (kr[r] != 0ull) mn = kr[r] < mn ? kr[r] : mn;
        mx = kr[r] > mx ? kr[r] : mx;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const unsigned long long a = __shfl_xor_sync(0xffffffffu, mn, o);
        const unsigned long long b = __shfl_xor_sync(0xffffffffu, mx, o);
        mn = a < mn ? a : mn;
        mx = b > mx ? b : mx;
    }
    if (lane == 0) {
        s_red[warp] = mn;
        s_red[kStepWarps + warp] = mx;
    }
    __syncthreads();
    {
        const unsigned long long a = lane < kStepWarps ? s_red[lane] : ~0ull;
        const unsigned long long b = lane < kStepWarps ? s_red[kStepWarps + lane] : 0ull;
        mn = a;
        mx = b;
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) {
            const unsigned long long c = __shfl_xor_sync(0xffffffffu, mn, o);
            const unsigned long long d = __shfl_xor_sync(0xffffffffu, mx, o);
            mn = c < mn ? c : mn;
            mx = d > mx ? d : mx;
        }
        mn = __shfl_sync(0xffffffffu, mn, 0);
        mx = __shfl_sync(0xffffffffu, mx, 0);
    }
    if (mx == 0ull) return ~0ull;
    const unsigned long long diff = mn ^ mx;
    if (diff == 0ull) return mx;
    int hi = 64 - __clzll((long long)diff);
    unsigned long long prefix = hi >= 64 ? 0ull : (mx >> hi) << hi;
    bool first = true;
    while (hi > 0) {
        // a 12-bit first digit (then 11-bit ones) below the prefix every candidate shares
        const int width = hi >= (first ? 12 : 11) ? (first ? 12 : 11) : hi;
        const int shift = hi - width;
        const int nbins = 1 << width;
        for (int i = tid; i < 4096; i += kStepThreads) hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const unsigned long long k = kr[r];
            if (k != 0ull && (hi >= 64 || (k >> hi) == (prefix >> hi)))
                atomicAdd(&hist[(uint32_t)(k >> shift) & (nbins - 1)], 1u);
        }
        __syncthreads();
        block_find_bin(hist, nbins < 256 ? 256 : nbins, need, s_d, s_above, s_wtot);
        const int d = *s_d;
        const uint32_t in_bin = hist[d];
        prefix |= (unsigned long long)d << shift;
        need -= *s_above;
        __syncthreads();
        if (in_bin == need) return prefix;
        if (in_bin <= (uint32_t)kStepThreads) {
            // the bin's members (distinct keys) -> the need-th largest by counting ranks;
            // warp-aggregated compaction into the histogram's space
            unsigned long long *cand = reinterpret_cast<unsigned long long *>(hist);
            if (tid == 0) *s_above = 0u;
            __syncthreads();
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const unsigned long long k = kr[r];
                const bool m = k != 0ull && (k >> shift) == (prefix >> shift);
                const unsigned bal = __ballot_sync(0xffffffffu, m);
                if (bal) {
                    uint32_t base = 0;
                    if (lane == 0) base = atomicAdd(s_above, (uint32_t)__popc(bal));
                    base = __shfl_sync(0xffffffffu, base, 0);
                    if (m) cand[base + __popc(bal & ((1u << lane) - 1u))] = k;
                }
            }
            __syncthreads();
            if (tid < (int)in_bin) {
                const unsigned long long mine = cand[tid];
                uint32_t rank = 0;
                for (uint32_t j = 0; j < in_bin; ++j) rank += cand[j] > mine ? 1u : 0u;
                if (rank == need - 1u) s_red[0] = mine;
            }
            __syncthreads();
            const unsigned long long t = s_red[0];
            __syncthreads();
            return t;
        }
        first = false;
        hi = shift;
    }
    return prefix;
}

// The score of a 32-bit order-preserving score key (NaN for the NaN key 0).
__device__ __forceinline__ float score_of_key(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// CTA-wide: the need-th largest of the nonzero 64-bit keys in keys[0..n), n <= 8 x 512.
// The keys' scores (upper halves) fall into 4096 bins linear in the score value, which
// spreads them where bins on the key's top bits would crowd a few exponents; the threshold
// bin then holds a few keys, ranked exactly. When the bins cannot split the keys (equal
// scores, no finite range, more than one CTA's threads of keys in the threshold bin) the
// radix select takes over.
__device__ unsigned long long select_kth_key64_lin(const unsigned long long *keys, uint32_t n, uint32_t need,
                                                   uint32_t *hist, int *s_d, uint32_t *s_above, uint32_t *s_wtot,
                                                   unsigned long long *s_red, float *s_fred,
                                                   unsigned long long *cand, uint32_t *s_ncand) {
    constexpr int R = 8;
    constexpr int kBins = 4096;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t need0 = need;
    if (tid == 0) *s_ncand = 0u;                  // the bin's candidates, counted below
    unsigned long long kr[R];
    float vr[R];
    float vmin = FLT_MAX, vmax = -FLT_MAX;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const uint32_t i = tid + r * kStepThreads;
        kr[r] = i < n ? keys[i] : 0ull;
        vr[r] = score_of_key((uint32_t)(kr[r] >> 32));
        if (kr[r] != 0ull && fabsf(vr[r]) <= FLT_MAX) {
            vmin = fminf(vmin, vr[r]);
            vmax = fmaxf(vmax, vr[r]);
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        vmin = fminf(vmin, __shfl_xor_sync(0xffffffffu, vmin, o));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    }
    if (lane == 0) {
        s_fred[warp] = vmin;
        s_fred[kStepWarps + warp] = vmax;
    }
    for (int i = tid; i < kBins; i += kStepThreads) hist[i] = 0;
    __syncthreads();
    vmin = lane < kStepWarps ? s_fred[lane] : FLT_MAX;
    vmax = lane < kStepWarps ? s_fred[kStepWarps + lane] : -FLT_MAX;
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {
        vmin = fminf(vmin, __shfl_xor_sync(0xffffffffu, vmin, o));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    }
    vmin = __shfl_sync(0xffffffffu, vmin, 0);
    vmax = __shfl_sync(0xffffffffu, vmax, 0);
    const float scale = (float)(kBins - 2) / (vmax - vmin);
    if (!(vmax > vmin && scale > 0.f && scale <= FLT_MAX))
        return select_kth_key64_reg(keys, n, need, hist, s_d, s_above, s_wtot, s_red);
    // bins non-decreasing in the key: NaN / -inf lowest, +inf highest
    auto bin_of = [&](float v) -> int {
        if (v != v || v == -INFINITY) return 0;
        if (v == INFINITY) return kBins - 1;
        return min((int)((v - vmin) * scale), kBins - 2);
    };
#pragma unroll
    for (int r = 0; r < R; ++r)
        if (kr[r] != 0ull) atomicAdd(&hist[bin_of(vr[r])], 1u);
    __syncthreads();
    block_find_bin(hist, kBins, need, s_d, s_above, s_wtot);
    // hist, s_d and s_above are not written again on this path, so they are read without a
    // further barrier; every thread reads the same values and takes the same branch
    const int d = *s_d;
    const uint32_t in_bin = hist[d];
    need -= *s_above;
    if (in_bin > (uint32_t)kStepThreads) {
        __syncthreads();                            // every thread has read them: the fallback rewrites them
        return select_kth_key64_reg(keys, n, need0, hist, s_d, s_above, s_wtot, s_red);
    }
    // the bin's members (into `cand`, beside the keys) -> the need-th largest of them by
    // counting ranks (distinct keys)
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const bool m = kr[r] != 0ull && bin_of(vr[r]) == d;
        const unsigned bal = __ballot_sync(0xffffffffu, m);
        if (bal) {
            uint32_t base = 0;
            if (lane == 0) base = atomicAdd(s_ncand, (uint32_t)__popc(bal));
            base = __shfl_sync(0xffffffffu, base, 0);
            if (m) cand[base + __popc(bal & ((1u << lane) - 1u))] = kr[r];
        }
    }
    __syncthreads();
    if (tid < (int)in_bin) {
        const unsigned long long mine = cand[tid];
        uint32_t rank = 0;
        for (uint32_t j = 0; j < in_bin; ++j) rank += cand[j] > mine ? 1u : 0u;
        if (rank == need - 1u) s_red[0] = mine;
    }
    __syncthreads();
    // s_red[0] holds the result until the caller's next barrier (the caller writes it no earlier)
    return s_red[0];
}

// Warp 0: sum of vals[0..count) (shared memory) -> *out. Other warps skip.
__device__ __forceinline__ void warp_sum_prefix(const uint32_t *vals, int count, int *out) {
    if (threadIdx.x < 32) {
        uint32_t sum = 0;
        for (int j = threadIdx.x; j < count; j += 32) sum += vals[j];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (threadIdx.x == 0) *out = (int)sum;
    }
}

// Sum each of NV values over the warp's 32 lanes; afterwards the lane holds the total of
// value index `idx` (returned). Reduce-scatter: each level halves the values a lane keeps,
// so the whole reduction takes NV - 1 + log2(32/NV) shuffles instead of 5 NV.
template <int NV>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[NV], int lane, int *idx) {
    int base = 0;
#pragma unroll
    for (int level = 0; (NV >> level) > 1; ++level) {
        const int n = NV >> level;          // values still held
        const int o = 16 >> level;          // exchange distance
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
        if (up) base += n / 2;
    }
    float r = v[0];
#pragma unroll
    for (int o = 16 / NV; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    *idx = base;
    return r;
}

__device__ __forceinline__ unsigned long long key64_of(uint32_t key, int64_t blk) {
    return ((unsigned long long)key << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)blk);
}

// Published keys per CTA for a row split over c CTAs: 2 x 512 / c, a power of two in [16, 512]
// (a CTA holds 512 / c selected blocks on average; 16 leaves a wide margin at c = 152).
__device__ __forceinline__ int pub_count(int c) {
    int k = 16;
    while (k < kMaxPub && k * c < 2 * kBlockTopK) k <<= 1;
    return k;
}

// 8-byte asynchronous global -> shared copy (through L1), completed with the 16-byte ones.
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}

// Eight E4M3 codes (byte k = dim k) -> fp32, exactly (E4M3 -> f16 -> f32 are both exact).
__device__ __forceinline__ void e4m3x8_to_f32(const uint2 &v, float (&f)[8]) {
    const uint32_t w[2] = {v.x, v.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint32_t h0, h1;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h0) : "h"((uint16_t)(w[i] & 0xFFFFu)));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h1) : "h"((uint16_t)(w[i] >> 16)));
        f[4 * i + 0] = __half2float(__ushort_as_half((unsigned short)(h0 & 0xFFFFu)));
        f[4 * i + 1] = __half2float(__ushort_as_half((unsigned short)(h0 >> 16)));
        f[4 * i + 2] = __half2float(__ushort_as_half((unsigned short)(h1 & 0xFFFFu)));
        f[4 * i + 3] = __half2float(__ushort_as_half((unsigned short)(h1 >> 16)));
    }
}

// One E4M3 code -> fp32, exactly.
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)c));
    return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// Bytes one token of an attention chunk occupies in shared memory: its K row and V row of
// every KV head, bf16; or, with FP8 K/V, the K codes and V codes of every KV head followed by
// their scales (two fp32 per KV head each). Both are multiples of 16 bytes.
template <bool KV8>
__device__ __forceinline__ int chunk_tok_bytes(int Hkv) {
    return KV8 ? Hkv * (2 * kHeadDim + 16) : Hkv * 4 * kHeadDim;
}

// Gather one attention chunk: the K and V rows (all KV heads) of up to kAttnTok tokens of
// the row's token sequence (list blocks, then the query's own block) into shared memory,
// bf16 rows, as 16-byte async copies.
__device__ void gather_chunk_bf16(const StepArgs &a, uint16_t *dst, int j_base, int n, int n_list, bool dense,
                                  const int32_t *sel, int64_t nb, int64_t base, int p, int row, int row_elems) {
    const int tok_elems = 2 * row_elems;
    const int gran_per_tok = tok_elems * 2 / 16;                       // 16-byte granules per token
    for (int gidx = threadIdx.x; gidx < n * gran_per_tok; gidx += kStepThreads) {
        const int i = gidx / gran_per_tok;
        const int rem = gidx - i * gran_per_tok;
        const int is_v = rem >= gran_per_tok / 2;
        const int gpos = rem - is_v * (gran_per_tok / 2);
        const int j = j_base + i;
        int64_t tk;
        if (j < kRatio * n_list) {
            const int64_t blk = dense ? (j >> 2) : sel[j >> 2];
            if (blk < 0 || blk >= nb) {               // never expected: flag it, read a safe row
                record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereStep, row);
                tk = p;
            } else {
                tk = kRatio * blk + (j & 3);
            }
        } else {
            tk = kRatio * nb + (j - kRatio * n_list);
        }
        const uint16_t *src = (is_v ? a.v_cache : a.k_cache) + (base + tk) * row_elems + gpos * 8;
        cp_async16(smem_u32(dst + (size_t)i * tok_elems + is_v * row_elems + gpos * 8), src);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// The same chunk with FP8 K/V: per token, the K codes and V codes of every KV head, then their
// scale pairs, as 16-byte (codes) and 8-byte (scale pairs) async copies.
__device__ void gather_chunk_fp8kv(const StepArgs &a, unsigned char *dst, int j_base, int n, int n_list, bool dense,
                                   const int32_t *sel, int64_t nb, int64_t base, int p, int row) {
    const int Hkv = a.n_kv_heads;
    const int tok_bytes = chunk_tok_bytes<true>(Hkv);
    const int row_bytes = Hkv * kHeadDim;                              // one token's K (or V) codes
    const int n_gran = row_bytes / 8;                                  // 16-byte pieces of K and V
    const int units = n_gran + 2 * Hkv;                                // + 8-byte scale pairs
    for (int gidx = threadIdx.x; gidx < n * units; gidx += kStepThreads) {
        const int i = gidx / units;
        const int rem = gidx - i * units;
        const int j = j_base + i;
        int64_t tk;
        if (j < kRatio * n_list) {
            const int64_t blk = dense ? (j >> 2) : sel[j >> 2];
            if (blk < 0 || blk >= nb) {               // never expected: flag it, read a safe row
                record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereStep, row);
                tk = p;
            } else {
                tk = kRatio * blk + (j & 3);
            }
        } else {
            tk = kRatio * nb + (j - kRatio * n_list);
        }
        unsigned char *tdst = dst + (size_t)i * tok_bytes;
        if (rem < n_gran) {
            const int is_v = rem >= n_gran / 2;
            const int gpos = rem - is_v * (n_gran / 2);
            cp_async16(smem_u32(tdst + is_v * row_bytes + gpos * 16),
                       (is_v ? a.v_codes : a.k_codes) + (base + tk) * row_bytes + gpos * 16);
        } else {
            const int su = rem - n_gran;                                   // 0 .. 2 Hkv - 1
            const int is_v = su >= Hkv;
            const int h = su - is_v * Hkv;
            cp_async8(smem_u32(tdst + 2 * row_bytes + (is_v * Hkv + h) * 8),
                      (is_v ? a.v_scales : a.k_scales) + ((base + tk) * Hkv + h) * 2);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Per-token bookkeeping of the row cache for the two chunks in flight, in the score-key area
// (dead during attention): source rows, and the slot and claim of a token that may fill.
struct RcChunk {
    const uint16_t *k_src[kAttnTok], *v_src[kAttnTok];
    int64_t slot[kAttnTok];                  // -1: nothing to fill
    unsigned long long claim[kAttnTok];
    int64_t flat[kAttnTok];
};

// The bf16 chunk with the row cache: one thread per token decides hit or miss (marking the
// slot, or claiming it), then the granules are copied from the cache or from host memory.
__device__ void gather_chunk_rc(const StepArgs &a, uint16_t *dst, RcChunk *rc, int j_base, int n, int n_list,
                                bool dense, const int32_t *sel, int64_t nb, int64_t base, int p, int row,
                                int row_elems, int64_t slot_lo, int64_t slot_n) {
    const int tok_elems = 2 * row_elems;
    const int gran_per_tok = tok_elems * 2 / 16;
    for (int i = threadIdx.x; i < n; i += kStepThreads) {
        const int j = j_base + i;
        int64_t tk;
        bool cacheable = false;
        if (j < kRatio * n_list) {
            const int64_t blk = dense ? (j >> 2) : sel[j >> 2];
            if (blk < 0 || blk >= nb) {
                record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereStep, row);
                tk = p;
            } else {
                tk = kRatio * blk + (j & 3);
                cacheable = true;
            }
        } else {
            tk = kRatio * nb + (j - kRatio * n_list);
        }
        const int64_t flat = base + tk;
        const uint16_t *k_src = a.k_cache + flat * row_elems, *v_src = a.v_cache + flat * row_elems;
        int64_t fill = -1;
        unsigned long long claim = 0ull;
        if (cacheable) {
            const int64_t slot = slot_lo + tk % slot_n;
            if (__ldcg(a.rc_tag + slot) == flat) {            // hit: read the cached row
                a.rc_hit[slot] = a.rc_epoch;
                k_src = a.rc_rows + slot * tok_elems;
                v_src = k_src + row_elems;
            } else {                                          // miss: claim the slot
                claim = ((unsigned long long)a.rc_epoch << 32) | (uint32_t)flat;
                atomicMax(a.rc_claim + slot, claim);
                fill = slot;
            }
        }
        rc->k_src[i] = k_src;
        rc->v_src[i] = v_src;
        rc->slot[i] = fill;
        rc->claim[i] = claim;
        rc->flat[i] = flat;
    }
    __syncthreads();
    for (int gidx = threadIdx.x; gidx < n * gran_per_tok; gidx += kStepThreads) {
        const int i = gidx / gran_per_tok;
        const int rem = gidx - i * gran_per_tok;
        const int is_v = rem >= gran_per_tok / 2;
        const int gpos = rem - is_v * (gran_per_tok / 2);
        cp_async16(smem_u32(dst + (size_t)i * tok_elems + is_v * row_elems + gpos * 8),
                   (is_v ? rc->v_src[i] : rc->k_src[i]) + gpos * 8);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// After the row's last cache read: the claims this CTA won (and whose slot no token hit in this
// step) write a chunk's rows, still in shared memory, and their tags.
__device__ void fill_rc(const StepArgs &a, const uint16_t *rows, const RcChunk *rc, int n, int row_elems,
                        int *s_ok) {
    const int tok_elems = 2 * row_elems;
    const int gran_per_tok = tok_elems * 2 / 16;
    for (int i = threadIdx.x; i < n; i += kStepThreads) {
        const int64_t slot = rc->slot[i];
        s_ok[i] = slot >= 0 && __ldcg(a.rc_claim + slot) == rc->claim[i] && __ldcg(a.rc_hit + slot) != a.rc_epoch;
    }
    __syncthreads();
    for (int gidx = threadIdx.x; gidx < n * gran_per_tok; gidx += kStepThreads) {
        const int i = gidx / gran_per_tok;
        if (!s_ok[i]) continue;
        const int rem = gidx - i * gran_per_tok;
        *reinterpret_cast<uint4 *>(a.rc_rows + rc->slot[i] * tok_elems + rem * 8) =
            *reinterpret_cast<const uint4 *>(rows + (size_t)i * tok_elems + rem * 8);
    }
    for (int i = threadIdx.x; i < n; i += kStepThreads)
        if (s_ok[i]) a.rc_tag[rc->slot[i]] = rc->flat[i];
}

// One chunk of either format into ring half `half` (64 KiB).
template <bool KV8>
__device__ __forceinline__ void gather_chunk(const StepArgs &a, unsigned char *ring, int j_base, int n, int n_list,
                                             bool dense, const int32_t *sel, int64_t nb, int64_t base, int p,
                                             int row) {
    if constexpr (KV8)
        gather_chunk_fp8kv(a, ring, j_base, n, n_list, dense, sel, nb, base, p, row);
    else
        gather_chunk_bf16(a, reinterpret_cast<uint16_t *>(ring), j_base, n, n_list, dense, sel, nb, base, p, row,
                          a.n_kv_heads * kHeadDim);
}

// This CTA's share of the caller's next read (its grid slice, in 16-byte units), issued as
// L2 prefetch hints of up to 64 KiB by a few threads. Called once, when the CTA's own
// pooled-key stream is done, so the prefetch uses HBM time the exchanges below leave idle.
__device__ __forceinline__ void prefetch_next_read(const StepArgs &a) {
    if (a.next_read == nullptr || a.next_read_bytes < 16) return;
    const int64_t units = a.next_read_bytes >> 4;
    const int64_t u0 = units * blockIdx.x / gridDim.x, u1 = units * (blockIdx.x + 1) / gridDim.x;
    constexpr int64_t kPiece = 4096;                       // 64 KiB
    for (int64_t u = u0 + (int64_t)threadIdx.x * kPiece; u < u1; u += (int64_t)kStepThreads * kPiece)
        bulk_prefetch_l2(a.next_read + u * 16, (uint32_t)(min(kPiece, u1 - u) * 16));
}

template <int G, bool F8, bool KV8, bool RC = false>
__global__ void __launch_bounds__(kStepThreads, 1) decode_step_kernel(StepArgs a) {
    constexpr int kRows = F8 ? kChunkRows8 : kChunkRows;      // key rows per ring stage
    constexpr int kRowBytes = F8 ? kIdxDim : kIdxDim * 2;
    extern __shared__ __align__(128) unsigned char smem[];
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem + kKeysOff);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem + kHistOff);
    uint16_t *q_b = reinterpret_cast<uint16_t *>(smem + kQOff);
    uint16_t *newrow = reinterpret_cast<uint16_t *>(smem + kNewRowOff);
    uint8_t *newrow8 = reinterpret_cast<uint8_t *>(smem + kNewRowOff);
    const uint32_t scale0 = smem_u32(smem + kScaleOff);                 // FP8 only
    uint16_t *rawrows = reinterpret_cast<uint16_t *>(smem + kRawOff);
    unsigned long long *ring64 = reinterpret_cast<unsigned long long *>(smem + kRingOff);
    const uint32_t mbar0 = smem_u32(smem + kMbarOff);
    const uint32_t ring0 = smem_u32(smem + kRingOff);

    __shared__ RowPart s_part;
    __shared__ int s_flag, s_d, s_overflow;
    __shared__ uint32_t s_above, s_n;
    __shared__ unsigned long long s_kmin;
    __shared__ unsigned long long s_kth[kMaxStepCtas];
    __shared__ unsigned long long s_red[2 * kStepWarps];
    __shared__ int32_t s_sel[kBlockTopK];
    __shared__ uint32_t s_cnt[kMaxStepCtas];
    __shared__ uint32_t s_wsum[kStepWarps];
    __shared__ float s_m[2 * kMaxGroup], s_l[2 * kMaxGroup], s_alpha[2 * kMaxGroup];
    __shared__ int32_t s_ctx[kMaxStepRows], s_tok_off[kMaxStepRows + 1], s_blk_off[kMaxStepRows + 1];
    __shared__ int32_t s_debug;
    __shared__ unsigned long long s_pubk[32];
    __shared__ float s_fred[2 * kStepWarps];
    __shared__ float s_amax[5];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hq = a.n_q_heads, Hkv = a.n_kv_heads;
    // launched as a programmatic dependent of the previous step: its CTAs may be resident
    // before that step has finished; nothing in global memory is touched before it has
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- metadata in one round trip (partition in warp 0, offsets in warps 1-2)
    if (warp == 0) {
        partition_rows(a.ctx_len, a.B, &s_part);
        if (lane < a.B) s_ctx[lane] = a.ctx_len[lane];
        if (lane + 32 < a.B) s_ctx[lane + 32] = a.ctx_len[lane + 32];
    } else if (warp == 1) {
        for (int i = lane; i <= a.B; i += 32) s_tok_off[i] = a.tok_off[i];
    } else if (warp == 2) {
        for (int i = lane; i <= a.B; i += 32) s_blk_off[i] = a.blk_off[i];
    } else if (warp == 3 && lane == 0) {
        for (int s = 0; s < kRingStages; ++s) {
            mbar_init(mbar0 + 8 * s, 1);                              // full: the stage's bytes
            mbar_init(mbar0 + 8 * (kRingStages + s), kStepWarps);     // empty: every warp read it
        }
        fence_mbar_init();
    } else if (warp == 4 && lane == 0) {
        s_debug = __ldcg(&a.hdr->debug);
    }
    __syncthreads();
    const bool tracing = s_debug == kDebugTrace;
    unsigned long long *trace = a.trace + (size_t)blockIdx.x * kTraceSlots;
#define STEP_TRACE(i) \
    if (tracing && tid == 0) trace[i] = globaltimer_ns()
    STEP_TRACE(0);
    const int row = s_part.row, jj = s_part.jj, cr = s_part.cr, first = s_part.first;

    // ---- row geometry (identical in every CTA of the row)
    const int p = s_ctx[row];
    const int64_t base = s_tok_off[row], end = s_tok_off[row + 1];
    const int64_t boff = s_blk_off[row];
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
    const int n_tma = owner_new ? n_mine - 1 : n_mine;        // block nb-1 is scored from the re-pooled row
    const int n_chunks = dense ? 0 : (n_tma + kRows - 1) / kRows;
    const unsigned char *gsrc = F8 ? a.codes + (boff + lo) * kIdxDim
                                   : reinterpret_cast<const unsigned char *>(a.pooled + (boff + lo) * kIdxDim);
    // stage c of the ring: its key rows (and, FP8, their scales) on full mbarrier c
    auto issue_stage = [&](int c, int stage) {
        const int rows = min(kRows, n_tma - c * kRows);
        const uint32_t bytes = (uint32_t)rows * kRowBytes;
        int64_t s0 = 0;
        uint32_t sbytes = 0;
        if (F8) scale_run(boff + lo + (int64_t)c * kRows, rows, &s0, &sbytes);
        mbar_arrive_expect_tx(mbar0 + 8 * stage, bytes + sbytes);
        bulk_g2s(ring0 + stage * kChunkBytes, gsrc + (int64_t)c * kChunkBytes, bytes, mbar0 + 8 * stage);
        if (F8) bulk_g2s(scale0 + stage * kScaleStageBytes, a.scales + s0, sbytes, mbar0 + 8 * stage);
    };

    // ---- 2a. start streaming this CTA's pooled rows (the latency overlaps what follows)
    uint32_t g0 = 0;                      // barrier generation at launch (thread 0 only)
    if (tid == 0) {
        for (int c = 0; c < n_chunks && c < kRingStages; ++c) issue_stage(c, c);
        g0 = ld_acquire_u32(&rs->gen);
    }
    // the query rows for the attention step, bf16, prefetched now
    for (int i = tid; i < Hq * kHeadDim / 8; i += kStepThreads)
        cp_async16(smem_u32(q_b + i * 8), a.q + (int64_t)row * Hq * kHeadDim + i * 8);
    asm volatile("cp.async.commit_group;" ::: "memory");
    // ---- 1a. the four raw key rows of block nb-1 (pooled after the scan, off its critical path)
    if (owner_new && tid < kRatio * kIdxDim / 8)
        cp_async16(smem_u32(rawrows + tid * 8), a.raw_idx_k + (base + kRatio * (nb - 1)) * kIdxDim + tid * 8);
    asm volatile("cp.async.commit_group;" ::: "memory");
    STEP_TRACE(1);

    if (dense) {                          // dense rows re-pool block nb-1 here (no scan)
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        uint16_t v = 0;
        if (owner_new && tid < kIdxDim) {
            const double s4 = (((double)bf16_bits_to_float(rawrows[tid]) +
                                (double)bf16_bits_to_float(rawrows[kIdxDim + tid])) +
                               (double)bf16_bits_to_float(rawrows[2 * kIdxDim + tid])) +
                              (double)bf16_bits_to_float(rawrows[3 * kIdxDim + tid]);
            v = double_to_bf16_rne(s4 * 0.25);
            if (!F8) a.pooled[(boff + nb - 1) * kIdxDim + tid] = v;
        }
        if (F8 && owner_new) quantize_newest(a, boff + nb - 1, true, v, newrow8, s_amax);   // CTA-uniform
        prefetch_next_read(a);
    }

    bool balanced = dense;                // the row's whole selection is known to every CTA
    int bar_k = 0;                        // barriers completed by this row in this launch
    unsigned long long t64 = 0ull;        // exact threshold key (dense: select all)
    int out_off = (int)lo;                // this CTA's first output slot (dense: lo)
    if (!dense) {
        // ---- 2b. scan: bulk copies into a 4-stage ring, scores -> keys + histogram
        for (int i = tid; i < kHistBins; i += kStepThreads) hist[i] = 0;
        // bf16: lane l holds dims 4l .. 4l+3 of 8 rows at a time (dot4_bf16 order); FP8: 8 lanes
        // per row, 16 dims per lane
        float qf[F8 ? 16 : 4];
        if constexpr (F8) {
            float qa[8], qb[8];
            unpack8(ldg_nc_v4(a.q_idx + (int64_t)row * kIdxDim + (lane & 7) * 16), qa);
            unpack8(ldg_nc_v4(a.q_idx + (int64_t)row * kIdxDim + (lane & 7) * 16 + 8), qb);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                qf[e] = qa[e];
                qf[8 + e] = qb[e];
            }
        } else {
            load_q4(a.q_idx + (int64_t)row * kIdxDim, lane, qf);
        }
        const int g8 = lane >> 3, c8 = lane & 7;
        __syncthreads();
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
            const int rows_c = min(kRows, n_tma - c * kRows);
            if constexpr (F8) {
                // 16 warps x 16 rows: each 8-lane group takes one row per step; the score is
                // formed as in index_score_fp8_kernel (same products, order and scale multiply)
                const uint8_t *buf8 = smem + kRingOff + (size_t)stage * kChunkBytes;
                const float *sbuf = reinterpret_cast<const float *>(smem + kScaleOff + (size_t)stage * kScaleStageBytes) +
                                    ((boff + lo + (int64_t)c * kRows) & 3);
#pragma unroll
                for (int it = 0; it < kRows / (4 * kStepWarps); ++it) {
                    const int r = (warp * (kRows / kStepWarps)) + it * 4 + g8;
                    float s = 0.f;
                    if (r < rows_c) {
                        float f[16];
                        e4m3x16_to_f32(*reinterpret_cast<const uint4 *>(buf8 + r * kIdxDim + c8 * 16), f);
#pragma unroll
                        for (int e = 0; e < 16; ++e) s = fmaf(f[e], qf[e], s);
                    }
#pragma unroll
                    for (int o = 4; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                    if (c8 == 0 && r < rows_c) {
                        const uint32_t key = score_key(s * sbuf[r]);
                        keys[c * kRows + r] = key;
                        atomicAdd(&hist[key >> kHistShift], 1u);
                    }
                }
            } else {
                const uint16_t *buf =
                    reinterpret_cast<const uint16_t *>(smem + kRingOff + (size_t)stage * kChunkBytes);
                // 16 warps x 8 rows: 8-byte loads (one row per warp instruction, no bank
                // conflicts), one reduce-scatter for the 8 rows; lanes 4i hold row i's score
                constexpr int kR = kRows / kStepWarps;
                float part[kR];
#pragma unroll
                for (int i = 0; i < kR; ++i) {
                    const int r = warp * kR + i;
                    const uint2 x = r < rows_c ? *reinterpret_cast<const uint2 *>(buf + r * kIdxDim + 4 * lane)
                                               : make_uint2(0u, 0u);
                    part[i] = dot4_bf16(x, qf);
                }
                const float s = reduce_rows<kR>(part, lane);
                const int r = warp * kR + row_of_lane<kR>(lane);
                if ((lane & (32 / kR - 1)) == 0 && r < rows_c) {
                    const uint32_t key = score_key(s);
                    keys[c * kRows + r] = key;
                    atomicAdd(&hist[key >> kHistShift], 1u);
                }
            }
            // the stage is refilled once every warp has read it; no block-wide barrier per chunk
            __syncwarp();
            if (lane == 0) mbar_arrive(mbar0 + 8 * (kRingStages + stage));
            if (tid == 0 && c + kRingStages < n_chunks) {
                if (!mbar_wait_bounded(mbar0 + 8 * (kRingStages + stage), (c / kRingStages) & 1, kWaitLimitNs)) {
                    record_error(a.hdr, QSA_ERR_DEVICE_TIMEOUT, kWhereStep, row);   // the others time out too
                } else {
                    fence_proxy_async_smem();
                    issue_stage(c + kRingStages, stage);
                }
            }
        }
        prefetch_next_read(a);
        // ---- 1b. re-pool block nb-1: exact fp64 mean of its four raw keys, one RNE to bf16
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        uint16_t v = 0;
        if (owner_new && tid < kIdxDim) {
            const double s4 = (((double)bf16_bits_to_float(rawrows[tid]) +
                                (double)bf16_bits_to_float(rawrows[kIdxDim + tid])) +
                               (double)bf16_bits_to_float(rawrows[2 * kIdxDim + tid])) +
                              (double)bf16_bits_to_float(rawrows[3 * kIdxDim + tid]);
            v = double_to_bf16_rne(s4 * 0.25);
            if (!F8) {
                newrow[tid] = v;
                a.pooled[(boff + nb - 1) * kIdxDim + tid] = v;
            }
        }
        if constexpr (F8) {
            if (owner_new) quantize_newest(a, boff + nb - 1, true, v, newrow8, s_amax);   // CTA-uniform
        }
        __syncthreads();
        if (owner_new && warp == 0) {          // the freshly pooled block, from shared memory
            float s = 0.f;
            if constexpr (F8) {
                if (lane < 8) {
                    float f[16];
                    e4m3x16_to_f32(*reinterpret_cast<const uint4 *>(newrow8 + c8 * 16), f);
#pragma unroll
                    for (int e = 0; e < 16; ++e) s = fmaf(f[e], qf[e], s);
                }
#pragma unroll
                for (int o = 4; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                s *= s_amax[4];
            } else {
                float p1[1] = {dot4_bf16(*reinterpret_cast<const uint2 *>(newrow + 4 * lane), qf)};
                s = reduce_rows<1>(p1, lane);
            }
            if (lane == 0) {
                const uint32_t key = score_key(s);
                keys[n_mine - 1] = key;
                atomicAdd(&hist[key >> kHistShift], 1u);
            }
        }
        if (tid == 0) {
            s_n = 0;
            s_cnt[0] = 0;
        }
        __syncthreads();
        STEP_TRACE(2);

        // ---- 3. publish this CTA's exact local top-K. Slot kMaxPub holds 0 when the CTA
        // published every key it has, else its K-th largest key (the smallest published).
        const int K = pub_count(cr);
        unsigned long long *pub = a.pub + (size_t)blockIdx.x * (kMaxPub + 1);
        // with K <= 32 the keys gather in shared memory and are published in block order,
        // so a reader ranks a CTA's selected keys by block id with one ballot
        unsigned long long *dst = K <= 32 ? s_pubk : pub;
        if (K <= 32) {
            if (tid < 32) s_pubk[tid] = 0ull;
            __syncthreads();
        }
        if (n_mine <= K) {
            for (int i = tid; i < K; i += kStepThreads) dst[i] = i < n_mine ? key64_of(keys[i], lo + i) : 0ull;
            if (tid == 0) pub[kMaxPub] = 0ull;
        } else {
            block_find_bin(hist, kHistBins, (uint32_t)K, &s_d, &s_above, s_wsum);
            const uint32_t lb = (uint32_t)s_d;
            // members of the bins >= lb: the top K plus the rest of bin lb
            for (int i = tid; i < n_mine; i += kStepThreads) {
                const uint32_t key = keys[i];
                if ((key >> kHistShift) >= lb) {
                    const uint32_t slot = atomicAdd(&s_n, 1u);
                    if (slot < (uint32_t)(kRingBytes / 8)) ring64[slot] = key64_of(key, lo + i);
                }
            }
            __syncthreads();
            const uint32_t nc = min(s_n, (uint32_t)(kRingBytes / 8));
            if (nc <= (uint32_t)kStepThreads) {
                // rank by counting: the candidate with rank r goes to slot r
                if (tid < (int)nc) {
                    const unsigned long long mine = ring64[tid];
                    uint32_t rank = 0;
                    for (uint32_t j = 0; j < nc; ++j) rank += ring64[j] > mine ? 1u : 0u;
                    if (rank < (uint32_t)K) dst[rank] = mine;
                    if (rank == (uint32_t)K - 1u) pub[kMaxPub] = mine;
                }
            } else {
                // threshold value with exactly K keys at or above it (need not be a key itself)
                const unsigned long long tk = select_kth_key64(ring64, nc, (uint32_t)K, hist, &s_d, &s_above, s_wsum,
                                                               s_red, ring64 + nc, (uint32_t)(kRingBytes / 8) - nc,
                                                               &s_cnt[1]);
                if (tid == 0) s_kmin = ~0ull;
                __syncthreads();
                for (uint32_t i = tid; i < nc; i += kStepThreads) {
                    const unsigned long long k = ring64[i];
                    if (k >= tk) {
                        const uint32_t slot = atomicAdd(&s_cnt[0], 1u);
                        if (slot < (uint32_t)K) dst[slot] = k;
                        atomicMin(&s_kmin, k);
                    }
                }
                __syncthreads();
                if (tid == 0) pub[kMaxPub] = s_kmin;
            }
        }
        if (K <= 32) {                    // ascending block ids; empty slots (0) last
            __syncthreads();
            if (tid < K) {
                const unsigned long long mine = s_pubk[tid];
                const uint32_t bm = mine ? 0xFFFFFFFFu - (uint32_t)mine : 0xFFFFFFFFu;
                uint32_t r = 0;
                for (int j = 0; j < K; ++j) {
                    const unsigned long long o = s_pubk[j];
                    const uint32_t bo = o ? 0xFFFFFFFFu - (uint32_t)o : 0xFFFFFFFFu;
                    r += (bo < bm || (bo == bm && j < tid)) ? 1u : 0u;
                }
                pub[r] = mine;
            }
        }
        STEP_TRACE(3);

        // ---- 4. one barrier; every CTA derives the same threshold and offsets
        const int stall = s_debug == kDebugStallBarrier ? 1 : 0;
        if (bar_sync_fast(rs, g0, bar_k, cr + stall, false, a.hdr, row, &s_flag) < 0) return;
        ++bar_k;
        STEP_TRACE(4);
        const unsigned long long *pub_row = a.pub + (size_t)first * (kMaxPub + 1);
        const int n_slots = cr * K;
        const int log2k = __ffs(K) - 1;
        for (int i = tid; i < n_slots; i += kStepThreads)
            ring64[i] = __ldcg(&pub_row[(size_t)(i >> log2k) * (kMaxPub + 1) + (i & (K - 1))]);
        for (int j = tid; j < cr; j += kStepThreads) s_kth[j] = __ldcg(&pub_row[(size_t)j * (kMaxPub + 1) + kMaxPub]);
        __syncthreads();
        STEP_TRACE(14);
        // empty slots hold 0, below every real key, so they never reach the threshold;
        // exactly 512 published keys are >= t64
        t64 = n_slots <= 8 * kStepThreads
                  ? select_kth_key64_lin(ring64, (uint32_t)n_slots, kBlockTopK, hist, &s_d, &s_above, s_wsum, s_red,
                                         s_fred, ring64 + n_slots, &s_n)
                  : select_kth_key64(ring64, (uint32_t)n_slots, kBlockTopK, hist, &s_d, &s_above, s_wsum, s_red,
                                     ring64 + n_slots, (uint32_t)(kRingBytes / 8 - n_slots), &s_n);
        STEP_TRACE(15);
        // a CTA with unpublished keys whose K-th key reaches the threshold might hold more
        if (tid == 0) s_overflow = 0;
        for (int i = tid; i < kBlockTopK; i += kStepThreads) s_sel[i] = -1;
        if (K <= 32) {
            // one segment of K lanes per publishing CTA: a ballot gives its selected count
            __syncthreads();
            const int seg = lane / K, slot = lane % K;
            const unsigned segmask = K == 32 ? 0xffffffffu : (((1u << K) - 1u) << (seg * K));
            for (int j0 = warp * (32 / K); j0 < cr; j0 += kStepWarps * (32 / K)) {
                const int j = j0 + seg;
                const unsigned long long k = j < cr ? ring64[(j << log2k) + slot] : 0ull;
                const unsigned bal = __ballot_sync(0xffffffffu, j < cr && k >= t64);
                if (slot == 0 && j < cr) {
                    s_cnt[j] = (uint32_t)__popc(bal & segmask);
                    if (s_kth[j] != 0ull && s_kth[j] >= t64) s_overflow = 1;
                }
            }
        } else {
            for (int j = tid; j < cr; j += kStepThreads) s_cnt[j] = 0;
            __syncthreads();
            for (int j = tid; j < cr; j += kStepThreads)
                if (s_kth[j] != 0ull && s_kth[j] >= t64) s_overflow = 1;
            // offsets: selected published keys of every earlier CTA of the row
            for (int i = tid; i < n_slots; i += kStepThreads)
                if (ring64[i] >= t64) atomicAdd(&s_cnt[i >> log2k], 1u);
        }
        __syncthreads();
        if (!s_overflow && K <= 64) {
            // Every CTA rebuilds the row's whole ascending selection from the published keys:
            // exclusive prefix of the per-CTA counts, then each selected key's slot is its
            // CTA's offset plus the number of selected keys of that CTA with a lower block id.
            if (warp == 0) {
                uint32_t run = 0;
                for (int j0 = 0; j0 < cr; j0 += 32) {
                    const uint32_t v = j0 + lane < cr ? s_cnt[j0 + lane] : 0u;
                    uint32_t inc = v;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
                        if (lane >= o) inc += t;
                    }
                    if (j0 + lane < cr) s_cnt[j0 + lane] = run + inc - v;
                    run += __shfl_sync(0xffffffffu, inc, 31);
                }
            }
            __syncthreads();
            if (K <= 32) {
                // a CTA's keys are published in block order: the rank by block id among its
                // selected keys is the number of selected lanes below in the segment
                const int seg = lane / K, slot = lane % K;
                const unsigned segmask = K == 32 ? 0xffffffffu : (((1u << K) - 1u) << (seg * K));
                for (int j0 = warp * (32 / K); j0 < cr; j0 += kStepWarps * (32 / K)) {
                    const int j = j0 + seg;
                    const unsigned long long k = j < cr ? ring64[(j << log2k) + slot] : 0ull;
                    const bool sel = j < cr && k >= t64;
                    const unsigned bal = __ballot_sync(0xffffffffu, sel);
                    if (sel) {
                        const uint32_t pos = s_cnt[j] + (uint32_t)__popc(bal & segmask & ((1u << lane) - 1u));
                        if (pos < (uint32_t)kBlockTopK) s_sel[pos] = (int32_t)(0xFFFFFFFFu - (uint32_t)k);
                    }
                }
            } else {
                for (int i = tid; i < n_slots; i += kStepThreads) {
                    const unsigned long long k = ring64[i];
                    if (k >= t64) {
                        const int j = i >> log2k;
                        const uint32_t blk = 0xFFFFFFFFu - (uint32_t)k;
                        uint32_t r = 0;
                        for (int s2 = 0; s2 < K; ++s2) {
                            const unsigned long long k2 = ring64[(j << log2k) + s2];
                            r += (k2 >= t64 && 0xFFFFFFFFu - (uint32_t)k2 < blk) ? 1u : 0u;
                        }
                        const uint32_t pos = s_cnt[j] + r;
                        if (pos < (uint32_t)kBlockTopK) s_sel[pos] = (int32_t)blk;
                    }
                }
            }
            __syncthreads();
            balanced = true;
        } else if (!s_overflow) {
            warp_sum_prefix(s_cnt, jj, &s_flag);
            __syncthreads();
            out_off = s_flag;
        } else {
            // ---- exact fallback: global histogram -> threshold bin -> candidates -> threshold
            // (the shared histogram was reused as radix scratch: rebuild it from the keys)
            for (int i = tid; i < kHistBins; i += kStepThreads) hist[i] = 0;
            __syncthreads();
            for (int i = tid; i < n_mine; i += kStepThreads) atomicAdd(&hist[keys[i] >> kHistShift], 1u);
            __syncthreads();
            uint32_t *ghist = a.hist + (size_t)row * kHistBins;
            for (int i = tid; i < kHistBins; i += kStepThreads)
                if (hist[i]) atomicAdd(&ghist[i], hist[i]);
            const int rb1 = bar_arrive(rs, g0, bar_k, cr, a.hdr, row, &s_flag);
            if (rb1 < 0) return;
            if (rb1 == 1) {
                for (int i = tid; i < kHistBins; i += kStepThreads) {
                    hist[i] = __ldcg(&ghist[i]);
                    ghist[i] = 0;
                }
                __syncthreads();
                block_find_bin(hist, kHistBins, kBlockTopK, &s_d, &s_above, s_wsum);
                if (tid == 0) {
                    rs->t1 = s_d;
                    rs->need = kBlockTopK - (int)s_above;
                }
                bar_release(rs, g0, bar_k);
            }
            ++bar_k;
            __syncthreads();
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
                if (is_c && slot < (uint32_t)nb) cands[slot] = key64_of(key, lo + i);
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
            const int rb2 = bar_arrive(rs, g0, bar_k, cr, a.hdr, row, &s_flag);
            if (rb2 < 0) return;
            if (rb2 == 1) {
                const uint32_t n_c = min(__ldcg(&rs->cand_count), (uint32_t)nb);
                const uint32_t need = (uint32_t)__ldcg(&rs->need);
                const bool in_smem = n_c <= (uint32_t)(kRingBytes / 8);
                if (in_smem)
                    for (uint32_t i = tid; i < n_c; i += kStepThreads) ring64[i] = __ldcg(&cands[i]);
                __syncthreads();
                const unsigned long long *src = in_smem ? ring64 : cands;
                const unsigned long long tt =
                    n_c ? select_kth_key64(src, n_c, need, hist, &s_d, &s_above, s_wsum, s_red) : ~0ull;
                for (int i = tid; i < cr; i += kStepThreads) s_cnt[i] = 0;
                __syncthreads();
                for (uint32_t i = tid; i < n_c; i += kStepThreads) {
                    const unsigned long long k = src[i];
                    if (k >= tt) {
                        const int64_t b = (int64_t)(0xFFFFFFFFu - (uint32_t)k);
                        int j = (int)(b * cr / nb);
                        while (j + 1 < cr && nb * (j + 1) / cr <= b) ++j;
                        while (j > 0 && nb * j / cr > b) --j;
                        atomicAdd(&s_cnt[j], 1u);
                    }
                }
                __syncthreads();
                for (int j = tid; j < cr; j += kStepThreads) s_cnt[j] += (uint32_t)__ldcg(&rs->definite[j]);
                __syncthreads();
                if (warp == 0) {            // exclusive prefix over the CTAs of the row
                    uint32_t run = 0;
                    for (int j0 = 0; j0 < cr; j0 += 32) {
                        const uint32_t v = j0 + lane < cr ? s_cnt[j0 + lane] : 0u;
                        uint32_t inc = v;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
                            if (lane >= o) inc += t;
                        }
                        if (j0 + lane < cr) rs->offset[j0 + lane] = (int32_t)(run + inc - v);
                        run += __shfl_sync(0xffffffffu, inc, 31);
                    }
                    if (lane == 0) {
                        rs->t64 = tt;
                        rs->cand_count = 0;
                        if (run != (uint32_t)kBlockTopK) record_error(a.hdr, QSA_ERR_DEVICE_BOUNDS, kWhereStep, row);
                    }
                }
                bar_release(rs, g0, bar_k);
            }
            ++bar_k;
            __syncthreads();
            t64 = __ldcg(&rs->t64);
            out_off = __ldcg(&rs->offset[jj]);
        }
        STEP_TRACE(5);
    }

    // ---- 5a. selected blocks, ascending, and their output slots. A balanced sparse row writes
    // an equal share of the rebuilt list; otherwise each CTA lists its own range's blocks.
    int32_t *blocks_row = a.blocks + (int64_t)row * kBlockTopK;
    int nsel = 0;
    if (balanced && !dense) {
        nsel = kBlockTopK;
        for (int i = kBlockTopK * jj / cr + tid; i < kBlockTopK * (jj + 1) / cr; i += kStepThreads)
            blocks_row[i] = s_sel[i];
    }
    for (int base_i = 0; base_i < n_mine && !(balanced && !dense); base_i += kStepThreads) {
        const int i = base_i + tid;
        const bool take = i < n_mine && (dense || key64_of(keys[i], lo + i) >= t64);
        const unsigned bal = __ballot_sync(0xffffffffu, take);
        if (lane == 0) s_wsum[warp] = __popc(bal);
        __syncthreads();
        const uint32_t wc = lane < kStepWarps ? s_wsum[lane] : 0u;
        uint32_t inc = wc;
#pragma unroll
        for (int o = 1; o < kStepWarps; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        const int total = (int)__shfl_sync(0xffffffffu, inc, kStepWarps - 1);
        int before = nsel + (int)(__shfl_sync(0xffffffffu, inc, warp) - __shfl_sync(0xffffffffu, wc, warp));
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
    STEP_TRACE(6);

    // ---- 5b. attention over this CTA's tokens (+ the query's own block in the last CTA).
    // Tokens go in chunks of 32: each chunk's K and V rows (all KV heads) are gathered into
    // one half of the ring with 16-byte async copies, two chunks in flight, and computed from
    // shared memory. The scores' keys and histogram are dead now: q (fp32) and the chunk's
    // logits reuse their space.
    // token sequence: the list's blocks (4 tokens each) then the query's own block; a balanced
    // row splits it evenly over its CTAs, otherwise each CTA takes its own list (+ the tail in
    // the row's last CTA)
    const int n_tail_row = (int)(p - kRatio * nb + 1);
    const int n_list = dense ? (int)nb : nsel;
    int t_lo = 0, t_hi = kRatio * nsel + (jj == cr - 1 ? n_tail_row : 0);
    if (balanced) {
        const int n_total = kRatio * n_list + n_tail_row;
        t_lo = n_total * jj / cr;
        t_hi = n_total * (jj + 1) / cr;
    }
    const int n_tok = t_hi - t_lo;
    const int tok_bytes = chunk_tok_bytes<KV8>(Hkv);                   // K rows | V rows (| scales)
    const int row_bytes = KV8 ? Hkv * kHeadDim : 2 * Hkv * kHeadDim;   // one token's K (or V) row
    float *pw = reinterpret_cast<float *>(smem + kHistOff);            // [Hq][kAttnTok]
    unsigned char *const kv_ring = smem + kRingOff;                    // two halves of 64 KiB
    const int n_att_chunks = (n_tok + kAttnTok - 1) / kAttnTok;
    asm volatile("cp.async.wait_group 0;" ::: "memory");            // the prefetched query
    __syncthreads();                                                   // ring, keys, hist are free
    RcChunk *const rcc = reinterpret_cast<RcChunk *>(smem + kKeysOff);   // RC: [2], chunks in flight
    const int64_t rc_lo = RC ? (int64_t)row * a.rc_slots / a.B : 0;
    const int64_t rc_n = RC ? (int64_t)(row + 1) * a.rc_slots / a.B - rc_lo : 1;
    auto gather = [&](int c) {
        const int n = min(kAttnTok, n_tok - c * kAttnTok);
        if constexpr (RC)
            gather_chunk_rc(a, reinterpret_cast<uint16_t *>(kv_ring + (size_t)(c & 1) * (kRingBytes / 2)), rcc + (c & 1),
                            t_lo + c * kAttnTok, n, n_list, dense, s_sel, nb, base, p, row, Hkv * kHeadDim, rc_lo,
                            rc_n);
        else
            gather_chunk<KV8>(a, kv_ring + (size_t)(c & 1) * (kRingBytes / 2), t_lo + c * kAttnTok, n, n_list, dense,
                              s_sel, nb, base, p, row);
    };
    for (int c = 0; c < n_att_chunks && c < 2; ++c) gather(c);
    if (tid < Hq) {
        s_m[tid] = -INFINITY;
        s_l[tid] = 0.f;
    }
    const int kv_t = tid >> 8, d_t = tid & 255;          // PV ownership: (KV head, dim)
    // logits ownership: a warp takes HW of one KV head's G query heads (their 8 dims per lane
    // in registers) and every wpg-th token of the chunk, so K is read once per token and group
    constexpr int HW = G < 8 ? G : 8;
    constexpr int NH = G / HW;
    const int n_groups = Hkv * NH, wpg = kStepWarps / n_groups;
    const int grp = warp / wpg, tsub = warp % wpg;
    const int kv_l = grp / NH, hs_l = grp % NH;
    uint4 qr[HW];                                          // bf16 x 8 per head, unpacked in the dot
#pragma unroll
    for (int g = 0; g < HW; ++g)
        qr[g] = grp < n_groups ? *reinterpret_cast<const uint4 *>(q_b + (kv_l * G + hs_l * HW + g) * kHeadDim + lane * 8)
                               : make_uint4(0, 0, 0, 0);
    float acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = 0.f;
    for (int c = 0; c < n_att_chunks; ++c) {
        const int t0 = c * kAttnTok;
        const int n = min(kAttnTok, n_tok - t0);
        const unsigned char *buf = kv_ring + (size_t)(c & 1) * (kRingBytes / 2);
        if (c + 1 < n_att_chunks) asm volatile("cp.async.wait_group 1;" ::: "memory");
        else asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();
        if (c == 0) STEP_TRACE(10);
        // logits: each warp's HW heads against every wpg-th token (8 dims per lane), the
        // HW partial dots reduced and scattered over the lanes at once
        if (grp < n_groups) {
            for (int i = tsub; i < n; i += wpg) {
                const unsigned char *tok = buf + (size_t)i * tok_bytes;
                float kf[8];
                float ks = 1.f;   // FP8 K: the scale of this lane's 128-dim group (lanes 0-15, 16-31)
                if constexpr (KV8) {
                    e4m3x8_to_f32(*reinterpret_cast<const uint2 *>(tok + kv_l * kHeadDim + lane * 8), kf);
                    ks = reinterpret_cast<const float *>(tok + 2 * row_bytes)[kv_l * 2 + (lane >> 4)];
                } else {
                    unpack8(*reinterpret_cast<const uint4 *>(tok + kv_l * kHeadDim * 2 + lane * 16), kf);
                }
                float v[HW];
#pragma unroll
                for (int g = 0; g < HW; ++g) {
                    float qf[8];
                    unpack8(qr[g], qf);
                    float sum = kf[0] * qf[0];   // bf16 x bf16 and bf16 x E4M3 products are exact in fp32
#pragma unroll
                    for (int e = 1; e < 8; ++e) sum = fmaf(kf[e], qf[e], sum);
                    v[g] = KV8 ? sum * ks : sum;
                }
                int idx = 0;
                const float tot = warp_reduce_scatter<HW>(v, lane, &idx);
                if ((lane & (32 / HW - 1)) == 0) pw[(kv_l * G + hs_l * HW + idx) * kAttnTok + i] = tot * a.scale_log2;
            }
        }
        __syncthreads();
        if (c == 0) STEP_TRACE(11);
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
            if constexpr (KV8) {
                const unsigned char *vcol = buf + row_bytes + kv_t * kHeadDim + d_t;
                const unsigned char *vscl = buf + 2 * row_bytes + (Hkv + kv_t) * 8 + (d_t >> 7) * 4;
#pragma unroll 4
                for (int i = 0; i < n; ++i) {
                    const float v = e4m3_to_f32(vcol[(size_t)i * tok_bytes]) *
                                    *reinterpret_cast<const float *>(vscl + (size_t)i * tok_bytes);
#pragma unroll
                    for (int g = 0; g < G; ++g) acc[g] = fmaf(pw[(kv_t * G + g) * kAttnTok + i], v, acc[g]);
                }
            } else {
                const int tok_elems = tok_bytes / 2;
                const uint16_t *vcol = reinterpret_cast<const uint16_t *>(buf) + tok_elems / 2 + kv_t * kHeadDim + d_t;
#pragma unroll 4
                for (int i = 0; i < n; ++i) {
                    const float v = bf16_bits_to_float(vcol[(size_t)i * tok_elems]);
#pragma unroll
                    for (int g = 0; g < G; ++g) acc[g] = fmaf(pw[(kv_t * G + g) * kAttnTok + i], v, acc[g]);
                }
            }
        }
        __syncthreads();
        if (c == 0) STEP_TRACE(12);
        if (c + 2 < n_att_chunks) gather(c + 2);
    }
    // partial of this CTA. The row's region holds (m, l) per CTA, [cr][2 Hq], then the acc
    // values in blocks of 32 outputs, [Hq x 256 / 32][cr][32]: a warp writes one 128-byte
    // line per block, and a merging CTA reads each source's line of a block at once.
    float *rowpart = a.part + (size_t)first * Hq * (kHeadDim + 2);
    float *ml_r = rowpart, *acc_r = rowpart + (size_t)cr * 2 * Hq;
    if (tid < Hq) {
        ml_r[(size_t)jj * 2 * Hq + tid] = s_m[tid];
        ml_r[(size_t)jj * 2 * Hq + Hq + tid] = s_l[tid];
    }
    if (kv_t < Hkv) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int o = (kv_t * G + g) * kHeadDim + d_t;
            acc_r[((size_t)(o >> 5) * cr + jj) * 32 + (o & 31)] = acc[g];
        }
    }
    STEP_TRACE(7);

    // ---- 6. merge the row's partials; each CTA finishes a slice of the Hq x 256 outputs
    if (bar_sync_fast(rs, g0, bar_k, cr, true, a.hdr, row, &s_flag) < 0) return;
    ++bar_k;
    __syncthreads();
    if constexpr (RC) {                              // no CTA of the row reads the cache any more
        // the last two chunks are still in the ring's two halves
        for (int cl = max(n_att_chunks - 2, 0); cl < n_att_chunks; ++cl) {
            fill_rc(a, reinterpret_cast<const uint16_t *>(kv_ring + (size_t)(cl & 1) * (kRingBytes / 2)), rcc + (cl & 1),
                    min(kAttnTok, n_tok - cl * kAttnTok), Hkv * kHeadDim, reinterpret_cast<int *>(smem + kHistOff));
            __syncthreads();
        }
    }
    STEP_TRACE(8);
    // the next launch on the stream may be scheduled now (it waits for this one to finish)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int n_out = Hq * kHeadDim;
    const int o_lo = n_out * jj / cr, o_hi = n_out * (jj + 1) / cr;
    const int h_lo = o_lo / kHeadDim, h_hi = o_hi > o_lo ? (o_hi - 1) / kHeadDim : h_lo - 1;
    const int nh = h_hi - h_lo + 1;
    float *w_s = reinterpret_cast<float *>(smem + kRingOff);           // [nh][cr] m, then weights
    float *l_s = w_s + 2 * kMaxGroup * kMaxStepCtas;                    // [nh][cr] l
    float *red = l_s + 2 * kMaxGroup * kMaxStepCtas;                    // [warps][32]
    constexpr int kJ = kMaxStepCtas / kStepWarps;                       // sources per warp
    const int b0 = o_lo >> 5, b1 = o_hi > o_lo ? (o_hi - 1) >> 5 : b0 - 1;
    // one round trip: (m, l) of the slice's heads and the first block of acc values
    for (int idx = tid; idx < nh * cr; idx += kStepThreads) {
        const int h = h_lo + idx / cr, j = idx % cr;
        w_s[idx] = __ldcg(&ml_r[(size_t)j * 2 * Hq + h]);
        l_s[idx] = __ldcg(&ml_r[(size_t)j * 2 * Hq + Hq + h]);
    }
    // a slice spans at most two blocks of 32 outputs when the row has 128 CTAs or more: both
    // are loaded in the same round trip (further blocks, for fewer CTAs, one trip each)
    float v[kJ], v2[kJ];
    auto load_block = [&](int b, float (&dst)[kJ]) {
#pragma unroll
        for (int k = 0; k < kJ; ++k) {
            const int j = warp + k * kStepWarps;
            dst[k] = j < cr ? __ldcg(&acc_r[((size_t)b * cr + j) * 32 + lane]) : 0.f;
        }
    };
    if (b0 <= b1) load_block(b0, v);
    if (b0 + 1 <= b1) load_block(b0 + 1, v2);
    __syncthreads();
    STEP_TRACE(13);
    for (int hh = warp; hh < nh; hh += kStepWarps) {
        float M = -INFINITY;
        for (int j = lane; j < cr; j += 32) M = fmaxf(M, w_s[hh * cr + j]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float L = 0.f;
        for (int j = lane; j < cr; j += 32) {
            const float mj = w_s[hh * cr + j];
            const float wj = (mj == -INFINITY) ? 0.f : exp2f(mj - M);
            w_s[hh * cr + j] = wj;
            L = fmaf(l_s[hh * cr + j], wj, L);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        if (lane == 0) {
            s_m[hh] = M;
            s_l[hh] = L;
        }
    }
    __syncthreads();
    for (int b = b0; b <= b1; ++b) {
        if (b == b0 + 1) {
#pragma unroll
            for (int k = 0; k < kJ; ++k) v[k] = v2[k];
        } else if (b > b0 + 1) {
            load_block(b, v);
        }
        const int h = b >> 3;                                           // 8 blocks of 32 per head
        const float *wv = w_s + (h - h_lo) * cr;
        float sacc = 0.f;
#pragma unroll
        for (int k = 0; k < kJ; ++k) {
            const int j = warp + k * kStepWarps;
            if (j < cr) sacc = fmaf(v[k], wv[j], sacc);
        }
        red[warp * 32 + lane] = sacc;
        __syncthreads();
        if (warp == 0) {
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < kStepWarps; ++w) tot += red[w * 32 + lane];
            const int o = b * 32 + lane;
            if (o >= o_lo && o < o_hi) {
                const float L = s_l[h - h_lo];
                a.out[(int64_t)row * n_out + o] = float_to_bf16_bits(tot / L);
                if (a.lse != nullptr && (o & (kHeadDim - 1)) == 0)
                    a.lse[(int64_t)row * Hq + h] = (s_m[h - h_lo] + log2f(L)) * kLn2;
            }
        }
        __syncthreads();
    }
    STEP_TRACE(9);
#undef STEP_TRACE
}

// ------------------------------------------------------------------------------ launch helpers
// Each translation unit that includes this header instantiates the kernels of one K/V format.

// Co-resident CTAs of decode_step_kernel<G, F8, KV8> on device `dev` (cached; 0 on error).
template <int G, bool F8, bool KV8, bool RC = false>
int step_ctas_g(int dev) {
    static int cache[64];   // per device, 0 = unknown
    int &slot = cache[dev];
    if (slot == 0) {
        auto kern = decode_step_kernel<G, F8, KV8, RC>;
        const int smem = (int)step_smem<F8>();
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
        int sms = 0, per_sm = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStepThreads, smem) != cudaSuccess)
            return 0;
        if (per_sm < 1) return 0;
        slot = min(sms * per_sm, kMaxStepCtas);
    }
    return slot;
}

// Cooperative launch (every CTA co-resident: the row barriers need it) as a programmatic
// dependent of the previous kernel on the stream.
template <int G, bool F8, bool KV8, bool RC = false>
cudaError_t launch_step_g(const StepArgs &a, int ctas, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = step_smem<F8>();
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, decode_step_kernel<G, F8, KV8, RC>, a);
}

template <bool F8, bool KV8, bool RC = false>
int step_grid_for(int G, int dev) {
    switch (G) {
        case 1: return step_ctas_g<1, F8, KV8, RC>(dev);
        case 2: return step_ctas_g<2, F8, KV8, RC>(dev);
        case 4: return step_ctas_g<4, F8, KV8, RC>(dev);
        case 8: return step_ctas_g<8, F8, KV8, RC>(dev);
        case 16: return step_ctas_g<16, F8, KV8, RC>(dev);
        default: return 0;
    }
}

template <bool F8, bool KV8, bool RC = false>
cudaError_t step_launch_for(const StepArgs &a, int G, int ctas, cudaStream_t st) {
    switch (G) {
        case 1: return launch_step_g<1, F8, KV8, RC>(a, ctas, st);
        case 2: return launch_step_g<2, F8, KV8, RC>(a, ctas, st);
        case 4: return launch_step_g<4, F8, KV8, RC>(a, ctas, st);
        case 8: return launch_step_g<8, F8, KV8, RC>(a, ctas, st);
        case 16: return launch_step_g<16, F8, KV8, RC>(a, ctas, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// Grid size and launch of the FP8-K/V kernels (decode_step_kv8.cu) and of the row-cache kernels
// (bf16 keys and K/V, decode_step_rc.cu).
int step_grid_kv8(int G, bool fp8_keys, int dev);
cudaError_t step_launch_kv8(const StepArgs &a, int G, bool fp8_keys, int ctas, cudaStream_t st);
int step_grid_rc(int G, int dev);
cudaError_t step_launch_rc(const StepArgs &a, int G, int ctas, cudaStream_t st);

}  // namespace qsa
