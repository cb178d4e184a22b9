// a3 — fixed-budget block selection: the min(512, nb) best blocks of each row,
// ties to the lower block id, written in ascending id order ("3090x3で 314 万コンテキスト",
// section "なぜ"; tie rule as in "125B MoE を 3090 3 枚で運用する vLLM 最適化編" section 3.3).
//
// One CTA per row. Long rows (at least 16,384 blocks) first try one streaming pass: a
// sample of every 64th score sets value-linear bins and a cut keeping about 3 x 512 of the
// row; the pass gathers every score at or above the cut as an exact 64-bit key, and the
// top 512 of those are resolved by bins and a rank among the boundary bin's members. When
// fewer than 512 clear the cut (or too many), or for shorter rows, three streaming passes
// over the row (the first from HBM, the others mostly from L2):
//   1. the row's finite max and min;
//   2. a histogram over 4096 bins that are linear in the score value (monotone in the
//      score, so bins above the one holding the k-th best are wholly selected). Linear
//      bins spread scores evenly, where bins on the float's top bits crowd a few
//      exponents and serialise the shared-memory atomics;
//   3. the blocks in higher bins are appended to the selection, the blocks in the k-th
//      bin become candidates, ranked exactly by their 64-bit keys (score key, then lower
//      id first) with a bitonic sort in shared memory.
// The 512 ids are then sorted ascending. Rows the bins cannot split (all scores equal,
// no finite range, or more than 4096 candidates in one bin) take an exact three-digit
// radix select on the 32-bit score keys instead.
//
// Two more modes serve the fused prefill selection (qsa_prefill_select): in candidate mode
// a row's candidates come from the scoring epilogue (every score at or above a floor that
// at least 512 scores reach, already in ascending block order), so the top 512 are the
// keys at or above the 512th largest, compacted in order with no sort; rows whose
// candidates overflowed are flagged. In fallback mode only the flagged rows run, streaming
// the full scores as above.
#include "qsa_internal.cuh"

#include <float.h>

namespace qsa {

constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kLinBins = 4096;
constexpr int kCandCap = 4096;
constexpr int kCandBins = 1024;                 // bins over the sampled path's candidates
constexpr int kScanBatch = 4;                   // 16-byte loads a thread keeps in flight per sweep
static_assert(kCandCap * 2 >= kLinBins, "the histogram lives in the candidate buffer");

// Calls f(i, v, valid) over the row with every thread taking the same number of calls
// (so f may use warp votes); 16-byte loads for the aligned body.
template <class F>
__device__ __forceinline__ void row_scan(const float *__restrict__ s, int64_t nb, F &&f) {
    const int tid = threadIdx.x;
    const int64_t mis = (int64_t)(((16 - ((uintptr_t)s & 15)) & 15) >> 2);   // elements before 16-B alignment
    const int64_t head = mis < nb ? mis : nb;
    if (head > 0) {
        const bool ok = tid < head;
        f((int64_t)tid, ok ? __ldg(s + tid) : 0.f, ok);
    }
    const int64_t nvec = (nb - head) >> 2;
    const float4 *v4 = reinterpret_cast<const float4 *>(s + head);
    for (int64_t j0 = 0; j0 < nvec; j0 += kScanBatch * kTopkThreads) {
        float4 x[kScanBatch];                    // all loads of the batch in flight at once
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u) {
            const int64_t j = j0 + u * kTopkThreads + tid;
            x[u] = j < nvec ? __ldg(v4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u) {
            const int64_t j = j0 + u * kTopkThreads + tid;
            const bool ok = j < nvec;
            const int64_t i = head + 4 * j;
            f(i, x[u].x, ok);
            f(i + 1, x[u].y, ok);
            f(i + 2, x[u].z, ok);
            f(i + 3, x[u].w, ok);
        }
    }
    const int64_t t0 = head + 4 * nvec;
    if (t0 < nb) {
        const bool ok = t0 + tid < nb;
        f(t0 + tid, ok ? __ldg(s + t0 + tid) : 0.f, ok);
    }
}

// The score of a 64-bit key (score key << 32 | ~id): NaN for the NaN key.
__device__ __forceinline__ float key_score(uint64_t key) {
    const uint32_t k = (uint32_t)(key >> 32);
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Bin of a score, non-decreasing in the score for any vmin and scale > 0 (values outside
// the range clamp to the end bins): NaN and -inf lowest, +inf highest.
__device__ __forceinline__ int lin_bin(float v, float vmin, float scale) {
    if (v != v || v == -INFINITY) return 0;
    if (v == INFINITY) return kLinBins - 1;
    const float t = (v - vmin) * scale;
    if (!(t > 0.f)) return 0;
    return t >= (float)(kLinBins - 2) ? kLinBins - 2 : (int)t;
}

// Block-wide: the bin b* (counting from the top) where the running count first reaches
// `need`, and the count strictly above it. Each thread owns kLinBins / kTopkThreads bins.
template <int NBINS = kLinBins>
__device__ void find_bin_from_top(const uint32_t *hist, uint32_t need, int *b_out, uint32_t *above_out,
                                  uint32_t *wtot) {
    constexpr int per = NBINS / kTopkThreads;
    static_assert(per >= 1 && NBINS % kTopkThreads == 0, "bins per thread");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t h[per], sum = 0;
#pragma unroll
    for (int k = 0; k < per; ++k) {
        h[k] = hist[tid * per + k];
        sum += h[k];
    }
    uint32_t suf = sum;                       // inclusive suffix sum within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += v;
    }
    if (lane == 0) wtot[warp] = suf;
    __syncthreads();
    uint32_t higher = 0;
    for (int w = warp + 1; w < kTopkWarps; ++w) higher += wtot[w];
    const uint32_t above = higher + suf - sum;        // count in bins above this thread's
    if (above < need && above + sum >= need) {
        uint32_t run = above;
        int b = per - 1;
        for (; b > 0; --b) {
            if (run + h[b] >= need) break;
            run += h[b];
        }
        *b_out = tid * per + b;
        *above_out = run;
    }
    __syncthreads();
}

// Bitonic sort of n (a power of two, <= 4096) 64-bit keys in shared memory.
__device__ void bitonic_u64(uint64_t *a, int n, bool descending) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += kTopkThreads) {
                const int l = i ^ j;
                if (l > i) {
                    const bool up = ((i & k) == 0) != descending;
                    const uint64_t x = a[i], y = a[l];
                    if ((x > y) == up) {
                        a[i] = y;
                        a[l] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
}

__device__ void bitonic_i32_asc(int32_t *a, int n) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += kTopkThreads) {
                const int l = i ^ j;
                if (l > i) {
                    const bool up = (i & k) == 0;
                    const int32_t x = a[i], y = a[l];
                    if ((x > y) == up) {
                        a[i] = y;
                        a[l] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
}

// Exact fallback: three-digit (11/11/10-bit) radix select on the 32-bit keys, then one
// pass in index order keeping every key > T and the first `need` keys == T.
__device__ void radix_select_row(const float *__restrict__ s, int64_t nb, int32_t *out, uint32_t *hist,
                                 uint32_t *wtot, int *s_b, uint32_t *s_above, uint32_t *written_out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0, pmask = 0, need = kBlockTopK;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = shifts[pass];
        const uint32_t dmask = (1u << widths[pass]) - 1u;
        for (int i = tid; i < kLinBins; i += kTopkThreads) hist[i] = 0;
        __syncthreads();
        for (int64_t i = tid; i < nb; i += kTopkThreads) {
            const uint32_t key = score_key(__ldg(s + i));
            if ((key & pmask) == prefix) atomicAdd(&hist[(key >> sh) & dmask], 1u);
        }
        __syncthreads();
        find_bin_from_top(hist, need, s_b, s_above, wtot);
        prefix |= (uint32_t)*s_b << sh;
        pmask |= dmask << sh;
        need -= *s_above;
        __syncthreads();
    }
    const uint32_t T = prefix, need_eq = need;
    uint32_t written = 0, eq_seen = 0;
    for (int64_t base = 0; base < nb; base += kTopkThreads) {
        const int64_t i = base + tid;
        const uint32_t key = i < nb ? score_key(__ldg(s + i)) : 0u;
        const bool gt = i < nb && key > T;
        const bool eq = i < nb && key == T;
        const unsigned beq = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) wtot[warp] = __popc(beq);
        __syncthreads();
        uint32_t eq_before = eq_seen, eq_total = 0;
        for (int w = 0; w < kTopkWarps; ++w) {
            if (w < warp) eq_before += wtot[w];
            eq_total += wtot[w];
        }
        eq_before += __popc(beq & ((1u << lane) - 1u));
        const bool take = gt || (eq && eq_before < need_eq);
        const unsigned bt = __ballot_sync(0xffffffffu, take);
        __syncthreads();
        if (lane == 0) wtot[warp] = __popc(bt);
        __syncthreads();
        uint32_t pos = written, t_total = 0;
        for (int w = 0; w < kTopkWarps; ++w) {
            if (w < warp) pos += wtot[w];
            t_total += wtot[w];
        }
        pos += __popc(bt & ((1u << lane) - 1u));
        if (take && pos < kBlockTopK) out[pos] = (int32_t)i;
        written += t_total;
        eq_seen += eq_total;
        __syncthreads();
    }
    *written_out = written;
}

__global__ void __launch_bounds__(kTopkThreads, 3) topk_rows_kernel(const float *__restrict__ scores, int64_t ld,
                                                                    const int32_t *q_pos, int32_t *__restrict__ blocks,
                                                                    int32_t *__restrict__ count, WsHeader *hdr,
                                                                    TopkCandidates tc) {
    __shared__ uint64_t cand[kCandCap];        // the histogram shares this space (used before the candidates)
    uint32_t *hist = reinterpret_cast<uint32_t *>(cand);
    __shared__ int32_t sel[kBlockTopK];
    __shared__ uint32_t hist2[kCandBins];
    __shared__ uint64_t s_eq[kTopkThreads];
    __shared__ uint32_t s_neq;
    __shared__ uint32_t wtot[kTopkWarps];
    __shared__ float s_red[2][kTopkWarps];
    __shared__ int s_b;
    __shared__ uint32_t s_above, s_nsel, s_ncand, s_written;
    __shared__ uint64_t s_thr64;

    const int row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tc.fallback_only && tc.fb_rows[row] == 0) return;   // this row was settled from its candidates
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
    const float *s = scores != nullptr ? scores + (int64_t)row * ld : nullptr;   // none in candidate mode
    const unsigned lt = (1u << lane) - 1u;

    // Exact top 512 of nc candidate keys in cand[] (512 <= nc <= kCandCap): 1024 bins linear in
    // their scores, the threshold bin's members ranked by key, the sure ones taken directly;
    // the ids are written ascending. Returns false (nothing written) when the bins cannot
    // split the candidates. Called by every thread of the CTA.
    auto finish_candidates = [&](uint32_t nc) -> bool {
        // exact top 512 of the candidates: 1024 bins linear in their scores, the
        // threshold bin's members ranked by key, the sure ones taken directly
        float cmin = FLT_MAX, cmax = -FLT_MAX;
        for (uint32_t k = tid; k < nc; k += kTopkThreads) {
            const float v = key_score(cand[k]);
            if (fabsf(v) <= FLT_MAX) {
                cmin = fminf(cmin, v);
                cmax = fmaxf(cmax, v);
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
            cmin = fminf(cmin, __shfl_xor_sync(0xffffffffu, cmin, o));
        }
        if (lane == 0) {
            s_red[0][warp] = cmax;
            s_red[1][warp] = cmin;
        }
        for (int i = tid; i < kCandBins; i += kTopkThreads) hist2[i] = 0;
        if (tid == 0) {
            s_nsel = 0;
            s_neq = 0;
        }
        __syncthreads();
        cmax = s_red[0][0];
        cmin = s_red[1][0];
        for (int w = 1; w < kTopkWarps; ++w) {
            cmax = fmaxf(cmax, s_red[0][w]);
            cmin = fminf(cmin, s_red[1][w]);
        }
        const float cscale = cmax > cmin ? (float)(kCandBins - 2) / (cmax - cmin) : 0.f;
        if (cscale > 0.f && cscale <= FLT_MAX) {
            auto cbin = [&](float v) -> int {
                if (v != v || v == -INFINITY) return 0;
                if (v == INFINITY) return kCandBins - 1;
                const float t = (v - cmin) * cscale;
                if (!(t > 0.f)) return 0;
                return t >= (float)(kCandBins - 2) ? kCandBins - 2 : (int)t;
            };
            for (uint32_t k = tid; k < nc; k += kTopkThreads) atomicAdd(&hist2[cbin(key_score(cand[k]))], 1u);
            __syncthreads();
            find_bin_from_top<kCandBins>(hist2, kBlockTopK, &s_b, &s_above, wtot);
            const int bd = s_b;
            const uint32_t need_eq = kBlockTopK - s_above;
            const uint32_t n_eq = hist2[bd];
            if (n_eq <= (uint32_t)kTopkThreads) {
                // sure keys -> their ids; the threshold bin's keys -> a small list
                for (uint32_t k0 = 0; k0 < nc; k0 += kTopkThreads) {
                    const uint32_t k = k0 + tid;
                    const uint64_t key = k < nc ? cand[k] : 0ull;
                    const int b = k < nc ? cbin(key_score(key)) : -1;
                    const bool sure = b > bd, eq = b == bd;
                    const unsigned bs = __ballot_sync(0xffffffffu, sure);
                    const unsigned be = __ballot_sync(0xffffffffu, eq);
                    uint32_t o1 = 0, o2 = 0;
                    if (lane == 0) {
                        if (bs) o1 = atomicAdd(&s_nsel, (uint32_t)__popc(bs));
                        if (be) o2 = atomicAdd(&s_neq, (uint32_t)__popc(be));
                    }
                    o1 = __shfl_sync(0xffffffffu, o1, 0);
                    o2 = __shfl_sync(0xffffffffu, o2, 0);
                    if (sure) sel[o1 + __popc(bs & lt)] = (int32_t)(0xFFFFFFFFu - (uint32_t)key);
                    if (eq) s_eq[o2 + __popc(be & lt)] = key;
                }
                __syncthreads();
                if (tid < (int)n_eq) {
                    const uint64_t mine = s_eq[tid];
                    uint32_t rank = 0;
                    for (uint32_t j = 0; j < n_eq; ++j) rank += s_eq[j] > mine ? 1u : 0u;
                    if (rank < need_eq) sel[s_above + rank] = (int32_t)(0xFFFFFFFFu - (uint32_t)mine);
                }
                __syncthreads();
                bitonic_i32_asc(sel, kBlockTopK);
                for (int i = tid; i < kBlockTopK; i += kTopkThreads) out[i] = sel[i];
                if (tid == 0) {
                    count[row] = kBlockTopK;
                    if (s_nsel != s_above || s_neq != n_eq) record_error(hdr, QSA_ERR_DEVICE_BOUNDS, kWhereTopk, row);
                }
                return true;
            }
        }
        return false;
    };


    // Exact top 512 of nc candidate keys already in ascending block order in cand[]: the
    // 512th largest key by bins over their scores and a rank among the boundary bin's members,
    // then an order-preserving compaction of the keys at or above it (no sort). Returns false
    // (nothing written) when the bins cannot split the candidates.
    auto finish_ordered = [&](uint32_t nc) -> bool {
        float cmin = FLT_MAX, cmax = -FLT_MAX;
        for (uint32_t k = tid; k < nc; k += kTopkThreads) {
            const float v = key_score(cand[k]);
            if (fabsf(v) <= FLT_MAX) {
                cmin = fminf(cmin, v);
                cmax = fmaxf(cmax, v);
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
            cmin = fminf(cmin, __shfl_xor_sync(0xffffffffu, cmin, o));
        }
        if (lane == 0) {
            s_red[0][warp] = cmax;
            s_red[1][warp] = cmin;
        }
        for (int i = tid; i < kCandBins; i += kTopkThreads) hist2[i] = 0;
        if (tid == 0) s_neq = 0;
        __syncthreads();
        cmax = s_red[0][0];
        cmin = s_red[1][0];
        for (int w = 1; w < kTopkWarps; ++w) {
            cmax = fmaxf(cmax, s_red[0][w]);
            cmin = fminf(cmin, s_red[1][w]);
        }
        const float cscale = cmax > cmin ? (float)(kCandBins - 2) / (cmax - cmin) : 0.f;
        if (!(cscale > 0.f && cscale <= FLT_MAX)) return false;
        auto cbin = [&](float v) -> int {
            if (v != v || v == -INFINITY) return 0;
            if (v == INFINITY) return kCandBins - 1;
            const float t = (v - cmin) * cscale;
            if (!(t > 0.f)) return 0;
            return t >= (float)(kCandBins - 2) ? kCandBins - 2 : (int)t;
        };
        for (uint32_t k = tid; k < nc; k += kTopkThreads) atomicAdd(&hist2[cbin(key_score(cand[k]))], 1u);
        __syncthreads();
        find_bin_from_top<kCandBins>(hist2, kBlockTopK, &s_b, &s_above, wtot);
        const int bd = s_b;
        const uint32_t need_eq = kBlockTopK - s_above, n_eq = hist2[bd];
        if (n_eq > (uint32_t)kTopkThreads) return false;
        for (uint32_t k = tid; k < nc; k += kTopkThreads) {
            const uint64_t key = cand[k];
            if (cbin(key_score(key)) == bd) s_eq[atomicAdd(&s_neq, 1u)] = key;
        }
        __syncthreads();
        if (tid < (int)n_eq) {                  // the boundary bin's need_eq-th largest key
            const uint64_t mine = s_eq[tid];
            uint32_t rank = 0;
            for (uint32_t j = 0; j < n_eq; ++j) rank += s_eq[j] > mine ? 1u : 0u;
            if (rank == need_eq - 1u) s_thr64 = mine;
        }
        __syncthreads();
        const uint64_t t64 = s_thr64;
        // contiguous candidates per thread keep the order; a block scan places them
        const uint32_t per = (nc + kTopkThreads - 1) / kTopkThreads;
        const uint32_t i0 = min(nc, tid * per), i1 = min(nc, i0 + per);
        uint32_t cnt = 0;
        for (uint32_t k = i0; k < i1; ++k) cnt += cand[k] >= t64 ? 1u : 0u;
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) wtot[warp] = incl;
        __syncthreads();
        uint32_t pos = incl - cnt;
        for (int w = 0; w < warp; ++w) pos += wtot[w];
        for (uint32_t k = i0; k < i1; ++k) {
            const uint64_t key = cand[k];
            if (key >= t64) {
                if (pos < (uint32_t)kBlockTopK) out[pos] = (int32_t)(0xFFFFFFFFu - (uint32_t)key);
                ++pos;
            }
        }
        if (tid == 0) {
            count[row] = kBlockTopK;
            if (s_neq != n_eq) record_error(hdr, QSA_ERR_DEVICE_BOUNDS, kWhereTopk, row);
        }
        return true;
    };

    // ---- candidate mode: the row's candidates were gathered by the scoring epilogue (every
    // score at or above a floor that at least 512 scores reach), 64-bit keys in per-segment slots
    if (tc.slots != nullptr) {
        const uint8_t *cn = tc.scnt + (size_t)row * tc.n_segs;
        const uint64_t *sl = tc.slots + (size_t)row * tc.n_segs * kSelSlots;
        // ceil(n_segs / threads) consecutive segments per thread, so their loads spread widely
        const int per = (tc.n_segs + kTopkThreads - 1) / kTopkThreads;
        uint32_t c[kSelSegsPerThread], mine = 0;
        bool over = false;
#pragma unroll
        for (int k = 0; k < kSelSegsPerThread; ++k) {
            const int t = tid * per + k;
            c[k] = k < per && t < tc.n_segs ? cn[t] : 0u;
            over |= c[k] > (uint32_t)kSelSlots;
            mine += c[k];
        }
        uint32_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) wtot[warp] = incl;
        const bool any_over = __syncthreads_or(over);
        uint32_t base = incl - mine, total = 0;
        for (int w = 0; w < kTopkWarps; ++w) {
            total += wtot[w];
            if (w < warp) base += wtot[w];
        }
        const bool ok = !any_over && total >= (uint32_t)kBlockTopK && total <= (uint32_t)kCandCap;
        if (ok) {
#pragma unroll 1
            for (int k = 0; k < per; ++k) {
                if (c[k] == 0u) continue;
                const uint64_t *src = sl + (size_t)(tid * per + k) * kSelSlots;
                uint64_t x[kSelSlots];              // the segment's loads all in flight at once
#pragma unroll
                for (int e = 0; e < kSelSlots; ++e) x[e] = (uint32_t)e < c[k] ? __ldcg(src + e) : 0ull;
#pragma unroll
                for (int e = 0; e < kSelSlots; ++e)
                    if ((uint32_t)e < c[k]) cand[base + e] = x[e];
                base += c[k];
            }
        }
        __syncthreads();
        if (ok && finish_ordered(total)) return;
        if (tid == 0) {                        // left to the exact path over the stored scores
            tc.fb_rows[row] = 1;
            atomicExch(tc.fb_any, 1);
        }
        return;
    }

    // ---- one pass when a sample places the cut: every 64th score sets value-linear bins
    // and a bin cut keeping about 3 x 512 of the row; one streaming pass gathers every score
    // at or above a floor one bin below the cut as exact 64-bit keys. When at least 512
    // scores clear the floor the row's top 512 are among them. Otherwise (or if they
    // overflow the candidate buffer) the passes below decide.
    constexpr int kSampleStride = 64;
    const int64_t n_s = nb / kSampleStride;
    if (n_s >= 256) {
        float smin = FLT_MAX, smax = -FLT_MAX;
        bool any_s = false;
        for (int64_t k = tid; k < n_s; k += kTopkThreads) {
            const float v = __ldg(s + k * kSampleStride);
            if (fabsf(v) <= FLT_MAX) {
                smin = fminf(smin, v);
                smax = fmaxf(smax, v);
                any_s = true;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
            smin = fminf(smin, __shfl_xor_sync(0xffffffffu, smin, o));
        }
        if (lane == 0) {
            s_red[0][warp] = smax;
            s_red[1][warp] = smin;
        }
        for (int i = tid; i < kLinBins; i += kTopkThreads) hist[i] = 0;
        if (tid == 0) {
            s_ncand = 0;
            s_neq = 0;
        }
        const bool any_sample = __syncthreads_or(any_s);
        smax = s_red[0][0];
        smin = s_red[1][0];
        for (int w = 1; w < kTopkWarps; ++w) {
            smax = fmaxf(smax, s_red[0][w]);
            smin = fminf(smin, s_red[1][w]);
        }
        const float sscale = (float)(kLinBins - 2) / (smax - smin);
        if (any_sample && smax > smin && sscale > 0.f && sscale <= FLT_MAX) {
            for (int64_t k = tid; k < n_s; k += kTopkThreads)
                atomicAdd(&hist[lin_bin(__ldg(s + k * kSampleStride), smin, sscale)], 1u);
            __syncthreads();
            const int64_t want = 3 * ((int64_t)kBlockTopK * n_s + nb - 1) / nb + 8;
            find_bin_from_top(hist, (uint32_t)(want < n_s ? want : n_s), &s_b, &s_above, wtot);
            const int cut = s_b;
            __syncthreads();                    // the candidates overwrite the histogram
            // the candidates are every score at or above a floor one bin below the cut: a
            // threshold set, so when it holds at least 512 scores the row's top 512 are in it
            // (NaN fails the test and ranks below every number anyway)
            const float vlow = smin + (float)(cut - 1) / sscale;
            auto append = [&](int64_t i, float v, bool m) {
                const unsigned bal = __ballot_sync(0xffffffffu, m);
                if (bal) {
                    uint32_t base = 0;
                    if (lane == 0) base = atomicAdd(&s_ncand, (uint32_t)__popc(bal));
                    base = __shfl_sync(0xffffffffu, base, 0);
                    const uint32_t slot = base + __popc(bal & lt);
                    if (m && slot < (uint32_t)kCandCap)
                        cand[slot] = ((uint64_t)score_key(v) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)i);
                }
            };
            auto is_cand = [&](float v) { return v >= vlow; };
            const int64_t mis = (int64_t)(((16 - ((uintptr_t)s & 15)) & 15) >> 2);
            const int64_t head = mis < nb ? mis : nb;
            if (head > 0) {
                const bool okh = tid < head;
                const float v = okh ? __ldg(s + tid) : 0.f;
                append(tid, v, okh && is_cand(v));
            }
            const int64_t nvec = (nb - head) >> 2;
            const float4 *v4 = reinterpret_cast<const float4 *>(s + head);
            for (int64_t j0 = 0; j0 < nvec; j0 += kScanBatch * kTopkThreads) {
                float4 x[kScanBatch];                // all loads of the batch in flight at once
#pragma unroll
                for (int u = 0; u < kScanBatch; ++u) {
                    const int64_t j = j0 + u * kTopkThreads + tid;
                    x[u] = j < nvec ? __ldg(v4 + j) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                }
                // this lane's candidates of the batch as a bit mask; one warp scan gives slots
                uint32_t mk = 0;
#pragma unroll
                for (int u = 0; u < kScanBatch; ++u) {
                    mk |= (is_cand(x[u].x) ? 1u : 0u) << (4 * u);
                    mk |= (is_cand(x[u].y) ? 1u : 0u) << (4 * u + 1);
                    mk |= (is_cand(x[u].z) ? 1u : 0u) << (4 * u + 2);
                    mk |= (is_cand(x[u].w) ? 1u : 0u) << (4 * u + 3);
                }
                const uint32_t cnt = __popc(mk);
                uint32_t incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                uint32_t base = 0;
                if (lane == 31 && incl) base = atomicAdd(&s_ncand, incl);
                base = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
                // only the set bits: the score is read again (an L1 hit) rather than picked out of
                // the batch's registers by a runtime index
                while (mk) {
                    const int bit = __ffs(mk) - 1;
                    mk &= mk - 1u;
                    const int64_t i = head + 4 * (j0 + (bit >> 2) * kTopkThreads + tid) + (bit & 3);
                    if (base < (uint32_t)kCandCap)
                        cand[base] = ((uint64_t)score_key(__ldg(s + i)) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)i);
                    ++base;
                }
            }
            const int64_t t0 = head + 4 * nvec;
            if (t0 < nb) {
                const bool okt = t0 + tid < nb;
                const float v = okt ? __ldg(s + t0 + tid) : 0.f;
                append(t0 + tid, v, okt && is_cand(v));
            }
            __syncthreads();
            const uint32_t nc = s_ncand;
            if (nc >= (uint32_t)kBlockTopK && nc <= (uint32_t)kCandCap && finish_candidates(nc)) return;
        }
        __syncthreads();
    }

    // ---- pass 1: finite max and min
    float vmax = -FLT_MAX, vmin = FLT_MAX;
    bool any = false;
    row_scan(s, nb, [&](int64_t, float v, bool ok) {
        if (ok && fabsf(v) <= FLT_MAX) {
            vmax = fmaxf(vmax, v);
            vmin = fminf(vmin, v);
            any = true;
        }
    });
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
        vmin = fminf(vmin, __shfl_xor_sync(0xffffffffu, vmin, o));
    }
    if (lane == 0) {
        s_red[0][warp] = vmax;
        s_red[1][warp] = vmin;
    }
    for (int i = tid; i < kLinBins; i += kTopkThreads) hist[i] = 0;
    if (tid == 0) {
        s_nsel = 0;
        s_ncand = 0;
    }
    const bool any_finite = __syncthreads_or(any);
    vmax = s_red[0][0];
    vmin = s_red[1][0];
    for (int w = 1; w < kTopkWarps; ++w) {
        vmax = fmaxf(vmax, s_red[0][w]);
        vmin = fminf(vmin, s_red[1][w]);
    }
    const float scale = (float)(kLinBins - 2) / (vmax - vmin);
    // rows the linear bins cannot split take the exact radix select (uniform decision)
    bool linear = any_finite && vmax > vmin && scale > 0.f && scale <= FLT_MAX;

    if (linear) {
        // ---- pass 2: histogram of linear bins
        row_scan(s, nb, [&](int64_t, float v, bool ok) {
            if (ok) atomicAdd(&hist[lin_bin(v, vmin, scale)], 1u);
        });
        __syncthreads();
        find_bin_from_top(hist, kBlockTopK, &s_b, &s_above, wtot);
        if (hist[s_b] > kCandCap) linear = false;
    }
    const uint32_t n_in_bin = linear ? hist[s_b] : 0u;
    __syncthreads();                            // the candidates overwrite the histogram
    if (linear) {
        const int bstar = s_b;
        const uint32_t need_eq = kBlockTopK - s_above;
        // ---- pass 3: append the sure blocks, gather the k-th bin's candidates
        row_scan(s, nb, [&](int64_t i, float v, bool ok) {
            const int b = ok ? lin_bin(v, vmin, scale) : -1;
            const bool sure = b > bstar, maybe = b == bstar;
            const unsigned ms = __ballot_sync(0xffffffffu, sure);
            const unsigned mc = __ballot_sync(0xffffffffu, maybe);
            if (ms | mc) {
                uint32_t bs = 0, bc = 0;
                if (lane == 0) {
                    if (ms) bs = atomicAdd(&s_nsel, __popc(ms));
                    if (mc) bc = atomicAdd(&s_ncand, __popc(mc));
                }
                bs = __shfl_sync(0xffffffffu, bs, 0);
                bc = __shfl_sync(0xffffffffu, bc, 0);
                if (sure) sel[bs + __popc(ms & lt)] = (int32_t)i;
                if (maybe)
                    cand[bc + __popc(mc & lt)] =
                        ((uint64_t)score_key(v) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)i);
            }
        });
        __syncthreads();
        const int nc = (int)s_ncand;
        int n2 = 2;
        while (n2 < nc) n2 <<= 1;
        for (int i = nc + tid; i < n2; i += kTopkThreads) cand[i] = 0ull;   // pads sort last
        __syncthreads();
        bitonic_u64(cand, n2, true);
        const uint32_t base = s_nsel;           // == s_above
        for (uint32_t k = tid; k < need_eq; k += kTopkThreads)
            sel[base + k] = (int32_t)(0xFFFFFFFFu - (uint32_t)(cand[k] & 0xFFFFFFFFull));
        __syncthreads();
        bitonic_i32_asc(sel, kBlockTopK);
        for (int i = tid; i < kBlockTopK; i += kTopkThreads) out[i] = sel[i];
        if (tid == 0) {
            count[row] = kBlockTopK;
            if (base != s_above || nc != (int)n_in_bin)
                record_error(hdr, QSA_ERR_DEVICE_BOUNDS, kWhereTopk, row);
        }
        return;
    }
    radix_select_row(s, nb, out, hist, wtot, &s_b, &s_above, &s_written);
    if (tid == 0) {
        count[row] = kBlockTopK;
        if (s_written != kBlockTopK) record_error(hdr, QSA_ERR_DEVICE_BOUNDS, kWhereTopk, row);
    }
}

size_t topk_scratch_bytes(int Nq, int64_t ld) {
    (void)Nq;
    (void)ld;
    return 0;
}

cudaError_t launch_topk_with(const float *scores, int64_t ld, const int32_t *q_pos, int Nq, int32_t *blocks,
                             int32_t *count, WsHeader *hdr, const TopkCandidates &tc, cudaStream_t st) {
    if (Nq == 0) return cudaSuccess;
    topk_rows_kernel<<<Nq, kTopkThreads, 0, st>>>(scores, ld, q_pos, blocks, count, hdr, tc);
    return cudaGetLastError();
}

cudaError_t launch_topk_blocks(const float *scores, int64_t ld, const int32_t *q_pos, int Nq, int32_t *blocks,
                               int32_t *count, WsHeader *hdr, void *scratch, size_t scratch_bytes, cudaStream_t st) {
    (void)scratch;
    (void)scratch_bytes;
    if (Nq == 0) return cudaSuccess;
    topk_rows_kernel<<<Nq, kTopkThreads, 0, st>>>(scores, ld, q_pos, blocks, count, hdr, TopkCandidates{});
    return cudaGetLastError();
}

}  // namespace qsa
