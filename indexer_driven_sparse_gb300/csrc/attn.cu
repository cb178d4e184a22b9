// a4 + a5 — gathered-K/V GQA attention over a query's selected blocks plus its own
// block, as split partials (m, l, acc) merged by log-sum-exp.
//   "3090x3で 314 万コンテキスト", section "なぜ": a generated token reads K/V of exactly
//   2048 selected tokens; section "カーネルを書き換えずに済む": row address
//   (tok * n_kv_heads + kv_head) * head_dim + d.
//   "GLM-5.3 最適化 第2部", section "DCP": partials over disjoint key sets are merged by
//   log-sum-exp.
// One CTA handles one (row, KV head, split) and all G = Hq/Hkv query heads that share
// the KV head, so each gathered K/V row is read once for the whole group. Tokens are
// processed in chunks of 64 with an online softmax in base 2 (logits pre-scaled by
// scale * log2 e). Decode splits a row's <= 2052 attended tokens into 64-token splits
// that run on separate CTAs and merges them in a second kernel.
#include "qsa_internal.cuh"

namespace qsa {

constexpr int kAttnThreads = 256;            // one thread per head_dim element in the PV step
constexpr int kChunk = 64;
constexpr int kSplitTok = 64;
constexpr int kMaxSplits = (kMaxAttended + kSplitTok - 1) / kSplitTok;   // 33

struct RowGeom {
    int64_t base;     // flat index of the row's token 0
    int p;            // query position
    int nb;           // visible blocks
    int cnt;          // selected blocks
    int nJ;           // attended tokens
    bool ok;
};

__device__ __forceinline__ RowGeom row_geom(const AttnArgs &a, int row) {
    RowGeom g;
    if (a.tok_off != nullptr) {
        g.base = a.tok_off[row];
        g.p = a.ctx_len[row];
        const int64_t end = a.tok_off[row + 1];
        g.ok = g.p >= 0 && g.base >= 0 && end <= a.n_tok && g.base + g.p + 1 <= end;
    } else {
        g.base = 0;
        g.p = a.p0 + row;
        g.ok = g.p >= 0 && (int64_t)g.p + 1 <= a.n_tok;
    }
    g.nb = g.p >= 0 ? (g.p >> 2) : 0;
    g.cnt = a.count[row];
    g.ok = g.ok && g.cnt >= 0 && g.cnt <= min(kBlockTopK, g.nb);
    g.nJ = g.ok ? kRatio * g.cnt + (g.p - kRatio * g.nb + 1) : 0;
    return g;
}

template <int G, bool kSplit>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(AttnArgs a, WsHeader *hdr, float *__restrict__ part) {
    const int row = blockIdx.z, g = blockIdx.y, split = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int Hq = a.n_q_heads, Hkv = a.n_kv_heads;

    const RowGeom geo = row_geom(a, row);
    if (!geo.ok) {
        if (tid == 0 && split == 0 && g == 0) record_error(hdr, QSA_ERR_DEVICE_BOUNDS, a.where, row);
        return;
    }
    int j0 = 0, j1 = geo.nJ;
    if (kSplit) {
        j0 = split * kSplitTok;
        if (j0 >= geo.nJ) return;
        j1 = min(geo.nJ, j0 + kSplitTok);
    }

    __shared__ float qs[G][kHeadDim];
    __shared__ int64_t toks[kChunk];
    __shared__ float pw[G][kChunk];
    __shared__ float m_s[G], l_s[G], alpha_s[G];

    for (int i = tid; i < G * kHeadDim; i += kAttnThreads) {
        const int h = i / kHeadDim, d = i % kHeadDim;
        const uint16_t qb = a.q[((int64_t)row * Hq + g * G + h) * kHeadDim + d];
        qs[h][d] = bf16_bits_to_float(qb) * a.scale_log2;
    }
    if (tid < G) {
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.f;
    }
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.f;
    const int32_t *brow = a.blocks + (int64_t)row * kBlockTopK;
    __syncthreads();

    for (int c0 = j0; c0 < j1; c0 += kChunk) {
        const int n = min(kChunk, j1 - c0);
        if (tid < n) {
            const int j = c0 + tid;
            int tok;
            if (j < kRatio * geo.cnt) {
                const int b = brow[j >> 2];
                if (b < 0 || b >= geo.nb) {
                    record_error(hdr, QSA_ERR_DEVICE_BOUNDS, a.where, row);
                    tok = geo.p;                 // safe substitute; the status word flags the row
                } else {
                    tok = kRatio * b + (j & 3);
                }
            } else {
                tok = kRatio * geo.nb + (j - kRatio * geo.cnt);
            }
            toks[tid] = geo.base + tok;
        }
        __syncthreads();
        // logits: one warp per token, 8 dims per lane
        for (int i = warp; i < n; i += kAttnThreads / 32) {
            float kf[8];
            unpack8(ldg_nc_v4(a.k_cache + (toks[i] * Hkv + g) * kHeadDim + lane * 8), kf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) s = fmaf(kf[e], qs[h][lane * 8 + e], s);
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane == 0) pw[h][i] = s;
            }
        }
        __syncthreads();
        // online softmax: one warp per head
        for (int h = warp; h < G; h += kAttnThreads / 32) {
            const float x0 = lane < n ? pw[h][lane] : -INFINITY;
            const float x1 = lane + 32 < n ? pw[h][lane + 32] : -INFINITY;
            float cm = fmaxf(x0, x1);
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
            const float mo = m_s[h];
            const float mn = fmaxf(mo, cm);
            const float e0 = lane < n ? exp2f(x0 - mn) : 0.f;
            const float e1 = lane + 32 < n ? exp2f(x1 - mn) : 0.f;
            if (lane < n) pw[h][lane] = e0;
            if (lane + 32 < n) pw[h][lane + 32] = e1;
            float sm = e0 + e1;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
            if (lane == 0) {
                const float al = (mo == -INFINITY) ? 0.f : exp2f(mo - mn);
                alpha_s[h] = al;
                l_s[h] = l_s[h] * al + sm;
                m_s[h] = mn;
            }
        }
        __syncthreads();
        // PV: thread tid owns output dim d = tid
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] *= alpha_s[h];
        for (int i = 0; i < n; ++i) {
            const float v = bf16_bits_to_float(__ldg(a.v_cache + (toks[i] * Hkv + g) * kHeadDim + tid));
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] = fmaf(pw[h][i], v, acc[h]);
        }
        __syncthreads();
    }

    if (kSplit) {
        // partial layout per (row, kv head, split): m[G], l[G], acc[G][256]
        float *dst = part + (((int64_t)row * Hkv + g) * kMaxSplits + split) * (G * (kHeadDim + 2));
        if (tid < G) {
            dst[tid] = m_s[tid];
            dst[G + tid] = l_s[tid];
        }
#pragma unroll
        for (int h = 0; h < G; ++h) dst[2 * G + h * kHeadDim + tid] = acc[h];
    } else {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float o = acc[h] / l_s[h];
            a.out[((int64_t)row * Hq + g * G + h) * kHeadDim + tid] = float_to_bf16_bits(o);
        }
        if (a.lse != nullptr && tid < G) a.lse[(int64_t)row * Hq + g * G + tid] = (m_s[tid] + log2f(l_s[tid])) * kLn2;
    }
}

// LSE merge of a row's splits: one CTA per (query head, row), one thread per dim.
template <int G>
__global__ void __launch_bounds__(kAttnThreads) merge_kernel(AttnArgs a, const float *__restrict__ part) {
    const int h = blockIdx.x, row = blockIdx.y, tid = threadIdx.x;
    const RowGeom geo = row_geom(a, row);
    if (!geo.ok) return;
    const int n_split = (geo.nJ + kSplitTok - 1) / kSplitTok;
    const int g = h / G, hl = h % G;
    const float *src = part + ((int64_t)row * a.n_kv_heads + g) * kMaxSplits * (G * (kHeadDim + 2));
    const int stride = G * (kHeadDim + 2);
    float M = -INFINITY;
    for (int s = 0; s < n_split; ++s) M = fmaxf(M, src[s * stride + hl]);
    float L = 0.f, acc = 0.f;
    for (int s = 0; s < n_split; ++s) {
        const float* ps = src + s * stride;
        const float w = exp2f(ps[hl] - M);
        L = fmaf(ps[G + hl], w, L);
        acc = fmaf(ps[2 * G + hl * kHeadDim + tid], w, acc);
    }
    a.out[((int64_t)row * a.n_q_heads + h) * kHeadDim + tid] = float_to_bf16_bits(acc / L);
    if (a.lse != nullptr && tid == 0) a.lse[(int64_t)row * a.n_q_heads + h] = (M + log2f(L)) * kLn2;
}

size_t decode_scratch_bytes(int B, int Hq, int Hkv) {
    const int G = Hq / Hkv;
    return (size_t)B * Hkv * kMaxSplits * G * (kHeadDim + 2) * sizeof(float);
}

template <int G>
static cudaError_t launch_decode_g(const AttnArgs &a, WsHeader *hdr, float *part, cudaStream_t st) {
    dim3 grid(kMaxSplits, a.n_kv_heads, a.rows);
    attn_kernel<G, true><<<grid, kAttnThreads, 0, st>>>(a, hdr, part);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    merge_kernel<G><<<dim3(a.n_q_heads, a.rows), kAttnThreads, 0, st>>>(a, part);
    return cudaGetLastError();
}

cudaError_t launch_sparse_decode(const AttnArgs &a, WsHeader *hdr, void *scratch, size_t scratch_bytes,
                                 cudaStream_t st) {
    if (a.rows == 0) return cudaSuccess;
    if (scratch_bytes < decode_scratch_bytes(a.rows, a.n_q_heads, a.n_kv_heads)) return cudaErrorInvalidValue;
    float *part = static_cast<float *>(scratch);
    switch (a.n_q_heads / a.n_kv_heads) {
        case 1: return launch_decode_g<1>(a, hdr, part, st);
        case 2: return launch_decode_g<2>(a, hdr, part, st);
        case 4: return launch_decode_g<4>(a, hdr, part, st);
        case 8: return launch_decode_g<8>(a, hdr, part, st);
        case 16: return launch_decode_g<16>(a, hdr, part, st);
        default: return cudaErrorInvalidValue;
    }
}

// Per-query reference-order prefill: every chunk query attends its own selection in one
// CTA per (query, KV head). Used where the tensor-core interval walk does not apply.
template <int G>
static cudaError_t launch_rows_g(const AttnArgs &a, cudaStream_t st, WsHeader *hdr) {
    attn_kernel<G, false><<<dim3(1, a.n_kv_heads, a.rows), kAttnThreads, 0, st>>>(a, hdr, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_attn_rows(const AttnArgs &a, WsHeader *hdr, cudaStream_t st) {
    if (a.rows == 0) return cudaSuccess;
    switch (a.n_q_heads / a.n_kv_heads) {
        case 1: return launch_rows_g<1>(a, st, hdr);
        case 2: return launch_rows_g<2>(a, st, hdr);
        case 4: return launch_rows_g<4>(a, st, hdr);
        case 8: return launch_rows_g<8>(a, st, hdr);
        case 16: return launch_rows_g<16>(a, st, hdr);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qsa
