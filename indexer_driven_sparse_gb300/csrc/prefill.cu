// a6 — prefill chunk: every chunk query i at p0 + i attends its own selection
// ("3090x3で 314 万コンテキスト", section "ちなみにこの欠点").
#include "qsa_internal.cuh"

namespace qsa {

// the tensor-core path's plan (per query tile: its chunk records); the CUDA-core path needs none
size_t prefill_scratch_bytes(int Nc, int Hq, int Hkv) { return prefill_tc_plan_bytes(Nc, Hq, Hkv); }

cudaError_t launch_sparse_prefill(const AttnArgs &a, int interval_tokens, WsHeader *hdr, void *scratch,
                                  size_t scratch_bytes, cudaStream_t st) {
    if (a.rows == 0) return cudaSuccess;
    // tensor-core interval walk for 8 or 16 query heads per KV head; otherwise one CTA per
    // (query, KV head) on the CUDA cores
    if (prefill_tc_supported(a.n_q_heads, a.n_kv_heads))
        return launch_prefill_tc(a, interval_tokens, hdr, scratch, scratch_bytes, st);
    return launch_attn_rows(a, hdr, st);
}

}  // namespace qsa
