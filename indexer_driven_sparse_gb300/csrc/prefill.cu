// a6 — prefill chunk: every chunk query i at p0 + i attends its own selection
// ("3090x3で 314 万コンテキスト", section "ちなみにこの欠点").
#include "qsa_internal.cuh"

namespace qsa {

size_t prefill_scratch_bytes(int Nc, int Hq, int Hkv) {
    (void)Nc;
    (void)Hq;
    (void)Hkv;
    return 0;
}

cudaError_t launch_sparse_prefill(const AttnArgs &a, int interval_tokens, WsHeader *hdr, void *scratch,
                                  size_t scratch_bytes, cudaStream_t st) {
    (void)interval_tokens;
    (void)scratch;
    (void)scratch_bytes;
    return launch_attn_rows(a, hdr, st);
}

}  // namespace qsa
