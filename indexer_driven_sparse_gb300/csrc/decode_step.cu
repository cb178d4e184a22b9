// Fused decode layer-step: host side, and the kernels with bf16 K/V rows. The kernel
// template and its description are in decode_step.cuh; the FP8-K/V instantiations are
// compiled in decode_step_kv8.cu.
#include "decode_step.cuh"

namespace qsa {

StepLayout step_layout(int B, int64_t max_blocks, int Hq) { return step_layout_of(B, max_blocks, Hq); }

size_t decode_step_ws_bytes(int B, int64_t max_blocks, int Hq) { return step_layout(B, max_blocks, Hq).total; }

int decode_step_max_keys() { return kMaxKeys; }

RowCacheLayout row_cache_layout(int n_kv_heads, int64_t n_slots) {
    RowCacheLayout L;
    L.rows = 0;
    L.tag = (size_t)n_slots * 2 * n_kv_heads * kHeadDim * 2;
    L.hit = L.tag + (size_t)n_slots * 8;
    L.claim = L.hit + ((size_t)n_slots * 4 + 7) / 8 * 8;
    L.total = L.claim + (size_t)n_slots * 8;
    return L;
}

int decode_step_grid(int G, bool fp8_keys, bool fp8_kv, bool row_cache) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (row_cache) return fp8_keys || fp8_kv ? 0 : step_grid_rc(G, dev);
    if (fp8_kv) return step_grid_kv8(G, fp8_keys, dev);
    return fp8_keys ? step_grid_for<true, false>(G, dev) : step_grid_for<false, false>(G, dev);
}

cudaError_t launch_decode_step(StepArgs a, void *ws, cudaStream_t st) {
    const StepLayout L = step_layout(a.B, a.max_blocks, a.n_q_heads);
    char *w = static_cast<char *>(ws);
    a.hdr = reinterpret_cast<WsHeader *>(w);
    a.rows = reinterpret_cast<void *>(w + L.rows);
    a.hist = reinterpret_cast<uint32_t *>(w + L.hist);
    a.cands = reinterpret_cast<unsigned long long *>(w + L.cands);
    a.part = reinterpret_cast<float *>(w + L.part);
    a.pub = reinterpret_cast<unsigned long long *>(w + L.pub);
    a.trace = reinterpret_cast<unsigned long long *>(w + L.trace);
    const int G = a.n_q_heads / a.n_kv_heads;
    const bool fp8_keys = a.codes != nullptr;
    const bool fp8_kv = a.k_codes != nullptr;
    const bool rc = a.rc_rows != nullptr;
    const int ctas = decode_step_grid(G, fp8_keys, fp8_kv, rc);
    if (ctas < a.B || ctas == 0) return cudaErrorInvalidConfiguration;
    if (rc) return step_launch_rc(a, G, ctas, st);
    if (fp8_kv) return step_launch_kv8(a, G, fp8_keys, ctas, st);
    return fp8_keys ? step_launch_for<true, false>(a, G, ctas, st) : step_launch_for<false, false>(a, G, ctas, st);
}

}  // namespace qsa
