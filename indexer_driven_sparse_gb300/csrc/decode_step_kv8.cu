// Fused decode layer-step with FP8 K/V rows: the instantiations of decode_step_kernel with
// KV8 = true (both indexer-key formats), compiled beside the bf16-K/V ones.
#include "decode_step.cuh"

namespace qsa {

int step_grid_kv8(int G, bool fp8_keys, int dev) {
    return fp8_keys ? step_grid_for<true, true>(G, dev) : step_grid_for<false, true>(G, dev);
}

cudaError_t step_launch_kv8(const StepArgs &a, int G, bool fp8_keys, int ctas, cudaStream_t st) {
    return fp8_keys ? step_launch_for<true, true>(a, G, ctas, st) : step_launch_for<false, true>(a, G, ctas, st);
}

}  // namespace qsa
