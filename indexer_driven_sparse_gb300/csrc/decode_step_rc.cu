// Fused decode layer-step with the VRAM row cache in front of host-resident bf16 K/V: the
// instantiations of decode_step_kernel with RC = true (bf16 indexer keys and K/V rows).
#include "decode_step.cuh"

namespace qsa {

int step_grid_rc(int G, int dev) { return step_grid_for<false, false, true>(G, dev); }

cudaError_t step_launch_rc(const StepArgs &a, int G, int ctas, cudaStream_t st) {
    return step_launch_for<false, false, true>(a, G, ctas, st);
}

}  // namespace qsa
