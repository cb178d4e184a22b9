// Host launcher of the FP8 K/V dequantiser (fp8_keys.cu), used by the FP8 K/V prefill.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace qsa {

// FP8 K/V rows (codes [n_rows][256], scales [n_rows][2]) -> bf16 rows, each element
// code x scale rounded once to bf16: K rows into k_out and, when v_codes is not NULL, V rows
// into v_out in the same launch (n_rows 256-dim rows each).
cudaError_t launch_dequantize_kv_fp8(const uint8_t *k_codes, const float *k_scales, uint16_t *k_out,
                                     const uint8_t *v_codes, const float *v_scales, uint16_t *v_out, int64_t n_rows,
                                     cudaStream_t st);

}  // namespace qsa
