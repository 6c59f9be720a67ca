// Launcher of the per-row target draw at temperature T > 0 (sample.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gt {

// sample[r] = the Gumbel-max draw of logit row r (rows x V, row-major f32) at temperature
// T, seed and step. Returns a gt_status (GT_ERR_ARG for a temperature that is not finite
// and positive or whose reciprocal overflows).
int sample_launch(const float *logits, int rows, int V, float temperature, uint64_t seed,
                  uint64_t step, int32_t *sample, cudaStream_t s);

}  // namespace gt
