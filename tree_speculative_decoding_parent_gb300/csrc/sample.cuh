// Launcher of the per-row target draw at temperature T > 0 (sample.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gt {

// sample[r] = the Gumbel-max draw of logit row r (rows x V, row-major f32) at temperature
// T, seed and step. With ids != NULL the same pass also writes the row's top-k of the
// unscaled logits (k <= 16) to ids / vals [rows][k], as gt_vocab_topk would; err receives
// checked builds' reports. Returns a gt_status (GT_ERR_ARG for a temperature that is not
// finite and positive or whose reciprocal overflows).
int sample_launch(const float *logits, int rows, int V, float temperature, uint64_t seed,
                  uint64_t step, int32_t *sample, cudaStream_t s, int k = 0,
                  int32_t *ids = nullptr, float *vals = nullptr, int32_t *err = nullptr);

}  // namespace gt
