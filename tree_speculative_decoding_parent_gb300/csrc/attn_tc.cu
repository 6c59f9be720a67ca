// tcgen05 tree attention for bf16 (not yet enabled: every shape takes the SIMT path).
#include "attn_tc.cuh"
#include "gt_internal.cuh"

namespace gt {

bool attn_tc_supported(int, int) { return false; }

int attn_tc_launch(const void *, const void *, const void *, const uint64_t *, const int32_t *,
                   const int32_t *, int, int, int, int, int, float, const AttnWs &, int32_t *,
                   cudaStream_t) {
  return GT_ERR_SHAPE;
}

}  // namespace gt
