// Self-test of the bounded waits that every mbarrier wait of the tcgen05 kernels uses.
// The pages have no counterpart: this exists so that a test can make a wait run out on the
// GPU without a fault or a hang. One CTA waits on an mbarrier that nothing ever arrives
// on, through the same helper as the attention kernel with a short limit, and reports
// GT_ERR_TIMEOUT; nothing is in flight and no tensor memory is held, so it simply returns.
#include "gt_internal.cuh"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace gt {

__global__ void __launch_bounds__(32)
wait_timeout_kernel(uint64_t limit_ns, int32_t *err, int64_t *waited_ns) {
  pdl_enter();
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  const uint64_t t0 = tc::globaltimer();
  const bool arrived = tc::mbar_wait(&bar, 0, &abort_flag, limit_ns);  // nothing arrives
  const uint64_t t1 = tc::globaltimer();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!arrived) set_err(err, GT_ERR_TIMEOUT);
    if (waited_ns) *waited_ns = (int64_t)(t1 - t0);
  }
}

}  // namespace gt

using namespace gt;

GT_API int gt_selftest_wait_timeout(int64_t limit_ns, int32_t *err, int64_t *waited_ns,
                                    gt_stream_t stream) {
  GT_TRACE("gt_selftest_wait_timeout");
  if (limit_ns < 1 || limit_ns > 1000000000ll) return GT_ERR_ARG;
  if (!err) return GT_ERR_ARG;
  return launch(wait_timeout_kernel, dim3(1), dim3(32), 0, (cudaStream_t)stream,
                (uint64_t)limit_ns, err, waited_ns);
}
