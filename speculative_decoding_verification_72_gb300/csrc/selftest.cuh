// Self-test of the failure path every streaming kernel shares: a bounded
// mbarrier wait that nothing completes gives up after its limit, and the
// kernel reports SV_STATUS_TIMEOUT and returns instead of hanging.
#pragma once

#include "sv_common.cuh"

namespace sv {

// One thread-block of one warp: lane 0 initialises an mbarrier that expects
// one arrival, never arrives on it, and waits on its first phase with
// mbar_wait_bounded. No bulk copy is issued, so nothing is in flight when the
// block exits.
__global__ void __launch_bounds__(32) selftest_wait_kernel(int32_t* out_status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  fence_barrier_init();
  const bool completed = mbar_wait_bounded(smem_u32(&bar), 0);
  out_status[0] = completed ? 0 : SV_STATUS_TIMEOUT;
}

}  // namespace sv
