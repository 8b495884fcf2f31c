// Self-test of the bounded waits every pipelined kernel of the library uses
// (test hook).  One CTA of two warps: lane 0 of warp 0 waits, with a short
// limit, on an mbarrier nothing arrives on; lane 0 of warp 1 waits on
// another such barrier with the kernels' full limit.  When the short wait
// runs out it flags MLA_DEVERR_TIMEOUT and raises the CTA's abort flag, and
// the long wait must then give up at its next check instead of running to
// its own limit, which is how a stalled pipeline stage stops the other
// roles of its CTA.  Nothing faults, traps or spins without a bound.
#include <cuda_runtime.h>

#include "launch.h"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

__global__ void __launch_bounds__(64) selftest_wait_kernel(uint32_t* error_word, uint64_t limit_ns,
                                                           unsigned long long* elapsed_ns) {
  __shared__ uint64_t bars[2];
  __shared__ volatile int abort_s;
  if (threadIdx.x == 0) {
    abort_s = 0;
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    const uint64_t t0 = global_timer_ns();
    // phase 0 of either barrier never completes: nothing arrives
    const bool ok = warp == 0 ? mbar_wait(&bars[0], 0, error_word, &abort_s, limit_ns)
                              : mbar_wait(&bars[1], 0, nullptr, &abort_s);
    const uint64_t t1 = global_timer_ns();
    if (!ok && elapsed_ns != nullptr) elapsed_ns[warp] = static_cast<unsigned long long>(t1 - t0);
  }
}

}  // namespace

int launch_selftest_wait(uint32_t* error_word, int64_t limit_ns, unsigned long long* elapsed_ns,
                         cudaStream_t stream) {
  selftest_wait_kernel<<<1, 64, 0, stream>>>(error_word, static_cast<uint64_t>(limit_ns), elapsed_ns);
  return launch_status();
}

}  // namespace mla
