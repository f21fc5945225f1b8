// Self-test of the device-side failure reporting: a kernel whose wait can
// never be satisfied gives up after a short bound, records its code in the
// error word and returns, leaving the context usable. The waits are the same
// kinds the kernels use: an mbarrier phase (bounded by a poll count) and a
// counter in global memory (bounded by time on the global timer).
#include <cuda_runtime.h>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

namespace {

__global__ void selftest_wait_kernel(int kind, uint32_t limit, const unsigned* flag, uint32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  if (kind == 0) {
    // nothing ever arrives on the barrier
    mbar_wait_n(&bar, 0, err, kErrSelftestBarrier, limit);
  } else {
    // nothing ever raises the counter; limit in microseconds
    uint64_t t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
      if (v >= 1u) break;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > 1000ull * limit) {
        report_error(err, kErrSelftestFlag);
        break;
      }
      __nanosleep(256);
    }
  }
}

}  // namespace

cudaError_t launch_selftest_wait(int kind, uint32_t limit, const unsigned* flag, uint32_t* err,
                                 cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(kind, limit, flag, err);
  return cudaGetLastError();
}

}  // namespace qg
