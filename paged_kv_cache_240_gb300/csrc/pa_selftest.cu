// pa_selftest.cu -- a self-check of the kernels' bounded waits.
//
// Every wait inside the library's kernels goes through mbar_wait, which gives up
// after a limit and lets the kernel report PA_FLAG_TIMEOUT instead of hanging.
// The kernel here waits, with a limit the caller gives, on an mbarrier that no
// thread ever arrives at -- with no copy of any kind in flight -- and on one
// whose phase has already completed, and records what each wait returned.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa_dev {

__global__ void __launch_bounds__(64) pa_wait_selftest_kernel(long long limit,
                                                              long long* result, int32_t* err) {
  __shared__ uint64_t never, done;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&never, 1);
    mbar_init(&done, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_arrive(&done);  // phase 0 of `done` completes
  __syncthreads();
  if (warp == 0) {
    // one thread's wait, timed, then a wait that must succeed at once
    if (lane == 0) {
      const long long t0 = clock64();
      const bool ok = mbar_wait(&never, 0, limit);
      const long long t1 = clock64();
      result[0] = ok ? 0 : 1;
      result[3] = t1 - t0;
      if (!ok) set_flag(err, PA_FLAG_TIMEOUT);
    }
    const bool fine = __all_sync(0xffffffffu, mbar_wait(&done, 0, limit));
    if (lane == 0) result[2] = fine ? 1 : 0;
  } else {
    // a whole warp's wait whose verdict is the warp's vote (the tensor-memory
    // prefill kernel's form)
    const bool ok = __all_sync(0xffffffffu, mbar_wait(&never, 0, limit));
    if (lane == 0) {
      result[1] = ok ? 0 : 1;
      if (!ok) set_flag(err, PA_FLAG_TIMEOUT);
    }
  }
}

}  // namespace pa_dev

extern "C" pa_status pa_selftest_bounded_wait(long long limit_cycles, long long* result,
                                              int32_t* err_flag, void* stream) {
  if (limit_cycles < 1 || limit_cycles > pa_dev::kWaitLimitCycles || !result || !err_flag ||
      !pa_internal::aligned16(result) || !pa_internal::aligned16(err_flag))
    return PA_ERR_INVALID_ARG;
  pa_dev::pa_wait_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(
      limit_cycles, result, err_flag);
  return pa_internal::cuda_status(cudaGetLastError());
}
