// Self-test of the failure path every tcgen05 kernel relies on: a bounded mbarrier
// wait that runs out records MODA_ERR_TIMEOUT in the device status word, raises the
// CTA's abort flag, and every other wait of the CTA then gives up as well, so the
// kernel returns instead of hanging and the context stays usable.
//
// One CTA of 64 threads.  Warp 0 waits on an mbarrier that no thread arrives at, for
// at most `limit_ns`; warp 1 waits on the same barrier with no time limit of its own
// (the 2 s cap aside) and must leave as soon as warp 0 raises the abort flag.
#include "moda_common.cuh"
#include "sm103_ptx.cuh"

namespace moda {
namespace {

using namespace sm103;

__global__ void __launch_bounds__(64, 1) wait_selftest_kernel(int* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ volatile int abort_flag;
  __shared__ int timed_out, left_on_abort;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // expects one arrival that never comes
    abort_flag = 0;
    timed_out = 0;
    left_on_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    bool ok = mbar_try_wait(&bar, 0);
    const uint64_t t0 = globaltimer();
    while (!ok && globaltimer() - t0 < limit_ns) ok = mbar_try_wait(&bar, 0);
    if (__all_sync(0xffffffffu, !ok) && threadIdx.x == 0) {
      timed_out = 1;
      abort_flag = 1;
    }
  } else {
    // the abort flag, not the 2 s cap, must end this wait
    const uint64_t t0 = globaltimer();
    const bool ok = mbar_wait(&bar, 0, &abort_flag);
    const uint64_t waited = globaltimer() - t0;
    if (__all_sync(0xffffffffu, !ok && waited < kWaitLimitNs) && threadIdx.x == 32) left_on_abort = 1;
  }
  __syncthreads();
  // timeout recorded only when both waits gave up the designed way; anything else is a config error
  if (threadIdx.x == 0) record_status(status, (timed_out && left_on_abort) ? kStatusTimeout : kStatusConfig);
}

}  // namespace

cudaError_t launch_wait_selftest(int* status, uint64_t limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 64, 0, s>>>(status, limit_ns);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moda
