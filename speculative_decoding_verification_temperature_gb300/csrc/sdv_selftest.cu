// sdv_selftest.cu -- self-test of the failure path every asynchronous-copy
// wait relies on (no counterpart in the pages): a wait that can never
// complete must give up after its poll limit, report SD_DEV_TIMEOUT through
// the status word and let the kernel return normally.
#include "sdv_host.cuh"
#include "sdv_tma.cuh"

namespace sdv {

// One CTA: thread 0 initialises an mbarrier expecting one arrival that
// nobody makes and no copy targets (nothing is in flight); every thread
// then waits on its first phase through mbar_wait with `polls` as the
// limit.  After the wait the threads meet at a block barrier and thread 0
// records in out[0] how many threads saw the wait give up, and in out[1]
// the marker 1 that the kernel ran to its end.
__global__ void __launch_bounds__(kThreads)
    selftest_wait_kernel(unsigned polls, int32_t *dev_status, int32_t *out) {
  __shared__ uint64_t bar;
  __shared__ int gave_up;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    gave_up = 0;
  }
  __syncthreads();
  const bool ok = mbar_wait(&bar, 0, dev_status, polls);
  if (!ok) atomicAdd(&gave_up, 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    out[0] = gave_up;
    out[1] = 1;
  }
}

}  // namespace sdv

extern "C" sd_status sd_selftest_bounded_wait(int polls, int32_t *dev_status,
                                              int32_t *out, void *stream) {
  using namespace sdv;
  SDV_REQUIRE(polls >= 1 && polls <= (1 << 20), "polls=%d outside [1, 2^20]",
              polls);
  SDV_REQUIRE(out != nullptr, "out is null");
  int sms = 0;
  const sd_status st = check_device(&sms);
  if (st != SD_OK) return st;
  selftest_wait_kernel<<<1, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      (unsigned)polls, dev_status, out);
  SDV_CUDA(cudaGetLastError());
  return SD_OK;
}
