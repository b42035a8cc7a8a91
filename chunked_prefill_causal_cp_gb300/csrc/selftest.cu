// selftest.cu -- a check of the bounded-wait path that every kernel of the
// library uses, on the device it will run on.
//
// One warp waits, through the same warp_wait the attention kernels use, on an
// mbarrier that nothing completes.  The wait gives up after the library's wait
// limit, records CP_DEV_TIMEOUT in the caller's status word and raises the
// CTA's abort flag; a second wait then returns at once because the CTA has
// aborted.  Nothing faults or traps, and the context stays usable.
#include <cstdint>

#include "cp_internal.h"
#include "cp_ptx.cuh"

namespace cp {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(int* status, unsigned long long* out) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  volatile int* abort_p = &abort_flag;
  const uint64_t t0 = global_timer_ns();
  const bool ok1 = warp_wait(&bar, 0, abort_p, status);  // no arrival ever comes
  const uint64_t t1 = global_timer_ns();
  const bool ok2 = warp_wait(&bar, 0, abort_p, status);  // the CTA has aborted: returns at once
  const uint64_t t2 = global_timer_ns();
  if (threadIdx.x == 0) {
    out[0] = ok1 ? 1ull : 0ull;
    out[1] = t1 - t0;
    out[2] = ok2 ? 1ull : 0ull;
    out[3] = t2 - t1;
    out[4] = (unsigned long long)abort_flag;
  }
}

}  // namespace
}  // namespace cp

extern "C" int cp_selftest_bounded_wait(int32_t* dev_status, uint64_t* dev_out, void* stream) {
  if (!dev_status || !dev_out || (reinterpret_cast<uintptr_t>(dev_out) & 7u)) return CP_ERR_INVALID_ARG;
  cp::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      dev_status, reinterpret_cast<unsigned long long*>(dev_out));
  return cudaGetLastError() == cudaSuccess ? CP_OK : CP_ERR_CUDA;
}
