// Diagnostic: the bounded wait every kernel of the library uses, shown to end.
//
// One CTA initialises an mbarrier that nothing ever arrives on and waits for
// its phase with the same helper the kernels use, given a short limit.  The
// wait must give up, raise the CTA's abort flag and set the timeout bit, and
// the kernel must return normally: no hang, no trap, the context stays
// usable.  This is how the library's failure detection is exercised on a
// GPU without faulting it.
#include "../../include/pa.h"
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(128) bounded_wait_selftest_kernel(int32_t* status,
                                                                    unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag, err;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    err = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const unsigned long long t0 = global_timer_ns();
  // phase 0 never completes: nothing arrives
  const bool ok = mbar_wait(&bar, 0, &abort_flag, &err, limit_ns);
  const unsigned long long waited = global_timer_ns() - t0;
  __syncthreads();
  if (threadIdx.x == 0) {
    status[0] = ok ? 1 : 0;
    status[1] = err;
    status[2] = abort_flag;
    status[3] = static_cast<int32_t>(waited / 1000);   // microseconds
  }
}

}  // namespace pa

extern "C" int pa_selftest_bounded_wait(int64_t limit_ns, int32_t* d_status, void* stream) {
  if (!d_status || limit_ns <= 0 || limit_ns > 1000000000) {
    pa::set_error("pa_selftest_bounded_wait: d_status must be device memory and 0 < limit_ns <= 1e9");
    return PA_ERR_INVALID;
  }
  pa::bounded_wait_selftest_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      d_status, static_cast<unsigned long long>(limit_ns));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    pa::set_error(std::string("selftest launch: ") + cudaGetErrorString(e));
    return PA_ERR_CUDA;
  }
  return PA_OK;
}
