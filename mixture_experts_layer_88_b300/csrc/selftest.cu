// Failure-detection self-test: one thread waits, with the library's bounded
// barrier wait (the one every GEMM role uses), on an mbarrier that nothing
// arrives on.  The wait runs out after the given limit, the kernel records a
// timeout in the device error word and returns normally, so the context
// stays usable and moe_get_status() reports MOE_ERR_DEVICE_TIMEOUT.  Nothing
// here faults, traps or spins without a limit.
#include "common.cuh"
#include "tc.cuh"

namespace moe {
namespace {

__global__ void wait_timeout_kernel(unsigned long long limit_ns, unsigned* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  tc::mbar_init(&bar, 1);
  abort_flag = 0;
  tc::fence_mbar_init();
  const uint64_t deadline = tc::globaltimer_ns() + limit_ns;
  if (!tc::mbar_wait_bounded(&bar, 0, reinterpret_cast<volatile int*>(&abort_flag), deadline))
    atomicOr(status, ERRBIT_TIMEOUT);
}

}  // namespace

moe_status_t launch_wait_timeout_selftest(unsigned long long limit_ns, cudaStream_t stream) {
  unsigned* status = device_status_word();
  if (!status) return MOE_ERR_CUDA;
  TraceScope tr(stream, "selftest_wait_timeout");
  wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  return launch_status();
}

}  // namespace moe
