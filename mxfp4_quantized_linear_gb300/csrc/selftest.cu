// Self-test of the failure path of the bounded waits: one thread waits on an
// mbarrier that nothing ever arrives on, gives up after the given limit, and
// sets this unit's device flag, which mx_check_device_errors() then reports as
// MX_ERR_TIMEOUT.  No trap, fault or unbounded loop is involved.

#include "mx_common.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

__global__ void bounded_wait_kernel(unsigned long long limit_ns, int* waited_out) {
  __shared__ uint64_t bar;
  mbar_init(&bar, 1);
  fence_mbar_init();
  // nothing arrives: the phase never completes, the wait runs out
  *waited_out = mbar_wait_for(&bar, 0, limit_ns) ? 0 : 1;
}

}  // namespace

unsigned int take_error_flags_selftest() { return take_tu_error_flags(); }

}  // namespace mx

extern "C" int mx_selftest_bounded_wait(int limit_us, int* waited_out, void* stream) {
  using namespace mx;
  if (limit_us < 1 || limit_us > 100000) return set_error(MX_ERR_ARG, "limit_us=%d outside 1..100000", limit_us);
  if (!waited_out) return set_error(MX_ERR_ARG, "NULL pointer");
  bounded_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<unsigned long long>(limit_us) * 1000ull, waited_out);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MX_OK : set_error(MX_ERR_CUDA, "selftest launch: %s", cudaGetErrorString(e));
}
