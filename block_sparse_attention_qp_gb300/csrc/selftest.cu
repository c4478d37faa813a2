// Self-test of the device-side failure detection: a bounded wait that nothing satisfies.
//
// Every producer / consumer hand-off in the kernels waits on an mbarrier through sm100::mbar_wait,
// which gives up after a wall-clock limit, sets MSA_DEVICE_TIMEOUT in the workspace's status word
// and lets the kernel leave its loops.  msa_selftest_wait_timeout takes that path on purpose: one
// thread waits on a barrier that no thread arrives at, for limit_us microseconds, so a caller can
// check that the timeout is reported and that the context is still usable afterwards.
#include <stdio.h>

#include "../../include/msa.h"
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace msa {
namespace {

__global__ void wait_timeout_kernel(unsigned* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar, 1);
    sm100::mbar_fence_init();
    // phase 0 never completes: nothing arrives, so the wait runs into its limit
    sm100::mbar_wait(&bar, 0u, status, limit_ns);
  }
}

}  // namespace
}  // namespace msa

extern "C" {

int msa_selftest_wait_timeout(void* workspace, unsigned limit_us, void* stream) {
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 16 != 0) {
    msa::set_api_error("msa_selftest_wait_timeout: workspace must be non-null and 16-byte aligned");
    return MSA_ERR_INVALID_ARG;
  }
  if (limit_us == 0 || limit_us > 1000000u) {
    msa::set_api_error("msa_selftest_wait_timeout: limit_us must be in 1 .. 1000000");
    return MSA_ERR_INVALID_ARG;
  }
  cudaGetLastError();
  msa::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<unsigned*>(workspace), (unsigned long long)limit_us * 1000ull);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    char msg[160];
    snprintf(msg, sizeof(msg), "msa_selftest_wait_timeout: %s", cudaGetErrorString(e));
    msa::set_api_error(msg);
    return MSA_ERR_CUDA;
  }
  return MSA_OK;
}

}  // extern "C"
