// Self-test of the bounded device waits: a barrier nobody completes must end
// in V4_ERR_TIMEOUT in the status word, with the kernel returning normally.
#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace v4 {

namespace {

__global__ void wait_timeout_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    sm100::mbar_init(&bar, 1);          // one arrival expected, none ever made
    sm100::fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) (void)sm100::mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
  __syncwarp();
}

}  // namespace

}  // namespace v4

using namespace v4;

extern "C" v4_status v4_selftest_wait_timeout(int32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000)
    return set_error(V4_ERR_INVALID_ARG, "limit_us must be in [1, 1000000]");
  int* status = device_status_ptr();
  if (!status) return set_error(V4_ERR_CUDA, "device status word unavailable");
  wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_us * 1000ull, status);
  note_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(V4_ERR_CUDA, cudaGetErrorString(e));
  return V4_OK;
}
