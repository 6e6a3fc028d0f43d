// selftest.cu -- tps_selftest_wait_timeout: exercises the bounded-wait path
// every pipelined kernel uses, without hanging the GPU.  One thread waits on
// an mbarrier that nothing will ever arrive on; the wait gives up after
// `limit_ns`, records TPS_DEVERR_TIMEOUT in the device error word and the
// kernel returns normally, leaving the context usable.
#include <cuda_runtime.h>

#include "internal.cuh"
#include "ptx.cuh"
#include "tps.h"

namespace tps {

__global__ void wait_timeout_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_for(&bar, 0, &abort_flag, err, limit_ns);  // nobody arrives
  __syncthreads();
}

}  // namespace tps

extern "C" int tps_selftest_wait_timeout(uint64_t limit_ns, void* cuda_stream) {
  if (limit_ns == 0 || limit_ns > tps::kWaitLimitNs) return TPS_ERR_ARG;
  uint32_t* err = tps::device_error_word();
  if (err == nullptr) return TPS_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  tps::wait_timeout_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  tps::note_launch();
  return cudaPeekAtLastError() == cudaSuccess ? TPS_OK : TPS_ERR_CUDA;
}
