// Self-test of the device error path. One warp waits on an mbarrier that
// nothing ever arrives on, through the bounded wait every pipeline role of
// this library uses (mbar_wait_warp). The wait gives up after kWaitLimitNs
// and records DEV_TIMEOUT in this unit's error word; the kernel then
// returns, so the context stays usable. fa_last_device_error reads the word
// together with those of the attention and decode kernels.
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_common.h"
#include "fa_ptx.cuh"

namespace fa {

static __device__ uint32_t g_selftest_err;

__global__ void __launch_bounds__(32) wait_limit_selftest_kernel() {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  mbar_wait_warp(&bar, 0, &g_selftest_err);
}

cudaError_t launch_wait_limit_selftest(cudaStream_t stream) {
  wait_limit_selftest_kernel<<<1, 32, 0, stream>>>();
  return cudaGetLastError();
}

cudaError_t read_and_clear_selftest_error(uint32_t* out, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_selftest_err, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbolAsync(g_selftest_err, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice,
                              stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace fa
