// selftest.cu -- the timeout path of the library's bounded waits, made to
// run out on purpose without a fault: one thread waits, with the same bounded
// mbarrier wait every kernel of the library uses, on an mbarrier that nothing
// arrives at; when the limit passes it sets the timeout bit of the workspace
// error word and the kernel returns, leaving the context usable.
#include "common.cuh"
#include "tc.cuh"

namespace csa2 {

__global__ void wait_timeout_kernel(uint8_t* ws, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);                  // one arrival expected; none comes
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !tc::mbar_wait_bounded(&bar, 0, limit_ns)) raise_err(ws, CSA2_DEV_TIMEOUT);
}

}  // namespace csa2

extern "C" csa2_status csa2_selftest_wait_timeout(void* ws, size_t ws_bytes, uint32_t limit_us, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 256) return CSA2_ERR_INVALID_ARG;
  if (limit_us < 1 || limit_us > 1000000) return CSA2_ERR_INVALID_ARG;
  csa2::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint8_t*>(ws),
                                                                             uint64_t(limit_us) * 1000);
  return cudaGetLastError() == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA;
}
