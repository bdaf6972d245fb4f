// Self-test of the bounded waits every kernel of the library uses. One warp
// waits on a shared-memory mbarrier through mbar_wait_bounded, the helper
// behind all of the kernels' pipeline waits, for at most ``limit_ns``. With
// ``arrive`` = 0 nothing arrives: the wait gives up at the limit, records
// KVP_ERR_TIMEOUT in the error word and the kernel returns, leaving the
// context usable. With ``arrive`` = 1 lane 0 arrives first and the wait
// completes at once, recording nothing.
#include "common.cuh"

namespace kvp {
namespace {

__global__ void selftest_wait_kernel(unsigned long long limit_ns, int arrive, int32_t* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
  __syncwarp();
  mbar_wait_bounded(&bar, 0u, &abort_flag, err, limit_ns);
}

}  // namespace
}  // namespace kvp

extern "C" int kvp_selftest_wait(long long limit_ns, int arrive, int32_t* err, void* stream) {
  if (!err || limit_ns <= 0 || limit_ns > 1000000000LL || (arrive != 0 && arrive != 1)) return KVP_ERR_INVALID_ARG;
  kvp::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((unsigned long long)limit_ns, arrive,
                                                                             err);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}
