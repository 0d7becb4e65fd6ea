// Diagnostic of the error path that every kernel takes when a bounded device-side wait
// runs out: one thread waits on a shared-memory mbarrier that nothing ever completes,
// for at most `tries` try_wait rounds (each suspends for at most about 1 ms), records
// MOE_ERR_TIMEOUT in the workspace's control block exactly as the kernels do, and
// returns.  Nothing faults or hangs; the context stays usable, which the tests check by
// running the layer on the same stream afterwards.
#include "params.cuh"

namespace sesg {

__global__ void wait_timeout_kernel(Ctrl* ctrl, uint32_t tries) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival completes phase 0; none ever comes
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    bool done = false;
    for (uint32_t i = 0; i < tries && !done; ++i) done = mbar_try_wait(&bar, 0);
    if (!done) set_status(&ctrl->status, MOE_ERR_TIMEOUT);
  }
}

}  // namespace sesg

extern "C" moe_status_t moe_selftest_wait_timeout(void* ws, size_t ws_bytes, uint32_t tries, void* stream) {
  if (!ws || tries < 1 || tries > 4000) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < sizeof(sesg::Ctrl)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (reinterpret_cast<uintptr_t>(ws) % 256) return MOE_ERR_ALIGNMENT;
  sesg::wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(reinterpret_cast<sesg::Ctrl*>(ws), tries);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
