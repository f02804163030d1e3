// Self-check of the bounded device waits (failure detection without a fault):
// one warp waits on an mbarrier phase that nothing completes, gives up after
// the wall-clock limit every wait in the library uses, and reports
// OSCAR_STATUS_TIMEOUT in the status word. No copy is in flight, nothing is
// left pending, and the context stays usable (sm_103a).
#include "kernels.cuh"
#include "tma.cuh"

namespace oscar {
namespace {

__global__ void k_wait_probe(int* status) {
  __shared__ __align__(8) uint64_t bar_mem;
  const uint32_t bar = smem_addr(&bar_mem);
  if (threadIdx.x == 0) mbar_init(bar);     // arrival count 1; no thread ever arrives
  __syncwarp();
  const bool landed = __all_sync(0xffffffffu, mbar_wait(bar, 0));
  if (!landed && threadIdx.x == 0) flag(status, OSCAR_STATUS_TIMEOUT);
}

}  // namespace

int launch_wait_probe(int* status, cudaStream_t st) {
  k_wait_probe<<<1, 32, 0, st>>>(status);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_CUDA;
}

}  // namespace oscar
