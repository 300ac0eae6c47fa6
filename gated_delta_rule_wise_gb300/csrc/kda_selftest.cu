// kda_selftest.cu -- on-device check of the bounded-wait mechanism.
//
// One warp initialises an mbarrier that expects one arrival, never arrives,
// and waits on it with a poll limit.  The wait gives up, the kernel records
// KDA_ERR_TIMEOUT in the workspace's error word and returns normally: no
// trap, no fault, the context stays usable.
#include "kda_launch.cuh"
#include "kda_ptx.cuh"

namespace kda {
namespace {

__global__ void selftest_wait_kernel(WorkspaceHeader *hdr, unsigned spin_limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!ptx::mbar_wait(&bar, 0, spin_limit)) report_error(hdr, KDA_ERR_TIMEOUT, 0xE001u);
  }
}

}  // namespace

kda_status launch_selftest_wait(WorkspaceHeader *hdr, unsigned spin_limit, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(hdr, spin_limit);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
