// Self-test of the failure path that every kernel of this library shares: a
// bounded mbarrier wait that is never satisfied gives up after its limit and
// the kernel records MLA_ERR_TIMEOUT in the caller's error word, leaving the
// CUDA context usable.  Nothing here faults, traps or hangs: the wait ends
// by itself.
#include "internal.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

__global__ void __launch_bounds__(32) lost_wait_kernel(int *err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  // no thread ever arrives, so the barrier's first phase never completes
  if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0)) set_device_error(err, kDevTimeout);
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" __attribute__((visibility("default"))) mla_status mla_selftest_lost_wait(
    void *workspace, mla_stream_t stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MLA_ERR_WORKSPACE;
  lost_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<int *>(workspace));
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
