// Device self-test of the failure path: a bounded mbarrier wait that nothing
// will ever satisfy runs out, records H3LIN_E_TIMEOUT in the workspace status
// word, raises the CTA abort flag (a second waiter with a much longer limit
// gives up as soon as it sees it) and the kernel returns normally.  No trap,
// no fault: the context stays usable.
#include "h3lin_device.cuh"

namespace h3lin {
namespace {

__global__ void k_selftest_timeout(uint32_t* status, long long limit) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Abort ab{&abort_flag, status};
  if (threadIdx.x == 0) {
    mbar_wait(&bars[0], 0, ab, limit);            // no arrival will ever come
  } else if (threadIdx.x == 32) {
    mbar_wait(&bars[1], 0, ab, 64 * limit);       // ends on the abort flag, not its own limit
  }
  __syncthreads();
}

}  // namespace
}  // namespace h3lin

extern "C" h3lin_status h3lin_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int64_t wait_cycles,
                                                    cudaStream_t stream) {
  if (!workspace) return H3LIN_E_INVALID;
  if (workspace_bytes < h3lin::kHeaderBytes) return H3LIN_E_WORKSPACE;
  if (wait_cycles < 1 || wait_cycles > (int64_t(1) << 31)) return H3LIN_E_INVALID;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return H3LIN_E_ALIGN;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return H3LIN_E_CUDA;
  }
  uint32_t* status = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + h3lin::kStatusOffset);
  h3lin::k_selftest_timeout<<<1, 64, 0, stream>>>(status, static_cast<long long>(wait_cycles));
  if (cudaGetLastError() != cudaSuccess) return H3LIN_E_CUDA;
  return H3LIN_OK;
}
