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
  h3lin::trace_launch("k_selftest_timeout", 1, 1, 64, 0, "wait_cycles=%lld", static_cast<long long>(wait_cycles));
  h3lin::k_selftest_timeout<<<1, 64, 0, stream>>>(status, static_cast<long long>(wait_cycles));
  if (cudaGetLastError() != cudaSuccess) return H3LIN_E_CUDA;
  return H3LIN_OK;
}

// The bounds self-test: a store through index 1000 of a 16-byte window (4
// words) that starts at byte 512 of the workspace header; the address lies
// inside the header's amax-partial area (bytes 1024 ...), so even an unchecked
// store would stay inside the workspace.  With the check live it records
// H3LIN_E_BOUNDS and stores nothing.
namespace h3lin {
__global__ void k_selftest_bounds(uint32_t* status, uint32_t* window) {
  const int idx = 1000 / 4 + threadIdx.x;   // word index past the window's 4 words
  if (in_bounds(idx < 4, status)) window[idx] = 0xDEADBEEFu;
}
}  // namespace h3lin

extern "C" int32_t h3lin_bounds_build(void) {
#ifdef H3LIN_BOUNDS
  return 1;
#else
  return 0;
#endif
}

extern "C" h3lin_status h3lin_selftest_bounds(void* ws, size_t ws_bytes, cudaStream_t stream) {
#ifndef H3LIN_BOUNDS
  (void)ws; (void)ws_bytes; (void)stream;
  return H3LIN_E_UNSUPPORTED;
#else
  if (!ws) return H3LIN_E_INVALID;
  if (ws_bytes < h3lin::kHeaderBytes) return H3LIN_E_WORKSPACE;
  uint8_t* w = static_cast<uint8_t*>(ws);
  h3lin::trace_launch("k_selftest_bounds", 1, 1, 1, 0, "window=16 bytes index=250 words");
  h3lin::k_selftest_bounds<<<1, 1, 0, stream>>>(reinterpret_cast<uint32_t*>(w + h3lin::kStatusOffset),
                                                reinterpret_cast<uint32_t*>(w + 512));
  if (cudaGetLastError() != cudaSuccess) return H3LIN_E_CUDA;
  return H3LIN_OK;
#endif
}
