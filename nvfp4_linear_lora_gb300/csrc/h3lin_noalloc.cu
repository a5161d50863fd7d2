// h3lin_forward_noalloc: the forward projection for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain a workspace: a plugin loaded into a host
// application that owns every device allocation and hands its plugins no
// allocator, or a latency-bound loop whose rules forbid cudaMalloc/cudaFree
// (both can block on the device).  This entry point serves them with scratch
// memory that is part of the library image itself: a fixed-size array in
// device global memory, created when the library's module is loaded on a
// device and held until the process exits.
//
// Rules that follow from one shared, fixed array per device:
//  - Calls needing more than H3LIN_NOALLOC_SCRATCH_BYTES of scratch are
//    rejected with H3LIN_E_WORKSPACE before anything is enqueued.
//  - Every call on a device uses the same array and finds the previous call's
//    contents there.  Nothing has to be cleared: each region the kernels read
//    (amax partials, tensor scale, quantised activation, A(x), scaled B) is
//    written earlier in the same call.
//  - Calls that may overlap on the GPU (different streams, or different host
//    threads without ordering) race on the array and produce wrong results.
//    Order them on one stream.
//  - The device status word lives in the array too and is not readable by
//    the caller; host-side errors are returned as usual.
//  - The first call on each device resolves the array's device address
//    (cudaGetSymbolAddress, with that device current).  Make that first call
//    before any stream capture begins.
#include <mutex>

#include "h3lin_internal.h"

namespace h3lin {
namespace {

static_assert(H3LIN_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");

// The scratch itself.  In host code this name is only a handle for the CUDA
// runtime: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[H3LIN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device, resolved once per device.
h3lin_status scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return H3LIN_E_CUDA;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return H3LIN_E_CUDA;
    }
    addr[dev] = p;
  }
  *out = addr[dev];
  return H3LIN_OK;
}

}  // namespace
}  // namespace h3lin

extern "C" h3lin_status h3lin_forward_noalloc(const void* x, int64_t M, const float* pre_quant_scale,
                                              const h3lin_weight* weight, int32_t epilogue,
                                              const h3lin_adapter* adapter, float strength, void* out,
                                              int32_t out_dtype, cudaStream_t stream) {
  if (!weight) return H3LIN_E_INVALID;
  const bool lora = adapter != nullptr && strength != 0.0f;
  const int32_t rank = lora ? adapter->rank : 0;
  const size_t need = h3lin_forward_workspace_bytes(M, weight->K, weight->N, rank < 0 ? 0 : rank);
  if (need > H3LIN_NOALLOC_SCRATCH_BYTES) return H3LIN_E_WORKSPACE;
  void* scratch = nullptr;
  const h3lin_status s = h3lin::scratch_address(&scratch);
  if (s != H3LIN_OK) return s;
  return h3lin_forward(x, M, pre_quant_scale, weight, epilogue, adapter, strength, out, out_dtype, scratch,
                       H3LIN_NOALLOC_SCRATCH_BYTES, stream);
}
