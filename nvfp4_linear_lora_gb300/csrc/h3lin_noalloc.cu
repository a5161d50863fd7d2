// h3lin_forward_noalloc: the forward projection for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain a workspace: a plugin loaded into a host
// application that owns every device allocation and hands its plugins no
// allocator, or a latency-bound loop whose rules forbid cudaMalloc/cudaFree
// (both can block on the device).  This entry point serves them with scratch
// memory that is part of the library image itself: a fixed-size array in
// device global memory, created when the library's module is loaded into a
// CUDA context and held until that context is destroyed (for the primary
// context: until the process exits or calls cudaDeviceReset).
//
// Rules that follow from one shared, fixed array per context:
//  - Calls needing more than H3LIN_NOALLOC_SCRATCH_BYTES of scratch are
//    rejected with H3LIN_E_WORKSPACE before anything is enqueued.
//  - Every call in a context uses the same array and finds the previous
//    call's contents there.  Each region the kernels read (amax partials,
//    tensor scale, quantised activation, A(x), scaled B) is written earlier in
//    the same call; only the status word carries over (see below).
//  - Calls that may overlap on the GPU (different streams, or different host
//    threads without ordering) race on the array and produce wrong results.
//    Order them on one stream.
//  - The device status word (a timed-out device wait) lives in the array and
//    is sticky: h3lin_noalloc_read_status reads and clears it.
//  - The array's device address belongs to a context, not to a device.  It is
//    looked up (cudaGetSymbolAddress, with that context current) on the first
//    call made with a context current, and looked up again whenever a call
//    finds a context it has not seen (after cudaDeviceReset, or when the host
//    application makes its own driver context current).  Make the first call
//    in each context before any stream capture begins.
#include <mutex>

#include "h3lin_internal.h"

namespace h3lin {
namespace {

static_assert(H3LIN_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");

// The scratch itself.  In host code this name is only a handle for the CUDA
// runtime: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[H3LIN_NOALLOC_SCRATCH_BYTES];

// Driver calls that identify the current context (fetched through the
// runtime's entry-point query: the library does not link libcuda).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct CtxCalls {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const CtxCalls& ctx_calls() {
  static CtxCalls c;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      c.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    else
      cudaGetLastError();
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      c.get_id = reinterpret_cast<CtxGetIdFn>(p);
    else
      cudaGetLastError();
  });
  return c;
}

// Unique id of the current context (ids are never reused, unlike context
// handles); false when no context is current or the driver cannot tell.
bool current_ctx_id(unsigned long long* id) {
  const CtxCalls& c = ctx_calls();
  if (!c.get_current || !c.get_id) return false;
  CUcontext ctx = nullptr;
  if (c.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return c.get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_noalloc_scratch in the current context.  Cached per
// context id; a context not seen before (or no way to identify it) resolves
// the address again.
h3lin_status scratch_address(void** out) {
  constexpr int kSlots = 64;
  static std::mutex mu;
  static unsigned long long ids[kSlots] = {};
  static void* addrs[kSlots] = {};
  static int next = 0;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = 0;
  bool known = current_ctx_id(&id);
  if (known) {
    for (int i = 0; i < kSlots; ++i)
      if (addrs[i] != nullptr && ids[i] == id) {
        *out = addrs[i];
        return H3LIN_OK;
      }
  }
  void* p = nullptr;   // also makes the primary context current when none is
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return H3LIN_E_CUDA;
  }
  if (!known) known = current_ctx_id(&id);
  if (known) {
    ids[next] = id;
    addrs[next] = p;
    next = (next + 1) % kSlots;
  }
  *out = p;
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

extern "C" h3lin_status h3lin_noalloc_read_status(cudaStream_t stream, int32_t* device_status) {
  if (!device_status) return H3LIN_E_INVALID;
  void* scratch = nullptr;
  h3lin_status s = h3lin::scratch_address(&scratch);
  if (s != H3LIN_OK) return s;
  s = h3lin_read_status(scratch, stream, device_status);   // synchronises `stream`
  if (s != H3LIN_OK || *device_status == H3LIN_OK) return s;
  if (cudaMemsetAsync(static_cast<uint8_t*>(scratch) + h3lin::kStatusOffset, 0, sizeof(uint32_t), stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return H3LIN_E_CUDA;
  }
  return H3LIN_OK;
}
