// C ABI of the dynamic-LoRA NVFP4 linear: argument validation (on the host,
// before anything is enqueued), workspace layout, TMA tensor maps and the
// kernel sequence.  See include/h3lin.h for the contract of every call.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "h3lin_internal.h"

namespace h3lin {

bool trace_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("H3LIN_TRACE");
    return v != nullptr && v[0] != '\0' && !(v[0] == '0' && v[1] == '\0');
  }();
  return on;
}

void trace_launch(const char* kernel, long grid, int cluster, int block, int smem, const char* fmt, ...) {
  if (!trace_enabled()) return;
  char detail[256];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(detail, sizeof(detail), fmt, ap);
  va_end(ap);
  std::fprintf(stderr, "h3lin: %s grid=%ld cluster=%d block=%d smem=%d %s\n", kernel, grid, cluster, block, smem,
               detail);
}

namespace {

constexpr int64_t kMaxDim = int64_t(1) << 30;   // rows, N
constexpr int64_t kMaxK = int64_t(1) << 17;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- device
struct DeviceInfo {
  int sm_count = 0;
  int major = 0, minor = 0;
};

h3lin_status device_info(DeviceInfo* out) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return H3LIN_E_CUDA;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && have[dev]) {
    *out = cache[dev];
    return H3LIN_OK;
  }
  DeviceInfo d;
  if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return H3LIN_E_CUDA;
  }
  if (dev < 64) {
    cache[dev] = d;
    have[dev] = true;
  }
  *out = d;
  return H3LIN_OK;
}

h3lin_status require_device(DeviceInfo* d) {
  h3lin_status s = device_info(d);
  if (s != H3LIN_OK) return s;
  if (!(d->major == 10 && d->minor == 3)) return H3LIN_E_UNSUPPORTED;  // kernels are built for sm_103a
  return H3LIN_OK;
}

// ----------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// Scale bytes viewed as a 2-D tensor of 256-byte rows; a box of 8 rows is
// four 512-byte scale atoms (one pipeline stage of 128 rows x 256 K).
bool make_sf_map(CUtensorMap* m, const void* base, uint64_t bytes) {
  auto fn = encode_fn();
  if (!fn || bytes % 256 != 0 || bytes < 8 * 256) return false;
  cuuint64_t dims[2] = {256, bytes / 256};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {256, 8};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output [rows, cols] (bf16 or fp32) stored by 32-row x 64-byte boxes,
// 64-byte swizzle (the epilogue's staging layout).
bool make_out_map(CUtensorMap* m, void* base, bool f32, int64_t cols, int64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t esize = f32 ? 4 : 2;
  cuuint64_t dims[2] = {uint64_t(cols), uint64_t(rows)};
  cuuint64_t strides[1] = {uint64_t(cols) * esize};
  cuuint32_t box[2] = {uint32_t(64 / esize), 32};   // 32 rows x 64 bytes: one epilogue warp's staging block
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 output [rows, cols] in boxes of 16 rows x 16 columns (32 bytes) with
// the 32-byte swizzle: the fused RoPE epilogue's stores.
bool make_out16_map(CUtensorMap* m, void* base, int64_t cols, int64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {uint64_t(cols), uint64_t(rows)};
  cuuint64_t strides[1] = {uint64_t(cols) * 2};
  cuuint32_t box[2] = {16, 16};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Row-major 2-D tensor [rows, inner] with a 128-byte-swizzled box.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t rows,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool rank_ok(int64_t r) {
  if (r < 16) return false;
  if (r <= 256) return r % 16 == 0;
  return r <= 512 && r % 32 == 0;
}

struct ForwardLayout {
  size_t codes, scales, u, b, total;
};
ForwardLayout forward_layout(int64_t M, int64_t K, int64_t N, int64_t rank) {
  ForwardLayout L;
  const int64_t mpad = (M + 127) / 128 * 128;
  size_t off = align_up(kHeaderBytes, kRegionAlign);
  L.codes = off;
  off = align_up(off + size_t(M) * size_t(K / 2), kRegionAlign);
  L.scales = off;
  off = align_up(off + size_t(mpad) * size_t(K / 16), kRegionAlign);
  L.u = off;
  off = align_up(off + size_t(M) * size_t(rank) * 2, kRegionAlign);
  L.b = off;
  off = align_up(off + size_t(N) * size_t(rank) * 2, kRegionAlign);
  L.total = off;
  return L;
}

h3lin_status quantize_impl(const void* x, int64_t M, int64_t K, const float* pqs, void* codes, void* scales,
                           float* ts, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (M < 0 || M > kMaxDim || K < 64 || K > kMaxK || K % 64 != 0) return H3LIN_E_SHAPE;
  if (M == 0) return H3LIN_OK;   // no rows: nothing to quantise, no buffer touched
  if (!x || !codes || !scales || !ts || !ws) return H3LIN_E_INVALID;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(ws) || (pqs && !aligned16(pqs)) ||
      (reinterpret_cast<uintptr_t>(ts) & 3u))
    return H3LIN_E_ALIGN;
  if (ws_bytes < kHeaderBytes) return H3LIN_E_WORKSPACE;
  DeviceInfo d;
  h3lin_status s = require_device(&d);
  if (s != H3LIN_OK) return s;
  float* partials = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kPartialsOffset);
  uint32_t* status = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + kStatusOffset);
  const RowPlan plan = plan_rows(M, K, d.sm_count);
  if (launch_amax(x, int(M), int(K), pqs, partials, plan, nullptr, status, stream) != cudaSuccess)
    return H3LIN_E_CUDA;
  if (launch_quant(x, int(M), int(K), pqs, partials, plan.blocks, nullptr, codes, scales, ts, plan, nullptr,
                   nullptr, 0, 0.0f, nullptr, nullptr, 0, status, d.sm_count, stream) != cudaSuccess)
    return H3LIN_E_CUDA;
  return H3LIN_OK;
}

struct ForwardCall {
  const void* x;
  int64_t M, K, N, rank;
  const float* pqs;
  const h3lin_weight* w;
  const h3lin_adapter* adapter;
  float strength;
  bool lora, silu, f32out;
  void* out;
  uint8_t* ws;
  ForwardLayout L;
  DeviceInfo dev;
  bool produced = false;   // prepare: the amax partials were left in ws by a producer GEMM
};

// Where a producer GEMM leaves the amax of its output for the consuming
// projection (h3lin_forward_gemm_produce).
struct Producer {
  const float* pqs;   // the consumer's pre_quant_scale (null = 1)
  uint8_t* ws;        // the consumer's workspace
};

// The parameter rules of h3lin_qk_norm_rope (shared with the fused form).
h3lin_status validate_rope_params(const h3lin_rope_params* p) {
  if (!p) return H3LIN_E_INVALID;
  if (!std::isfinite(p->theta) || !(p->theta > 0.0f) || !std::isfinite(p->eps) || p->eps < 0.0f)
    return H3LIN_E_INVALID;
  if (p->heads < 1 || p->head_dim != 128 || p->rot_dims < 16 || p->rot_dims > p->head_dim ||
      p->rot_dims % 16 != 0 || int64_t(p->heads) * 3 * p->head_dim > kMaxDim)
    return H3LIN_E_SHAPE;
  int64_t sum = 0;
  for (int a = 0; a < 3; ++a) {
    if (p->axis_dims[a] < 0 || p->axis_dims[a] % 2 != 0) return H3LIN_E_SHAPE;
    sum += p->axis_dims[a];
  }
  return sum == p->rot_dims ? H3LIN_OK : H3LIN_E_SHAPE;
}

size_t rope_table_bytes(int64_t M) {
  return align_up(size_t((M + 15) / 16 * 16) * kRopePairs * sizeof(float2), kRegionAlign);
}

// Host-side validation shared by h3lin_forward and its two stages.  `need_x`
// / `need_out` say which side of the call is being checked.
h3lin_status validate_forward(const void* x, int64_t M, const float* pqs, const h3lin_weight* w, int32_t epilogue,
                              const h3lin_adapter* adapter, float strength, void* out, int32_t out_dtype, void* ws,
                              size_t ws_bytes, bool need_x, bool need_out, ForwardCall* c) {
  const bool empty = M == 0;   // no rows: a valid call that touches no buffer and enqueues nothing
  if ((!empty && ((need_x && !x) || (need_out && !out) || !ws)) || !w) return H3LIN_E_INVALID;
  if (!w->codes || !w->scales || !w->tensor_scale) return H3LIN_E_INVALID;
  if (epilogue != H3LIN_EPI_NONE && epilogue != H3LIN_EPI_SILU_MUL) return H3LIN_E_INVALID;
  if (out_dtype != H3LIN_OUT_BF16 && out_dtype != H3LIN_OUT_F32) return H3LIN_E_INVALID;
  if (!std::isfinite(strength)) return H3LIN_E_INVALID;
  const int64_t K = w->K, N = w->N;
  const bool silu = epilogue == H3LIN_EPI_SILU_MUL;
  if (M < 0 || M > kMaxDim || K < 64 || K > kMaxK || K % 64 != 0 || N < 128 || N > kMaxDim || N % 128 != 0)
    return H3LIN_E_SHAPE;
  if (silu && N % 256 != 0) return H3LIN_E_SHAPE;
  if ((!empty && ((need_x && !aligned16(x)) || (need_out && !aligned16(out)) || !aligned16(ws))) ||
      !aligned16(w->codes) || !aligned16(w->scales) || (pqs && !aligned16(pqs)) ||
      (reinterpret_cast<uintptr_t>(w->tensor_scale) & 3u))
    return H3LIN_E_ALIGN;
  const bool lora = adapter != nullptr && strength != 0.0f;
  int64_t rank = 0;
  if (lora) {
    if (!adapter->A || !adapter->B) return H3LIN_E_INVALID;
    if (!std::isfinite(adapter->alpha)) return H3LIN_E_INVALID;
    rank = adapter->rank;
    if (!rank_ok(rank)) return H3LIN_E_SHAPE;
    if (!aligned16(adapter->A) || !aligned16(adapter->B)) return H3LIN_E_ALIGN;
  }
  c->M = M;
  if (empty) return H3LIN_OK;
  c->L = forward_layout(M, K, N, rank);
  if (ws_bytes < c->L.total) return H3LIN_E_WORKSPACE;
  h3lin_status s = require_device(&c->dev);
  if (s != H3LIN_OK) return s;
  c->x = x;
  c->M = M;
  c->K = K;
  c->N = N;
  c->rank = rank;
  c->pqs = pqs;
  c->w = w;
  c->adapter = adapter;
  c->strength = strength;
  c->lora = lora;
  c->silu = silu;
  c->f32out = out_dtype == H3LIN_OUT_F32;
  c->out = out;
  c->ws = static_cast<uint8_t*>(ws);
  return H3LIN_OK;
}

// Every check of h3lin_forward_qk_rope and its GEMM stage (bf16 output, no
// SiLU*up), so that nothing is enqueued on error.
h3lin_status validate_qk_rope(const void* x, int64_t M, const float* pqs, const h3lin_weight* w,
                              const h3lin_adapter* adapter, float strength, const h3lin_rope_params* p,
                              const float* q_gain, const float* k_gain, const int32_t* positions, void* out,
                              void* ws, size_t ws_bytes, bool need_x, ForwardCall* c) {
  h3lin_status s = validate_rope_params(p);
  if (s != H3LIN_OK) return s;
  if (p->rot_dims != 2 * kRopePairs) return H3LIN_E_UNSUPPORTED;
  if (!w) return H3LIN_E_INVALID;
  if (w->N != int64_t(3) * p->heads * p->head_dim) return H3LIN_E_SHAPE;
  if (w->N % 256 != 0) return H3LIN_E_UNSUPPORTED;   // an odd head count: no CTA-pair tiles
  if (M > 0) {
    if (!q_gain || !k_gain || !positions) return H3LIN_E_INVALID;
    if (!aligned16(q_gain) || !aligned16(k_gain) || (reinterpret_cast<uintptr_t>(positions) & 3u))
      return H3LIN_E_ALIGN;
  }
  // the angle table follows h3lin_forward's regions: those must fit in the rest
  const size_t table = M > 0 && M <= kMaxDim ? rope_table_bytes(M) : 0;
  s = validate_forward(x, M, pqs, w, H3LIN_EPI_NONE, adapter, strength, out, H3LIN_OUT_BF16, ws,
                       ws_bytes >= table ? ws_bytes - table : 0, need_x, true, c);
  if (s != H3LIN_OK || c->M == 0) return s;
  return c->dev.sm_count >= 2 ? H3LIN_OK : H3LIN_E_UNSUPPORTED;
}

// amax pass (fused with u = A(x) when the adapter is active) + quantise pass.
// With c.produced the amax pass is skipped: the partials (and their count)
// were left in the workspace header by the producer GEMM of x.
h3lin_status enqueue_prepare(const ForwardCall& c, cudaStream_t stream) {
  uint32_t* status = reinterpret_cast<uint32_t*>(c.ws + kStatusOffset);
  float* ts_x = reinterpret_cast<float*>(c.ws + kTsOffset);
  float* partials = reinterpret_cast<float*>(c.ws + kPartialsOffset);
  const int* produced_count = reinterpret_cast<const int*>(c.ws + kProducedOffset);
  void* xq = c.ws + c.L.codes;
  void* xs = c.ws + c.L.scales;
  void* u = c.ws + c.L.u;
  void* bp = c.ws + c.L.b;
  const RowPlan plan = plan_rows(c.M, c.K, c.dev.sm_count);
  int nparts = plan.blocks;
  const float lora_k = c.lora ? c.strength * (c.adapter->alpha / float(c.rank)) : 0.0f;
  if (c.lora) {
    CUtensorMap tm_x, tm_a;
    const int parts = lora_rank_parts(c.M, int(c.rank), c.dev.sm_count);
    const int a_box = lora_a_box_rows(int(c.rank), parts);
    if (!make_map(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.x, c.K, c.M, c.K * 2, 64, 128)) return H3LIN_E_CUDA;
    if (!make_map(&tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.adapter->A, c.K, c.rank, c.K * 2, 64, a_box))
      return H3LIN_E_CUDA;
    if (c.produced) {   // one pass: quantise + u = A(x) + B'
      if (launch_quant_lora(tm_x, tm_a, int(c.M), int(c.K), int(c.rank), parts, a_box, c.pqs, partials,
                            produced_count, xq, xs, ts_x, u, status, c.adapter->B, bp, c.N * c.rank, lora_k,
                            c.w->tensor_scale, c.dev.sm_count, stream) != cudaSuccess)
        return H3LIN_E_CUDA;
      return H3LIN_OK;
    }
    if (launch_amax_lora(tm_x, tm_a, int(c.M), int(c.K), int(c.rank), parts, a_box, c.pqs, partials, u, status,
                         c.dev.sm_count, &nparts, stream) != cudaSuccess)
      return H3LIN_E_CUDA;
  } else if (!c.produced) {
    if (launch_amax(c.x, int(c.M), int(c.K), c.pqs, partials, plan, nullptr, status, stream) != cudaSuccess)
      return H3LIN_E_CUDA;
  }
  if (launch_quant(c.x, int(c.M), int(c.K), c.pqs, partials, nparts, c.produced ? produced_count : nullptr, xq, xs,
                   ts_x, plan,
                   c.lora ? c.adapter->B : nullptr, c.lora ? bp : nullptr, c.lora ? c.N * c.rank : 0, lora_k,
                   c.w->tensor_scale, c.lora ? u : nullptr, c.lora ? c.M * c.rank : 0, status, c.dev.sm_count,
                   stream) != cudaSuccess)
    return H3LIN_E_CUDA;
  return H3LIN_OK;
}

// FP4 GEMM + LoRA-up + epilogue reading the prepared workspace.  With a
// producer (bf16 output only) the amax of the output for the consuming
// projection is left in the producer's workspace: from the pair kernel's
// SiLU*up epilogue, else by an amax pass over the output.
// The fused Q/K RMSNorm + RoPE epilogue's inputs (h3lin_forward_qk_rope).
struct RopeCall {
  const h3lin_rope_params* p;
  const float* q_gain;
  const float* k_gain;
  const int32_t* positions;
};

h3lin_status enqueue_gemm(const ForwardCall& c, cudaStream_t stream, const Producer* prod = nullptr,
                          const RopeCall* rope = nullptr) {
  GemmArgs g;
  std::memset(&g, 0, sizeof(g));
  void* xq = c.ws + c.L.codes;
  if (!make_map(&g.tm_xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, c.K / 2, c.M, c.K / 2, 128, 128)) return H3LIN_E_CUDA;
  if (!make_map(&g.tm_wq, CU_TENSOR_MAP_DATA_TYPE_UINT8, c.w->codes, c.K / 2, c.N, c.K / 2, 128, 128))
    return H3LIN_E_CUDA;
  if (c.lora) {
    if (!make_map(&g.tm_u, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.ws + c.L.u, c.rank, c.M, c.rank * 2, 64, 128))
      return H3LIN_E_CUDA;
    if (!make_map(&g.tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.ws + c.L.b, c.rank, c.N, c.rank * 2, 64, 128))
      return H3LIN_E_CUDA;
  } else {
    g.tm_u = g.tm_xq;  // unused by the base-only kernels
    g.tm_b = g.tm_wq;
  }
  g.xs = c.ws + c.L.scales;
  g.ws = static_cast<const uint8_t*>(c.w->scales);
  g.ts_x = reinterpret_cast<const float*>(c.ws + kTsOffset);
  g.ts_w = c.w->tensor_scale;
  g.out = c.out;
  g.M = int(c.M);
  g.N = int(c.N);
  g.K = int(c.K);
  g.rank = int(c.rank);
  g.ldo = int(c.silu ? c.N / 2 : c.N);
  g.status = reinterpret_cast<uint32_t*>(c.ws + kStatusOffset);
  g.lora = c.lora;
  g.silu = c.silu;
  g.f32out = c.f32out;
  // CTA-pair kernel for N % 256 == 0 (and SiLU*up, whose N is a multiple of 256)
  g.pair = (c.N % 256 == 0) && c.dev.sm_count >= 2 &&
           make_sf_map(&g.tm_xs, g.xs, size_t((c.M + 127) / 128 * 128) * size_t(c.K / 16)) &&
           make_sf_map(&g.tm_ws, g.ws, size_t(c.N) * size_t(c.K / 16)) &&
           make_out_map(&g.tm_out, c.out, c.f32out, g.ldo, c.M);
  g.group_m = raster_group(c.N, c.K, g.pair ? 256 : 128);
  if (rope) {   // after the (cos, sin) table: the pair kernel's epilogue normalises and rotates Q and K
    if (!g.pair) return H3LIN_E_UNSUPPORTED;
    if (!make_out16_map(&g.tm_out16, c.out, g.ldo, c.M)) return H3LIN_E_CUDA;
    float4* cs = reinterpret_cast<float4*>(c.ws + c.L.total);
    const int axis[3] = {rope->p->axis_dims[0], rope->p->axis_dims[1], rope->p->axis_dims[2]};
    if (launch_rope_table(cs, int(c.M), axis, rope->p->theta, rope->positions, g.status, c.dev.sm_count,
                          stream) != cudaSuccess)
      return H3LIN_E_CUDA;
    g.rope = RopeEpi{cs, rope->q_gain, rope->k_gain, rope->p->heads, rope->p->eps};
  }
  const bool fused_amax = prod && g.pair && c.silu && !c.f32out;
  if (fused_amax) {
    g.amax_s = prod->pqs;
    g.amax_out = reinterpret_cast<float*>(prod->ws + kPartialsOffset);
    g.amax_count = reinterpret_cast<int*>(prod->ws + kProducedOffset);
  }
  if (launch_fp4gemm(g, c.dev.sm_count, stream) != cudaSuccess) return H3LIN_E_CUDA;
  if (prod && !fused_amax) {
    const RowPlan plan = plan_rows(c.M, g.ldo, c.dev.sm_count);
    if (launch_amax(c.out, int(c.M), g.ldo, prod->pqs, reinterpret_cast<float*>(prod->ws + kPartialsOffset), plan,
                    reinterpret_cast<int*>(prod->ws + kProducedOffset),
                    reinterpret_cast<uint32_t*>(prod->ws + kStatusOffset), stream) != cudaSuccess)
      return H3LIN_E_CUDA;
  }
  return H3LIN_OK;
}

}  // namespace
}  // namespace h3lin

using namespace h3lin;

extern "C" {

int32_t h3lin_abi_version(void) { return H3LIN_ABI_VERSION; }

const char* h3lin_status_string(h3lin_status s) {
  switch (s) {
    case H3LIN_OK: return "ok";
    case H3LIN_E_INVALID: return "invalid argument (null pointer, unknown enum or non-finite scalar)";
    case H3LIN_E_SHAPE: return "shape rule violated";
    case H3LIN_E_ALIGN: return "pointer not 16-byte aligned";
    case H3LIN_E_WORKSPACE: return "workspace too small";
    case H3LIN_E_CUDA: return "CUDA error while enqueueing";
    case H3LIN_E_TIMEOUT: return "device-side wait timed out";
    case H3LIN_E_UNSUPPORTED: return "device is not sm_103 (GB300), or the call is not in this build";
    case H3LIN_E_BOUNDS: return "a kernel index left its buffer (bounds build; the access was skipped)";
    default: return "unknown status";
  }
}

size_t h3lin_codes_bytes(int64_t rows, int64_t K) {
  if (rows < 1 || K < 64 || K % 64 != 0) return 0;
  return size_t(rows) * size_t(K / 2);
}

size_t h3lin_scales_bytes(int64_t rows, int64_t K) {
  if (rows < 1 || K < 64 || K % 64 != 0) return 0;
  return size_t((rows + 127) / 128 * 128) * size_t(K / 16);
}

size_t h3lin_quant_workspace_bytes(void) { return kHeaderBytes; }

size_t h3lin_forward_workspace_bytes(int64_t M, int64_t K, int64_t N, int32_t max_rank) {
  if (M < 0 || K < 64 || K % 64 != 0 || N < 1 || max_rank < 0) return 0;
  return forward_layout(M, K, N, max_rank).total;
}

h3lin_status h3lin_forward_workspace_regions(int64_t M, int64_t K, int64_t N, int32_t rank, size_t* offsets) {
  if (!offsets) return H3LIN_E_INVALID;
  if (M < 0 || K < 64 || K % 64 != 0 || N < 1 || rank < 0) return H3LIN_E_SHAPE;
  const ForwardLayout L = forward_layout(M, K, N, rank);
  offsets[0] = L.codes;
  offsets[1] = L.scales;
  offsets[2] = L.u;
  offsets[3] = L.b;
  offsets[4] = kTsOffset;
  offsets[5] = kStatusOffset;
  return H3LIN_OK;
}

h3lin_status h3lin_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!ws) return H3LIN_E_INVALID;
  if (ws_bytes < kHeaderBytes) return H3LIN_E_WORKSPACE;
  if (cudaMemsetAsync(ws, 0, kHeaderBytes, stream) != cudaSuccess) {
    cudaGetLastError();
    return H3LIN_E_CUDA;
  }
  return H3LIN_OK;
}

h3lin_status h3lin_quantize_act(const void* x, int64_t M, int64_t K, const float* pqs, void* codes, void* scales,
                                float* tensor_scale, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return quantize_impl(x, M, K, pqs, codes, scales, tensor_scale, ws, ws_bytes, stream);
}

h3lin_status h3lin_pack_weight(const void* w, int64_t N, int64_t K, void* codes, void* scales, float* tensor_scale,
                               void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (N < 1) return H3LIN_E_SHAPE;   // a weight has rows (an empty activation is a no-op instead)
  return quantize_impl(w, N, K, nullptr, codes, scales, tensor_scale, ws, ws_bytes, stream);
}

h3lin_status h3lin_forward(const void* x, int64_t M, const float* pqs, const h3lin_weight* w, int32_t epilogue,
                           const h3lin_adapter* adapter, float strength, void* out, int32_t out_dtype, void* ws,
                           size_t ws_bytes, cudaStream_t stream) {
  ForwardCall c;
  h3lin_status s = validate_forward(x, M, pqs, w, epilogue, adapter, strength, out, out_dtype, ws, ws_bytes, true,
                                    true, &c);
  if (s != H3LIN_OK || c.M == 0) return s;
  s = enqueue_prepare(c, stream);
  if (s != H3LIN_OK) return s;
  return enqueue_gemm(c, stream);
}

h3lin_status h3lin_forward_prepare(const void* x, int64_t M, const float* pqs, const h3lin_weight* w,
                                   const h3lin_adapter* adapter, float strength, void* ws, size_t ws_bytes,
                                   cudaStream_t stream) {
  ForwardCall c;
  h3lin_status s = validate_forward(x, M, pqs, w, H3LIN_EPI_NONE, adapter, strength, nullptr, H3LIN_OUT_BF16, ws,
                                    ws_bytes, true, false, &c);
  if (s != H3LIN_OK || c.M == 0) return s;
  return enqueue_prepare(c, stream);
}

h3lin_status h3lin_forward_gemm(int64_t M, const h3lin_weight* w, int32_t epilogue, const h3lin_adapter* adapter,
                                float strength, void* out, int32_t out_dtype, void* ws, size_t ws_bytes,
                                cudaStream_t stream) {
  ForwardCall c;
  h3lin_status s = validate_forward(nullptr, M, nullptr, w, epilogue, adapter, strength, out, out_dtype, ws,
                                    ws_bytes, false, true, &c);
  if (s != H3LIN_OK || c.M == 0) return s;
  return enqueue_gemm(c, stream);
}

h3lin_status h3lin_forward_gemm_produce(int64_t M, const h3lin_weight* w, int32_t epilogue,
                                        const h3lin_adapter* adapter, float strength, void* out, void* ws,
                                        size_t ws_bytes, const float* next_pqs, void* next_ws, size_t next_ws_bytes,
                                        cudaStream_t stream) {
  if (M > 0 && !next_ws) return H3LIN_E_INVALID;
  if ((next_ws && !aligned16(next_ws)) || (next_pqs && !aligned16(next_pqs))) return H3LIN_E_ALIGN;
  if (M > 0 && next_ws_bytes < kHeaderBytes) return H3LIN_E_WORKSPACE;
  ForwardCall c;
  h3lin_status s = validate_forward(nullptr, M, nullptr, w, epilogue, adapter, strength, out, H3LIN_OUT_BF16, ws,
                                    ws_bytes, false, true, &c);
  if (s != H3LIN_OK || c.M == 0) return s;
  const Producer p{next_pqs, static_cast<uint8_t*>(next_ws)};
  return enqueue_gemm(c, stream, &p);
}

h3lin_status h3lin_forward_prepare_produced(const void* x, int64_t M, const float* pqs, const h3lin_weight* w,
                                            const h3lin_adapter* adapter, float strength, void* ws, size_t ws_bytes,
                                            cudaStream_t stream) {
  ForwardCall c;
  h3lin_status s = validate_forward(x, M, pqs, w, H3LIN_EPI_NONE, adapter, strength, nullptr, H3LIN_OUT_BF16, ws,
                                    ws_bytes, true, false, &c);
  if (s != H3LIN_OK || c.M == 0) return s;
  c.produced = true;
  return enqueue_prepare(c, stream);
}

size_t h3lin_forward_qk_rope_workspace_bytes(int64_t M, int64_t K, int64_t N, int32_t max_rank) {
  if (M < 0 || K < 64 || K % 64 != 0 || N < 1 || max_rank < 0) return 0;
  return forward_layout(M, K, N, max_rank).total + rope_table_bytes(M);
}

h3lin_status h3lin_forward_gemm_qk_rope(int64_t M, const h3lin_weight* w, const h3lin_adapter* adapter,
                                        float strength, const h3lin_rope_params* p, const float* q_gain,
                                        const float* k_gain, const int32_t* positions, void* out, void* ws,
                                        size_t ws_bytes, cudaStream_t stream) {
  ForwardCall c;
  const h3lin_status s = validate_qk_rope(nullptr, M, nullptr, w, adapter, strength, p, q_gain, k_gain, positions,
                                          out, ws, ws_bytes, false, &c);
  if (s != H3LIN_OK || c.M == 0) return s;
  const RopeCall rc{p, q_gain, k_gain, positions};
  return enqueue_gemm(c, stream, nullptr, &rc);
}

h3lin_status h3lin_forward_qk_rope(const void* x, int64_t M, const float* pqs, const h3lin_weight* w,
                                   const h3lin_adapter* adapter, float strength, const h3lin_rope_params* p,
                                   const float* q_gain, const float* k_gain, const int32_t* positions, void* out,
                                   void* ws, size_t ws_bytes, cudaStream_t stream) {
  ForwardCall c;
  h3lin_status s = validate_qk_rope(x, M, pqs, w, adapter, strength, p, q_gain, k_gain, positions, out, ws, ws_bytes,
                                    true, &c);
  if (s != H3LIN_OK || c.M == 0) return s;
  if ((s = enqueue_prepare(c, stream)) != H3LIN_OK) return s;
  const RopeCall rc{p, q_gain, k_gain, positions};
  return enqueue_gemm(c, stream, nullptr, &rc);
}

size_t h3lin_mlp_workspace_bytes(int64_t M, int64_t K, int64_t N_gate_up, int64_t N_down, int32_t max_rank) {
  if (M < 0 || K < 64 || K % 64 != 0 || N_gate_up < 256 || N_gate_up % 256 != 0 || N_down < 1 || max_rank < 0)
    return 0;
  const size_t a = forward_layout(M, K, N_gate_up, max_rank).total;
  const size_t b = forward_layout(M, N_gate_up / 2, N_down, max_rank).total;
  return a > b ? a : b;
}

h3lin_status h3lin_mlp_forward(const void* x, int64_t M, const float* gu_pqs, const h3lin_weight* gate_up,
                               const h3lin_adapter* gu_adapter, float gu_strength, const float* down_pqs,
                               const h3lin_weight* down, const h3lin_adapter* down_adapter, float down_strength,
                               void* h, void* out, int32_t out_dtype, void* ws, size_t ws_bytes,
                               cudaStream_t stream) {
  if (!gate_up || !down) return H3LIN_E_INVALID;
  if (down->K != gate_up->N / 2) return H3LIN_E_SHAPE;
  ForwardCall a, b;
  h3lin_status s = validate_forward(x, M, gu_pqs, gate_up, H3LIN_EPI_SILU_MUL, gu_adapter, gu_strength, h,
                                    H3LIN_OUT_BF16, ws, ws_bytes, true, true, &a);
  if (s != H3LIN_OK) return s;
  s = validate_forward(h, M, down_pqs, down, H3LIN_EPI_NONE, down_adapter, down_strength, out, out_dtype, ws,
                       ws_bytes, true, true, &b);
  if (s != H3LIN_OK || M == 0) return s;
  // one workspace serves both projections: the down stages run after the
  // gate/up GEMM (stream order), and the producer epilogue writes only the
  // header's partials while that GEMM reads its own regions
  b.produced = true;
  if ((s = enqueue_prepare(a, stream)) != H3LIN_OK) return s;
  const Producer p{down_pqs, static_cast<uint8_t*>(ws)};
  if ((s = enqueue_gemm(a, stream, &p)) != H3LIN_OK) return s;
  if ((s = enqueue_prepare(b, stream)) != H3LIN_OK) return s;
  return enqueue_gemm(b, stream);
}

h3lin_status h3lin_read_status(const void* ws, cudaStream_t stream, int32_t* device_status) {
  if (!ws || !device_status) return H3LIN_E_INVALID;
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return H3LIN_E_CUDA;
  }
  uint32_t v = 0;
  if (cudaMemcpy(&v, static_cast<const uint8_t*>(ws) + kStatusOffset, sizeof(v), cudaMemcpyDeviceToHost) !=
      cudaSuccess) {
    cudaGetLastError();
    return H3LIN_E_CUDA;
  }
  *device_status = static_cast<int32_t>(v);
  return H3LIN_OK;
}

}  // extern "C"

extern "C" h3lin_status h3lin_qk_norm_rope(void* qkv, int64_t M, const h3lin_rope_params* p, const float* q_gain,
                                           const float* k_gain, const int32_t* positions, void* ws,
                                           size_t ws_bytes, cudaStream_t stream) {
  const h3lin_status v = validate_rope_params(p);
  if (v != H3LIN_OK) return v;
  if (M < 0 || M > kMaxDim) return H3LIN_E_SHAPE;
  if (M == 0) return H3LIN_OK;
  if (!qkv || !q_gain || !k_gain || !positions || !ws) return H3LIN_E_INVALID;
  if (!aligned16(qkv) || !aligned16(q_gain) || !aligned16(k_gain) || !aligned16(ws) ||
      (reinterpret_cast<uintptr_t>(positions) & 3u))
    return H3LIN_E_ALIGN;
  if (ws_bytes < kHeaderBytes) return H3LIN_E_WORKSPACE;
  DeviceInfo d;
  const h3lin_status s = require_device(&d);
  if (s != H3LIN_OK) return s;
  const int axis[3] = {p->axis_dims[0], p->axis_dims[1], p->axis_dims[2]};
  if (launch_qk_norm_rope(qkv, int(M), p->heads, p->rot_dims, axis, p->theta, p->eps, q_gain, k_gain, positions,
                          reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + kStatusOffset), d.sm_count,
                          stream) != cudaSuccess)
    return H3LIN_E_CUDA;
  return H3LIN_OK;
}

extern "C" h3lin_status h3lin_modulate_produce(const void* x, int64_t M, int64_t K, const float* table,
                                               int32_t table_rows, const int32_t* row_table, float eps, void* x_mod,
                                               const float* next_pqs, void* next_ws, size_t next_ws_bytes,
                                               cudaStream_t stream) {
  if (M < 0 || M > kMaxDim || K < 64 || K > 8192 || K % 64 != 0 || table_rows < 1) return H3LIN_E_SHAPE;
  if (!std::isfinite(eps) || eps < 0.0f) return H3LIN_E_INVALID;
  if (M == 0) return H3LIN_OK;
  if (!x || !table || !row_table || !x_mod || !next_ws) return H3LIN_E_INVALID;
  if (!aligned16(x) || !aligned16(table) || !aligned16(x_mod) || !aligned16(next_ws) ||
      (next_pqs && !aligned16(next_pqs)) || (reinterpret_cast<uintptr_t>(row_table) & 3u))
    return H3LIN_E_ALIGN;
  if (next_ws_bytes < kHeaderBytes) return H3LIN_E_WORKSPACE;
  DeviceInfo d;
  const h3lin_status s = require_device(&d);
  if (s != H3LIN_OK) return s;
  uint8_t* w = static_cast<uint8_t*>(next_ws);
  if (launch_modulate(x, int(M), int(K), table, table_rows, row_table, eps, x_mod, next_pqs,
                      reinterpret_cast<float*>(w + kPartialsOffset), reinterpret_cast<int*>(w + kProducedOffset),
                      reinterpret_cast<uint32_t*>(w + kStatusOffset), d.sm_count, stream) != cudaSuccess)
    return H3LIN_E_CUDA;
  return H3LIN_OK;
}

extern "C" h3lin_status h3lin_merge_lora(const void* w, int64_t N, int64_t K, const float* pre_quant_scale,
                                         const h3lin_adapter* adapter, float strength, void* w_out,
                                         cudaStream_t stream) {
  if (!w || !w_out || !adapter || !adapter->A || !adapter->B) return H3LIN_E_INVALID;
  if (N < 1 || K < 64 || K % 64 != 0 || N > (int64_t(1) << 30) || K > (int64_t(1) << 30)) return H3LIN_E_SHAPE;
  if (!rank_ok(adapter->rank)) return H3LIN_E_SHAPE;
  if (!std::isfinite(adapter->alpha) || !std::isfinite(strength)) return H3LIN_E_INVALID;
  if ((reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(w_out)) & 7u) return H3LIN_E_ALIGN;
  if (reinterpret_cast<uintptr_t>(pre_quant_scale) & 15u) return H3LIN_E_ALIGN;
  DeviceInfo d;
  const h3lin_status s = require_device(&d);
  if (s != H3LIN_OK) return s;
  const float c = strength * (adapter->alpha / static_cast<float>(adapter->rank));
  if (launch_merge_lora(w, adapter->A, adapter->B, pre_quant_scale, w_out, int(N), int(K), adapter->rank, c,
                        stream) != cudaSuccess)
    return H3LIN_E_CUDA;
  return H3LIN_OK;
}
