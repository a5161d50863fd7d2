// Modulation producer: the input of the QKV and gate/up projections made from
// the residual stream and the AdaLN table, segment-wise (MiniMax-H3 Ultra Fast
// README, "Active optimization stack", row "AdaLN"), emitted as the exact BF16
// LoRA input while the amax for the NVFP4 packing is reduced on the way
// (TURBO.md, h3-blackwell-runtime, "Implementation": modulation producer).
//
//   y     = (x - mean) / sqrt(var + eps)          per row, fp32, two passes
//   x_mod = bf16(fmaf(y, 1 + scale[t], shift[t])), t = row_table[row]
//   partial[cta] = max |fl(x_mod * s_next)| over the CTA's rows
//
// HBM-bound: 2 B read + 2 B written per element.  One row per CTA iteration
// (128 threads, grid-strided, many CTAs per SM): a thread keeps its
// 16-byte chunks c = t + 128 j of the row in registers across the two
// block reductions (mean, then the centred sum of squares); the table row is
// small and re-read through L1.  The amax needs no per-element multiply: a
// thread keeps the column-wise max |x_mod| of its chunks (packed bf16) and
// scales it by |s_next| once at the end, which is exact because rounding is
// monotone: max_r |fl(h_r * s)| = fl(max_r |h_r| * |s|).
#include "h3lin_device.cuh"

namespace h3lin {

constexpr int kModThreads = 128;

namespace {

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < kModThreads / 32; ++i) s += red[i];
  __syncthreads();                    // red is reused by the next reduction
  return s;
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&v)[8]) {
  v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
  v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
}

// CPT = 16-byte chunks per thread, ceil(K / 8 / kModThreads): the row stays in
// registers, sized for the K at hand (more CTAs per SM for smaller K).
template <int CPT>
__global__ void __launch_bounds__(kModThreads) k_modulate(const uint4* __restrict__ x, int M, int K,
                                                          const float* __restrict__ table, int T,
                                                          const int* __restrict__ row_table, float eps,
                                                          uint4* __restrict__ out, const float* __restrict__ pqs,
                                                          float* __restrict__ partials, int* __restrict__ count,
                                                          uint32_t* __restrict__ status) {
  __shared__ float red[kModThreads / 32];
  const int kc = K >> 3;
  const float inv_k = 1.0f / static_cast<float>(K);
  __nv_bfloat162 colmax[CPT][4];
#pragma unroll
  for (int j = 0; j < CPT; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) colmax[j][k] = __float2bfloat162_rn(0.0f);
  for (int row = blockIdx.x; row < M; row += gridDim.x) {
    uint4 w[CPT];
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      const int c = threadIdx.x + kModThreads * j;
      if (c < kc) {
        w[j] = __ldcs(x + int64_t(row) * kc + c);
        float v[8];
        unpack8(w[j], v);
#pragma unroll
        for (int k = 0; k < 8; ++k) s += v[k];
      }
    }
    const float mean = block_sum(s, red) * inv_k;
    float q = 0.0f;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      const int c = threadIdx.x + kModThreads * j;
      if (c < kc) {
        float v[8];
        unpack8(w[j], v);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float d = v[k] - mean;
          q = fmaf(d, d, q);
        }
      }
    }
    const float rstd = rsqrtf(fmaf(block_sum(q, red), inv_k, eps));
    int t = row_table[row];
    const bool bad = t < 0 || t >= T;
    if (bad) {                        // recorded; the row is written as zeros
      if (threadIdx.x == 0) atomicCAS(status, 0u, static_cast<uint32_t>(H3LIN_E_INVALID));
      t = 0;
    }
    const float* shift = table + int64_t(t) * 2 * K;
    const float* scale = shift + K;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      const int c = threadIdx.x + kModThreads * j;
      if (c < kc) {
        float v[8], o[8];
        unpack8(w[j], v);
        const float4 sh0 = __ldg(reinterpret_cast<const float4*>(shift) + 2 * c);
        const float4 sh1 = __ldg(reinterpret_cast<const float4*>(shift) + 2 * c + 1);
        const float4 sc0 = __ldg(reinterpret_cast<const float4*>(scale) + 2 * c);
        const float4 sc1 = __ldg(reinterpret_cast<const float4*>(scale) + 2 * c + 1);
        const float sh[8] = {sh0.x, sh0.y, sh0.z, sh0.w, sh1.x, sh1.y, sh1.z, sh1.w};
        const float sc[8] = {sc0.x, sc0.y, sc0.z, sc0.w, sc1.x, sc1.y, sc1.z, sc1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = bad ? 0.0f : fmaf((v[k] - mean) * rstd, 1.0f + sc[k], sh[k]);
        const uint4 r = make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                                   pack_bf16x2(o[6], o[7]));
        if (in_bounds(row < M && c < kc, status)) out[int64_t(row) * kc + c] = r;
        const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
          colmax[j][k] = __hmax2(colmax[j][k], __habs2(*reinterpret_cast<const __nv_bfloat162*>(&rw[k])));
      }
    }
  }
  // amax of the stored bf16 values times the consumer's per-channel scale
  float am = 0.0f;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + kModThreads * j;
    if (c < kc) {
      float ps[8] = {1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f, 1.0f};
      if (pqs) {
        const float4 p0 = __ldg(reinterpret_cast<const float4*>(pqs) + 2 * c);
        const float4 p1 = __ldg(reinterpret_cast<const float4*>(pqs) + 2 * c + 1);
        ps[0] = p0.x; ps[1] = p0.y; ps[2] = p0.z; ps[3] = p0.w;
        ps[4] = p1.x; ps[5] = p1.y; ps[6] = p1.z; ps[7] = p1.w;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(&colmax[j][k]);
        am = fmaxf(am, __fmul_rn(bf16lo(u), fabsf(ps[2 * k])));
        am = fmaxf(am, __fmul_rn(bf16hi(u), fabsf(ps[2 * k + 1])));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = am;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = red[0];
    for (int i = 1; i < kModThreads / 32; ++i) m = fmaxf(m, red[i]);
    partials[blockIdx.x] = m;
    if (blockIdx.x == 0) *count = static_cast<int>(gridDim.x);
  }
}

template <int CPT>
static cudaError_t launch_cpt(const void* x, int M, int K, const float* table, int T, const int* row_table, float eps,
                              void* out, const float* pqs, float* partials, int* count, uint32_t* status,
                              int sm_count, cudaStream_t st) {
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_modulate<CPT>, kModThreads, 0);
  if (e != cudaSuccess) return e;
  int grid = (per_sm > 0 ? per_sm : 1) * sm_count;
  if (grid > M) grid = M;
  if (grid > kMaxPartials) grid = kMaxPartials;
  trace_launch("k_modulate", grid, 1, kModThreads, 0, "M=%d K=%d chunks_per_thread=%d table_rows=%d", M, K, CPT, T);
  k_modulate<CPT><<<grid, kModThreads, 0, st>>>(static_cast<const uint4*>(x), M, K, table, T, row_table, eps,
                                                static_cast<uint4*>(out), pqs, partials, count, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_modulate(const void* x, int M, int K, const float* table, int T, const int* row_table, float eps,
                            void* out, const float* pqs, float* partials, int* count, uint32_t* status, int sm_count,
                            cudaStream_t st) {
  const int cpt = (K / 8 + kModThreads - 1) / kModThreads;
#define H3LIN_MOD_CASE(n)                                                                                       \
  case n:                                                                                                      \
    return launch_cpt<n>(x, M, K, table, T, row_table, eps, out, pqs, partials, count, status, sm_count, st);
  switch (cpt) {
    H3LIN_MOD_CASE(1)
    H3LIN_MOD_CASE(2)
    H3LIN_MOD_CASE(3)
    H3LIN_MOD_CASE(4)
    H3LIN_MOD_CASE(5)
    H3LIN_MOD_CASE(6)
    H3LIN_MOD_CASE(7)
    H3LIN_MOD_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef H3LIN_MOD_CASE
}

}  // namespace h3lin
