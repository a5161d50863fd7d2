// Merged-LoRA weights, the comparison mode of the dynamic path: the LoRA
// update folded into the weight before it is packed (MiniMax-H3 Turbo — one
// file, no Python, "What the conversion did", list "The rest.", item
// "Backbone"):
//
//   W'[n, k] = bf16_rn( W[n, k] + c * (sum_j B[n, j] * A[j, k]) / s[k] ),  c = strength * alpha / rank
//
// s = pre_quant_scale (1 when absent): the base branch multiplies x by s
// before quantising, the LoRA branch sees the original x (TURBO.md,
// h3-blackwell-runtime, "Implementation"), so the folded update is divided by
// s.  The sum runs over j in ascending order with FP32 fused multiply-adds,
// then c * sum / s and the addition are rounded to FP32 and the result once to
// bf16.  A one-off cost per adapter switch (2 N K r
// FLOP), so a plain CUDA-core tile kernel: each CTA owns 64 rows x 128
// columns of W', stages 32-wide slices of B and A in shared memory as FP32,
// and each thread accumulates 8 rows x 4 columns.
#include "h3lin_device.cuh"

namespace h3lin {
namespace {

constexpr int kMergeRows = 64;
constexpr int kMergeCols = 128;
constexpr int kMergeJ = 32;
constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads) k_merge_lora(const __nv_bfloat16* __restrict__ w,
                                                              const __nv_bfloat16* __restrict__ A,
                                                              const __nv_bfloat16* __restrict__ B,
                                                              const float* __restrict__ pqs,
                                                              __nv_bfloat16* w_out, int N, int K, int rank,
                                                              float c) {
  __shared__ float sB[kMergeRows][kMergeJ + 1];
  __shared__ float sA[kMergeJ][kMergeCols];
  const int n0 = blockIdx.y * kMergeRows, k0 = blockIdx.x * kMergeCols;
  const int tx = threadIdx.x & 31;          // 4 columns: k0 + 4 tx ..
  const int ty = threadIdx.x >> 5;          // 8 rows: n0 + 8 ty ..
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[i][q] = 0.0f;

  for (int j0 = 0; j0 < rank; j0 += kMergeJ) {
    // B slice [64 x 32] and A slice [32 x 128], zero outside the matrices
    for (int e = threadIdx.x; e < kMergeRows * kMergeJ; e += kMergeThreads) {
      const int r = e / kMergeJ, j = e % kMergeJ;
      const int n = n0 + r, jj = j0 + j;
      sB[r][j] = (n < N && jj < rank) ? __bfloat162float(B[static_cast<int64_t>(n) * rank + jj]) : 0.0f;
    }
    for (int e = threadIdx.x; e < kMergeJ * kMergeCols; e += kMergeThreads) {
      const int j = e / kMergeCols, col = e % kMergeCols;
      const int jj = j0 + j, k = k0 + col;
      sA[j][col] = (jj < rank && k < K) ? __bfloat162float(A[static_cast<int64_t>(jj) * K + k]) : 0.0f;
    }
    __syncthreads();
    const int jn = min(kMergeJ, rank - j0);
    for (int j = 0; j < jn; ++j) {
      const float4 a = *reinterpret_cast<const float4*>(&sA[j][4 * tx]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float b = sB[8 * ty + i][j];
        acc[i][0] = fmaf(b, a.x, acc[i][0]);
        acc[i][1] = fmaf(b, a.y, acc[i][1]);
        acc[i][2] = fmaf(b, a.z, acc[i][2]);
        acc[i][3] = fmaf(b, a.w, acc[i][3]);
      }
    }
    __syncthreads();
  }

  const int k = k0 + 4 * tx;
  if (k >= K) return;
  float s[4] = {1.0f, 1.0f, 1.0f, 1.0f};
  if (pqs) {
    const float4 v = *reinterpret_cast<const float4*>(pqs + k);
    s[0] = v.x; s[1] = v.y; s[2] = v.z; s[3] = v.w;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int n = n0 + 8 * ty + i;
    if (n >= N) break;
    const int64_t o = static_cast<int64_t>(n) * K + k;
    const uint2 wv = *reinterpret_cast<const uint2*>(w + o);
    const float w0 = bf16lo(wv.x), w1 = bf16hi(wv.x), w2 = bf16lo(wv.y), w3 = bf16hi(wv.y);
    uint2 r;
    r.x = pack_bf16x2(__fadd_rn(w0, __fdiv_rn(__fmul_rn(c, acc[i][0]), s[0])),
                      __fadd_rn(w1, __fdiv_rn(__fmul_rn(c, acc[i][1]), s[1])));
    r.y = pack_bf16x2(__fadd_rn(w2, __fdiv_rn(__fmul_rn(c, acc[i][2]), s[2])),
                      __fadd_rn(w3, __fdiv_rn(__fmul_rn(c, acc[i][3]), s[3])));
    *reinterpret_cast<uint2*>(w_out + o) = r;
  }
}

}  // namespace

cudaError_t launch_merge_lora(const void* w, const void* A, const void* B, const float* pqs, void* w_out, int N,
                              int K, int rank, float c, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((K + kMergeCols - 1) / kMergeCols),
                  static_cast<unsigned>((N + kMergeRows - 1) / kMergeRows));
  trace_launch("k_merge_lora", long(grid.x) * grid.y, 1, kMergeThreads, 0, "N=%d K=%d rank=%d", N, K, rank);
  k_merge_lora<<<grid, kMergeThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(w),
                                                   static_cast<const __nv_bfloat16*>(A),
                                                   static_cast<const __nv_bfloat16*>(B), pqs,
                                                   static_cast<__nv_bfloat16*>(w_out), N, K, rank, c);
  return cudaGetLastError();
}

}  // namespace h3lin
