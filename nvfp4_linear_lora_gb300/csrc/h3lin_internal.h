// Internal declarations shared by the host layer and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/h3lin.h"

namespace h3lin {

// Workspace header: [0] status word (u32), [4] tensor scale of the last
// quantised activation (f32), [8] number of amax partials a producer GEMM left
// for this workspace's next quantiser (i32), [kPartialsOffset ...] per-CTA
// amax partials.
constexpr size_t kStatusOffset = 0;
constexpr size_t kTsOffset = 4;
constexpr size_t kProducedOffset = 8;
constexpr size_t kPartialsOffset = 1024;
constexpr int kMaxPartials = 4096;
constexpr size_t kHeaderBytes = kPartialsOffset + kMaxPartials * sizeof(float);  // 17 KB
constexpr size_t kRegionAlign = 1024;

constexpr int kQuantThreads = 256;

// Launch tracing: with the environment variable H3LIN_TRACE set (to anything
// but "0"), every kernel launch is described on one stderr line before it is
// enqueued: kernel and variant, grid, cluster, block, dynamic shared memory,
// problem sizes and launch plan.  Read once per process (h3lin_api.cu).
bool trace_enabled();
void trace_launch(const char* kernel, long grid, int cluster, int block, int smem, const char* fmt, ...);

// Launch plans computed on the host.
struct RowPlan {   // k_amax / k_quant: each thread owns one 16-byte column chunk
  int blocks;      // grid size
  int rows_step;   // rows advanced per loop trip (threads per column chunk)
};
RowPlan plan_rows(int64_t M, int64_t K, int sm_count);

// Kernel launchers (enqueue only; arguments already validated).
// count_out (nullable): block 0 writes the number of partials there.
cudaError_t launch_amax(const void* x, int M, int K, const float* pqs, float* partials, const RowPlan& p,
                        int* count_out, uint32_t* status, cudaStream_t st);
// nparts_dev (nullable): the kernel reads the number of partials there instead
// of taking nparts (partials left by a producer GEMM).
cudaError_t launch_quant(const void* x, int M, int K, const float* pqs, const float* partials, int nparts,
                         const int* nparts_dev, void* codes, void* scales, float* ts_out, const RowPlan& p,
                         // optional: B' = bf16(B * lora_k / (ts * ts_w)), elems % 8 == 0; u (bf16,
                         // written by the amax pass) takes a power of two from B' for tiny tensor scales
                         const void* b_src, void* b_dst, int64_t b_elems, float lora_k, const float* ts_w,
                         void* u, int64_t u_elems, uint32_t* status, int sm_count, cudaStream_t st);
// Rank parts of the LoRA-down passes for M rows (1 at full size) and the
// matching box rows of A's tensor map (h3lin_quant.cu).
int lora_rank_parts(int64_t M, int rank, int sm_count);
int lora_a_box_rows(int rank, int parts);
// amax pass fused with u = A(x) (bf16 [M, rank]); returns grid size in *nparts.
cudaError_t launch_amax_lora(const CUtensorMap& tm_x, const CUtensorMap& tm_a, int M, int K, int rank, int parts,
                             int a_box_rows, const float* pqs, float* partials, void* u, uint32_t* status,
                             int sm_count, int* nparts, cudaStream_t st);
// The same TMA-staged pass with the amax already known (*nparts_dev partials
// from a producer GEMM): quantises x * s to codes + native scales and computes
// u = A(x) in one read of x; writes ts and, like launch_quant, B'.
cudaError_t launch_quant_lora(const CUtensorMap& tm_x, const CUtensorMap& tm_a, int M, int K, int rank, int parts,
                              int a_box_rows, const float* pqs, const float* partials, const int* nparts_dev,
                              void* codes, void* scales, float* ts_out, void* u, uint32_t* status,
                              const void* b_src, void* b_dst, int64_t b_elems, float lora_k, const float* ts_w,
                              int sm_count, cudaStream_t st);
// Q/K RMSNorm + split-half RoPE in the pair GEMM's epilogue (bf16 output of
// a fused QKV projection, head_dim 128, 96 rotated dimensions): the tiles of
// Q and K heads are normalised and rotated before they are stored, exactly as
// k_qk_norm_rope would do in place afterwards; V tiles are stored as usual.
struct RopeEpi {
  const float4* cs;      // the rows' (cos, sin) of the 48 rotation pairs (launch_rope_table's layout)
  const float* q_gain;   // [128]
  const float* k_gain;   // [128]
  int heads;             // Q heads (= K heads); the output is [Q | K | V]
  float eps;
};
constexpr int kRopePairs = 48;   // rotation pairs per head in the fused epilogue

// FP4 GEMM + optional LoRA-up + epilogue.
struct GemmArgs {
  CUtensorMap tm_xq, tm_wq, tm_u, tm_b;
  CUtensorMap tm_xs, tm_ws;   // scale bytes viewed as [bytes / 256, 256] (pair kernel)
  CUtensorMap tm_out;         // output [M, ldo], 32-row x 128-byte boxes (pair kernel)
  CUtensorMap tm_out16;       // output [M, ldo] bf16, 16-row x 16-column boxes, 32-byte swizzle (fused RoPE)
  const uint8_t* xs;
  const uint8_t* ws;
  const float* ts_x;
  const float* ts_w;
  void* out;
  int M, N, K, rank, ldo;
  int group_m;                // M-tiles per raster group (1 = N-fastest)
  uint32_t* status;
  bool lora, silu, f32out;
  bool pair;                  // use the CTA-pair kernel
  // producer epilogue (pair kernel, SiLU*up, bf16 output): amax partials of
  // |h * amax_s| for the consuming projection's quantiser; amax_out null = off
  const float* amax_s;
  float* amax_out;
  int* amax_count;
  // fused Q/K RMSNorm + RoPE (pair kernel, no SiLU, bf16 output); rope.cs null = off
  RopeEpi rope;
};
cudaError_t launch_fp4gemm(const GemmArgs& a, int sm_count, cudaStream_t st);

// M-tiles per raster group of the GEMM for a weight [N, K] and tiles of
// tile_rows rows (h3lin_gemm.cu).
int raster_group(int64_t N, int64_t K, int tile_rows);

// Q/K RMSNorm + split-half three-axis RoPE in place on qkv [M, 3 heads 128]
// (h3lin_rope.cu; arguments validated by h3lin_qk_norm_rope).
cudaError_t launch_qk_norm_rope(void* qkv, int M, int heads, int rot, const int (&axis_dims)[3], float theta,
                                float eps, const float* q_gain, const float* k_gain, const int* pos,
                                uint32_t* status, int sm_count, cudaStream_t st);
// The (cos, sin) table of the fused epilogue: for the 48 rotation pairs of
// every row, the same floats k_qk_norm_rope computes, in blocks of 16 rows:
// cs[(m / 16) * 24 * 16 + j * 16 + m % 16] = (cos, sin) of pairs 2j, 2j + 1
// of row m; ceil(M / 16) * 16 * 384 bytes.
cudaError_t launch_rope_table(float4* cs, int M, const int (&axis_dims)[3], float theta, const int* pos,
                              uint32_t* status, int sm_count, cudaStream_t st);

// Modulation producer (h3lin_modulate.cu): x_mod = bf16(LN(x) (1 + scale) +
// shift) per row's table row, plus amax partials of |x_mod * pqs| and their count.
cudaError_t launch_modulate(const void* x, int M, int K, const float* table, int T, const int* row_table, float eps,
                            void* out, const float* pqs, float* partials, int* count, uint32_t* status, int sm_count,
                            cudaStream_t st);

// W'[N, K] = bf16(W + c * (B[N, r] @ A[r, K]) / s[K]) (h3lin_merge.cu; s may be
// null = 1); in place allowed.
cudaError_t launch_merge_lora(const void* w, const void* A, const void* B, const float* pqs, void* w_out, int N,
                              int K, int rank, float c, cudaStream_t stream);

}  // namespace h3lin
