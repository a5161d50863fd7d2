// Q/K RMSNorm + partial split-half three-axis RoPE, in place on the QKV
// projection's bf16 output (MiniMax-H3 Ultra Fast README, "Active
// optimization stack", row "Attention projections"; "Kernel path", item 2).
// The arithmetic is stated in include/h3lin.h next to h3lin_qk_norm_rope.
//
// HBM-bound: every Q and K element is read and written once (4 B per
// element, 40 KB per row at 40 heads); V is not read.  Persistent CTAs (two
// per SM) stream rows through a shared-memory ring: warp 0 prefetches a row's
// Q and K (contiguous, heads * 512 bytes) with one cp.async.bulk and computes
// the row's rot/2 (cos, sin) pairs into the stage; warps 1-8 take the staged
// row, a half-warp per head at a time, a lane holding 8 consecutive
// dimensions: the sum of squares is reduced over the 16 lanes, the split-half
// partner of lane l is lane l +- rot/16, and the result goes straight to
// global memory (16-byte stores), so only the loads need the ring.
#include <cmath>

#include "h3lin_device.cuh"

namespace h3lin {

constexpr int kRopeConsumerWarps = 8;
constexpr int kRopeThreads = 32 * (1 + kRopeConsumerWarps);
constexpr int kRopeMaxPairs = 64;    // rot_dims <= 128
constexpr int kRopeCtaSmem = 113 * 1024;   // two CTAs per SM

struct RopeFreqs {
  float freq[kRopeMaxPairs];         // per pair: theta^(-2 j / axis_dims[a])
  int axis[kRopeMaxPairs];           // per pair: position axis
};

namespace {

// mbarrier tx expectation without an arrive (the arrives come from the lanes
// that wrote the stage's angles)
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__global__ void __launch_bounds__(kRopeThreads, 2) k_qk_norm_rope(__nv_bfloat16* qkv, int M, int heads, int half,
                                                                  float eps, const float* __restrict__ q_gain,
                                                                  const float* __restrict__ k_gain,
                                                                  const int* __restrict__ pos, uint32_t* status,
                                                                  int stages, RopeFreqs f) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int row_bytes = heads * 512;                           // Q and K of one row
  float* ang = reinterpret_cast<float*>(smem + stages * row_bytes);   // [stages][2][64]: cos, sin
  float* gain = ang + stages * 2 * kRopeMaxPairs;              // [2][128]: Q, K
  uint64_t* full = reinterpret_cast<uint64_t*>(gain + 256);
  uint64_t* empty = full + stages;
  int* abort_flag = reinterpret_cast<int*>(empty + stages);
  const Abort ab{abort_flag, status};

  const int warp = warp_id(), lane = lane_id();
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 32);
      mbar_init(&empty[s], kRopeConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x >= 32) {
    const int t = threadIdx.x - 32;   // 0 .. 255
    gain[t] = t < 128 ? q_gain[t] : k_gain[t - 128];
  }
  __syncthreads();
  const int64_t ld = int64_t(3) * heads * 128;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int st = 0;
    uint32_t ph = 0, filled = 0, fill_par = 0;
    for (int row = blockIdx.x; row < M; row += gridDim.x) {
      if (!mbar_wait(&empty[st], ph ^ 1, ab)) break;
      if (lane == 0) {
        mbar_expect_tx(&full[st], static_cast<uint32_t>(row_bytes));
        bulk_load(smem + st * row_bytes, qkv + int64_t(row) * ld, static_cast<uint32_t>(row_bytes), &full[st]);
      }
      filled |= 1u << st;
      fill_par = (fill_par & ~(1u << st)) | (ph << st);
      float* cs = ang + st * 2 * kRopeMaxPairs;
      for (int i = lane; i < half; i += 32) {
        const float a = __fmul_rn(static_cast<float>(pos[3 * int64_t(row) + f.axis[i]]), f.freq[i]);
        float sv, cv;
        sincosf(a, &sv, &cv);
        cs[i] = cv;
        cs[kRopeMaxPairs + i] = sv;
      }
      mbar_arrive(&full[st]);         // each lane: its angles are written
      if (++st == stages) { st = 0; ph ^= 1; }
    }
    // no copy may still be landing in shared memory when the CTA exits
    if (lane == 0)
      for (int s = 0; s < stages; ++s)
        if (filled & (1u << s)) mbar_drain(&full[s], (fill_par >> s) & 1);
  } else {
    // ----------------------------------------------------------- consumers
    const int t = threadIdx.x - 32;
    const int l16 = t & 15;                  // lane within the half-warp
    const int hw = t >> 4;                   // half-warp 0 .. 15
    const int d0 = 8 * l16;                  // first dimension of this lane
    const int shift = half / 8;              // lanes between split-half partners
    const int partner = d0 < half ? l16 + shift : (d0 < 2 * half ? l16 - shift : l16);
    const bool rotated = d0 < 2 * half;
    const int i0 = d0 < half ? d0 : (rotated ? d0 - half : 0);
    const int nhv = 2 * heads;               // Q heads, then K heads
    int st = 0;
    uint32_t ph = 0;
    for (int row = blockIdx.x; row < M; row += gridDim.x) {
      if (!mbar_wait(&full[st], ph, ab)) break;
      // this lane's 8 (cos, sin) pairs serve all its heads of the row; the
      // first half subtracts the partner's sine term, the second adds it
      const float* cs = ang + st * 2 * kRopeMaxPairs;
      float c8[8], s8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        c8[k] = rotated ? cs[i0 + k] : 1.0f;
        const float sv = rotated ? cs[kRopeMaxPairs + i0 + k] : 0.0f;
        s8[k] = d0 < half ? -sv : sv;
      }
      const uint8_t* data = smem + st * row_bytes + 16 * l16;
      __nv_bfloat16* out = qkv + int64_t(row) * ld + d0;
      for (int hv = hw; hv < nhv; hv += 2 * kRopeConsumerWarps) {   // equal trip counts within a warp (nhv even)
        const uint4 w4 = *reinterpret_cast<const uint4*>(data + hv * 256);
        float v[8] = {bf16lo(w4.x), bf16hi(w4.x), bf16lo(w4.y), bf16hi(w4.y),
                      bf16lo(w4.z), bf16hi(w4.z), bf16lo(w4.w), bf16hi(w4.w)};
        float ss = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) ss = fmaf(v[k], v[k], ss);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o, 16);
        const float r = rsqrtf(fmaf(ss, 1.0f / 128.0f, eps));
        const float* g = gain + (hv < heads ? 0 : 128) + d0;
        float y[8], pv[8], o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) y[k] = v[k] * r * g[k];
#pragma unroll
        for (int k = 0; k < 8; ++k) pv[k] = __shfl_sync(0xFFFFFFFFu, y[k], partner, 16);
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = fmaf(pv[k], s8[k], y[k] * c8[k]);
        if (in_bounds(row < M && hv < nhv && d0 + 8 <= 128, status))
          *reinterpret_cast<uint4*>(out + int64_t(hv) * 128) =
              make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                         pack_bf16x2(o[6], o[7]));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (++st == stages) { st = 0; ph ^= 1; }
    }
  }
}

// The rotation angles' (cos, sin) for the QKV GEMM's fused epilogue, with
// k_qk_norm_rope's angle arithmetic (float(pos) x the host-rounded frequency,
// one rounding, then sincosf), so the fused epilogue rotates by exactly the
// same values.  Layout: blocks of 16 rows; in a block, float4 j (pairs 2j and
// 2j + 1: cos, sin, cos, sin) of its 16 rows side by side, so that the 16
// rows an epilogue warp holds read one 256-byte run per float4.
__global__ void __launch_bounds__(256) k_rope_table(float4* __restrict__ cs, int M, const int* __restrict__ pos,
                                                    uint32_t* status, RopeFreqs f) {
  constexpr int kQuads = kRopePairs / 2;
  const int64_t n = (int64_t(M) + 15) / 16 * 16 * kQuads;   // whole 16-row blocks; rows >= M are skipped
  for (int64_t t = int64_t(blockIdx.x) * 256 + threadIdx.x; t < n; t += int64_t(gridDim.x) * 256) {
    const int64_t blk = t / (16 * kQuads);
    const int rem = static_cast<int>(t - blk * (16 * kQuads));
    const int j = rem >> 4;
    const int64_t row = blk * 16 + (rem & 15);
    if (row >= M) continue;
    float c[2], sn[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int i = 2 * j + e;
      const float a = __fmul_rn(static_cast<float>(pos[3 * row + f.axis[i]]), f.freq[i]);
      sincosf(a, &sn[e], &c[e]);
    }
    if (in_bounds(t < n, status)) cs[t] = make_float4(c[0], sn[0], c[1], sn[1]);   // t = blk 384 + j 16 + row % 16
  }
}

// Per pair i of the rot / 2 rotation pairs: theta^(-2 j / axis_dims[a]) (in
// double, rounded once to float) and its position axis a.
RopeFreqs rope_freqs(const int (&axis_dims)[3], float theta) {
  RopeFreqs f{};
  int i = 0;
  for (int a = 0; a < 3; ++a)
    for (int j = 0; j < axis_dims[a] / 2; ++j, ++i) {
      f.freq[i] = static_cast<float>(std::pow(static_cast<double>(theta), -2.0 * j / axis_dims[a]));
      f.axis[i] = a;
    }
  return f;
}

}  // namespace

cudaError_t launch_rope_table(float4* cs, int M, const int (&axis_dims)[3], float theta, const int* pos,
                              uint32_t* status, int sm_count, cudaStream_t st) {
  const RopeFreqs f = rope_freqs(axis_dims, theta);
  const int64_t n = (int64_t(M) + 15) / 16 * 16 * (kRopePairs / 2);   // whole 16-row blocks (rows >= M skipped)
  int64_t grid = (n + 255) / 256;
  if (grid > int64_t(8) * sm_count) grid = int64_t(8) * sm_count;
  if (grid < 1) grid = 1;
  trace_launch("k_rope_table", grid, 1, 256, 0, "M=%d pairs=%d", M, kRopePairs);
  k_rope_table<<<static_cast<unsigned>(grid), 256, 0, st>>>(cs, M, pos, status, f);
  return cudaGetLastError();
}

cudaError_t launch_qk_norm_rope(void* qkv, int M, int heads, int rot, const int (&axis_dims)[3], float theta,
                                float eps, const float* q_gain, const float* k_gain, const int* pos,
                                uint32_t* status, int sm_count, cudaStream_t st) {
  const RopeFreqs f = rope_freqs(axis_dims, theta);
  const int row_bytes = heads * 512;
  const int fixed = 128 + 256 * 4 + 64;                          // alignment, gains, flag
  const int per_stage = row_bytes + 2 * kRopeMaxPairs * 4 + 16;  // data, angles, two barriers
  int budget = kRopeCtaSmem;
  int stages = (budget - fixed) / per_stage;
  if (stages < 2) {                                              // wide rows: one CTA per SM
    budget = 227 * 1024;
    stages = (budget - fixed) / per_stage;
  }
  if (stages > 8) stages = 8;
  if (stages < 2) return cudaErrorInvalidValue;
  const int smem = fixed + stages * per_stage;
  cudaError_t e = cudaFuncSetAttribute(k_qk_norm_rope, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int grid = (budget == kRopeCtaSmem ? 2 : 1) * sm_count;
  if (grid > M) grid = M;
  trace_launch("k_qk_norm_rope", grid, 1, kRopeThreads, smem, "M=%d heads=%d rot=%d", M, heads, rot);
  k_qk_norm_rope<<<grid, kRopeThreads, smem, st>>>(static_cast<__nv_bfloat16*>(qkv), M, heads, rot / 2, eps, q_gain,
                                                   k_gain, pos, status, stages, f);
  return cudaGetLastError();
}

}  // namespace h3lin
