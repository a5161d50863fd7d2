// The NVFP4 base GEMM with the LoRA up-projection accumulated into the same
// TMEM tile, and the fused epilogue.
//
//   acc[m, n]  = sum_k E2M1(xq) E4M3(sx) * E2M1(wq) E4M3(sw)   (FP4 tensor cores)
//   acc[m, n] += sum_j u[m, j] * B'[n, j]                        (BF16 tensor cores)
//   y          = ts_x * ts_w * acc                               (B' carries 1/(ts_x ts_w);
//                                                                  epi_scale for tiny scales)
//   out        = y, or silu(y_gate) * y_up                       (bf16 or fp32, rows >= M masked)
//
// This is `NVFP4_base(x) + strength * (alpha/rank) * B(A(x))` of TURBO.md
// (h3-blackwell-runtime, "Implementation") with the fused gate/up SiLU*up of
// the MiniMax-H3 Ultra Fast README ("Active optimization stack", row MLP).
//
// Two kernels: the CTA-pair kernel (cta_group::2, 256 x 256 tiles; used when
// N is a multiple of 256 or for SiLU*up) and the single-CTA kernel below
// (128 x BN tiles, BN = 128 for the remaining shapes).
//
// Single-CTA kernel: persistent, warp-specialised, one 128 x BN tile per CTA iteration:
//   warp 0      TMA producer (operand tiles, block-scale atoms by bulk copy)
//   warp 1      TMEM owner; lane 0 issues tcgen05.cp of the scales and the MMAs
//   warps 2-9   epilogue: TMEM -> registers, release the accumulator, then
//               scale / SiLU*up / bf16 / store while the next tile runs
// Operand stage: A 128 rows x 256 FP4 (128 B rows, 128-byte swizzle), B BN
// rows, scale atoms 512 B per 128 rows x 64 K.  LoRA stages reuse the ring:
// u tile 128 x 64 bf16 and B' tile BN x 64 bf16.
#include "h3lin_device.cuh"

namespace h3lin {

constexpr int kGemmThreads = 320;

template <int BN>
struct GemmCfg {
  static constexpr int kABytes = 128 * 128;             // 128 rows x 128 B
  static constexpr int kBBytes = BN * 128;
  static constexpr int kSfaBytes = 4 * 512;              // 4 atoms (K = 256)
  static constexpr int kSfbBytes = (BN / 128) * 4 * 512;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kSfCols = 16 + 16 * (BN / 128);   // TMEM columns of one stage's scales
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 256;
  static constexpr int kTmemCols = 512;
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(BN + kStages * kSfCols <= kTmemCols, "TMEM budget");
};

// Tile t -> (tm, tn), rastered in groups of group_m M-tiles: within a group
// the M index moves fastest, so a group's panel of x (group_m tiles) stays in
// L2 while the weight panels stream past it.  group_m = 1 is N-fastest: each
// x panel is read once and the whole weight stays L2-resident (chosen on the
// host when the packed weight is small enough).
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m, int& tm, int& tn) {
  const int per_group = group_m * tiles_n;
  const int g = t / per_group;
  const int r = t - g * per_group;
  const int gm = min(group_m, tiles_m - g * group_m);
  tm = g * group_m + r % gm;
  tn = r / gm;
}

__device__ __forceinline__ float silu(float g) { return g * __frcp_rn(1.0f + __expf(-g)); }

// Store 8 consecutive epilogue values of one row: bf16 (16 bytes) or fp32 (32 bytes).
template <bool F32OUT>
__device__ __forceinline__ void store8(void* out_row, int col, const float (&h)[8]) {
  if (F32OUT) {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(out_row) + col);
    d[0] = make_float4(h[0], h[1], h[2], h[3]);
    d[1] = make_float4(h[4], h[5], h[6], h[7]);
  } else {
    uint4 o;
    o.x = pack_bf16x2(h[0], h[1]);
    o.y = pack_bf16x2(h[2], h[3]);
    o.z = pack_bf16x2(h[4], h[5]);
    o.w = pack_bf16x2(h[6], h[7]);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out_row) + col) = o;
  }
}

template <int BN, bool SILU, bool LORA, bool F32OUT>
__global__ void __launch_bounds__(kGemmThreads, 1) k_fp4gemm(
    const __grid_constant__ CUtensorMap tm_xq, const __grid_constant__ CUtensorMap tm_wq,
    const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_b,
    const uint8_t* __restrict__ xs, const uint8_t* __restrict__ ws, const float* __restrict__ ts_x,
    const float* __restrict__ ts_w, void* __restrict__ out, int M, int N, int K, int rank, int ldo, int group_m,
    uint32_t* __restrict__ status) {
  using C = GemmCfg<BN>;
  static_assert(!SILU || BN == 256, "SiLU*up pairs 128 gate and 128 up columns");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tmem_full = empty + C::kStages;
  uint64_t* tmem_empty = tmem_full + 1;
  uint64_t* drain_bar = tmem_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = warp_id(), lane = lane_id();
  constexpr int kEpiWarps = 8;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, kEpiWarps);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_xq);
    tma_prefetch_desc(&tm_wq);
    if (LORA) {
      tma_prefetch_desc(&tm_u);
      tma_prefetch_desc(&tm_b);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag, status};

  const int tiles_m = (M + 127) >> 7;
  const int tiles_n = SILU ? (N / 2) / 128 : N / BN;
  const int num_tiles = tiles_m * tiles_n;
  const int nk = (K + 255) >> 8;           // FP4 K chunks of 256
  const int nr = LORA ? (rank + 63) >> 6 : 0;  // LoRA chunks of 64
  const int k_atoms = K >> 6;              // scale atoms per 128-row block

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t filled = 0, fill_par = 0;
      int st = 0;
      uint32_t ph = 0;
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        int tm, tn;
        tile_coords(t, tiles_m, tiles_n, group_m, tm, tn);
        const int m0 = tm * 128;
        int brow[2];
        if (SILU) {
          brow[0] = tn * 128;
          brow[1] = N / 2 + tn * 128;
        } else {
          brow[0] = tn * BN;
          brow[1] = tn * BN + 128;
        }
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait(&empty[st], ph ^ 1, ab)) goto producer_done;
          const int nsub = min(4, (K - kc * 256) >> 6);
          uint8_t* base = smem + st * C::kStageBytes;
          const uint32_t tx = C::kABytes + C::kBBytes + nsub * 512 * (1 + BN / 128);
          mbar_arrive_expect_tx(&full[st], tx);
          tma_load_2d(base, &tm_xq, &full[st], kc * 128, m0);
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            tma_load_2d(base + C::kABytes + h * 16384, &tm_wq, &full[st], kc * 128, brow[h]);
          bulk_load(base + C::kABytes + C::kBBytes,
                    xs + (static_cast<int64_t>(tm) * k_atoms + kc * 4) * 512, nsub * 512, &full[st]);
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            bulk_load(base + C::kABytes + C::kBBytes + C::kSfaBytes + h * 2048,
                      ws + (static_cast<int64_t>(brow[h] >> 7) * k_atoms + kc * 4) * 512, nsub * 512, &full[st]);
          filled |= 1u << st;
          fill_par = (fill_par & ~(1u << st)) | (ph << st);
          if (++st == C::kStages) { st = 0; ph ^= 1; }
        }
        for (int rc = 0; rc < nr; ++rc) {
          if (!mbar_wait(&empty[st], ph ^ 1, ab)) goto producer_done;
          uint8_t* base = smem + st * C::kStageBytes;
          mbar_arrive_expect_tx(&full[st], 16384u + BN * 128u);
          tma_load_2d(base, &tm_u, &full[st], rc * 64, m0);
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            tma_load_2d(base + C::kABytes + h * 16384, &tm_b, &full[st], rc * 64, brow[h]);
          filled |= 1u << st;
          fill_par = (fill_par & ~(1u << st)) | (ph << st);
          if (++st == C::kStages) { st = 0; ph ^= 1; }
        }
      }
    producer_done:
      for (int s = 0; s < C::kStages; ++s)
        if (filled & (1u << s)) mbar_drain(&full[s], (fill_par >> s) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0, acc_ph = 0;
      const uint32_t idesc_f4 = idesc_nvfp4(BN);
      const uint32_t idesc_bf = idesc_bf16(BN);
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        if (!mbar_wait(tmem_empty, acc_ph ^ 1, ab)) goto mma_done;
        tc_fence_after();
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait(&full[st], ph, ab)) goto mma_done;
          tc_fence_after();
          const int nsub = min(4, (K - kc * 256) >> 6);
          const uint32_t a_addr = smem_u32(smem + st * C::kStageBytes);
          const uint32_t b_addr = a_addr + C::kABytes;
          const uint32_t sfa_addr = b_addr + C::kBBytes;
          const uint32_t sfb_addr = sfa_addr + C::kSfaBytes;
          const uint32_t sf_col = tmem + BN + st * C::kSfCols;
          for (int j = 0; j < nsub; ++j) {
            tmem_cp_sf_atom(sf_col + 4 * j, sdesc_sf_atom(sfa_addr + j * 512));
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tmem_cp_sf_atom(sf_col + 16 + (BN / 128) * 4 * j + 4 * h, sdesc_sf_atom(sfb_addr + h * 2048 + j * 512));
          }
          for (int j = 0; j < nsub; ++j) {
            mma_nvfp4(tmem, sdesc_kmajor_sw128(a_addr + j * 32), sdesc_kmajor_sw128(b_addr + j * 32), idesc_f4,
                      sf_col + 4 * j, sf_col + 16 + (BN / 128) * 4 * j, (kc | j) != 0);
          }
          tc_commit(&empty[st]);
          if (++st == C::kStages) { st = 0; ph ^= 1; }
        }
        for (int rc = 0; rc < nr; ++rc) {
          if (!mbar_wait(&full[st], ph, ab)) goto mma_done;
          tc_fence_after();
          const int nk16 = min(4, (rank - rc * 64) >> 4);
          const uint32_t a_addr = smem_u32(smem + st * C::kStageBytes);
          const uint32_t b_addr = a_addr + C::kABytes;
          for (int j = 0; j < nk16; ++j)
            mma_bf16(tmem, sdesc_kmajor_sw128(a_addr + j * 32), sdesc_kmajor_sw128(b_addr + j * 32), idesc_bf, 1u);
          tc_commit(&empty[st]);
          if (++st == C::kStages) { st = 0; ph ^= 1; }
        }
        tc_commit(tmem_full);
        acc_ph ^= 1;
      }
    mma_done:
      tc_commit(drain_bar);
      mbar_drain(drain_bar, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;     // which half of the tile's columns
    const EpiScale es = epi_scale(*ts_x, *ts_w);
    const float scale = es.a, post = es.b;
    const bool two = post != 1.0f;   // tiny tensor scales only
    uint32_t acc_ph = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      int tm, tn;
      tile_coords(t, tiles_m, tiles_n, group_m, tm, tn);
      if (!mbar_wait(tmem_full, acc_ph, ab)) break;
      tc_fence_after();
      const int row = tm * 128 + 32 * q + lane;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16);
      constexpr int kChunks = SILU ? 4 : BN / 64;   // x32 column loads per thread
      uint32_t v[kChunks][32];
      if (SILU) {
        tmem_ld32(taddr + half * 64, v[0]);
        tmem_ld32(taddr + half * 64 + 32, v[1]);
        tmem_ld32(taddr + 128 + half * 64, v[2]);
        tmem_ld32(taddr + 128 + half * 64 + 32, v[3]);
      } else {
#pragma unroll
        for (int i = 0; i < kChunks; ++i) tmem_ld32(taddr + half * (BN / 2) + 32 * i, v[i]);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty);
      acc_ph ^= 1;
      if (row < M) {
        void* out_row = static_cast<uint8_t*>(out) + static_cast<int64_t>(row) * ldo * (F32OUT ? 4 : 2);
        if (SILU) {
          const int col0 = tn * 128 + half * 64;
#pragma unroll
          for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              float hv[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                float g = __fmul_rn(scale, __uint_as_float(v[i][8 * w + e]));
                float u = __fmul_rn(scale, __uint_as_float(v[2 + i][8 * w + e]));
                if (two) {
                  g = __fmul_rn(g, post);
                  u = __fmul_rn(u, post);
                }
                hv[e] = __fmul_rn(silu(g), u);
              }
              if (in_bounds(col0 + 32 * i + 8 * w + 8 <= ldo, status)) store8<F32OUT>(out_row, col0 + 32 * i + 8 * w, hv);
            }
          }
        } else {
          const int col0 = tn * BN + half * (BN / 2);
#pragma unroll
          for (int i = 0; i < kChunks; ++i) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              float hv[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                hv[e] = __fmul_rn(scale, __uint_as_float(v[i][8 * w + e]));
                if (two) hv[e] = __fmul_rn(hv[e], post);
              }
              if (in_bounds(col0 + 32 * i + 8 * w + 8 <= ldo, status)) store8<F32OUT>(out_row, col0 + 32 * i + 8 * w, hv);
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BN, bool SILU, bool LORA, bool F32OUT>
static cudaError_t launch_variant(const GemmArgs& a, int sm_count, cudaStream_t st) {
  using C = GemmCfg<BN>;
  auto kern = k_fp4gemm<BN, SILU, LORA, F32OUT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  const int tiles_m = (a.M + 127) / 128;
  const int tiles_n = SILU ? (a.N / 2) / 128 : a.N / BN;
  const int tiles = tiles_m * tiles_n;
  const int grid = tiles < sm_count ? tiles : sm_count;
  trace_launch("k_fp4gemm", grid, 1, kGemmThreads, C::kSmem, "BN=%d silu=%d lora=%d f32out=%d M=%d N=%d K=%d rank=%d "
               "tiles=%d raster_group=%d", BN, int(SILU), int(LORA), int(F32OUT), a.M, a.N, a.K, a.rank, tiles,
               a.group_m);
  kern<<<grid, kGemmThreads, C::kSmem, st>>>(a.tm_xq, a.tm_wq, a.tm_u, a.tm_b, a.xs, a.ws, a.ts_x, a.ts_w,
                                             a.out, a.M, a.N, a.K, a.rank, a.ldo, a.group_m,
                                             a.status);
  return cudaGetLastError();
}


// ============================================================ CTA-pair kernel
// Pair tile 256 x 256: the two CTAs of a cluster each own 128 output rows and
// issue one tcgen05 MMA of M = 256 together (cta_group::2).  Each CTA loads its
// own 128 rows of A, 128 of the 256 B rows, the scale atoms of its A rows and
// of all 256 B rows; every TMA load of both CTAs is counted on the leader's
// barrier.
//   warp 0        producer
//   warp 1        (leader) MMA issuer
//   warps 2-7     (leader) scale atoms -> TMEM, two tcgen05.cp each per
//                 stage: a copy costs its issuing thread a long issue slot, so
//                 six issuing warps keep the twelve copies of a stage off the
//                 critical path (they overlap the previous stage's MMAs)
//   warps 8-23    epilogue, four per TMEM lane quarter: each warp reads its 32
//                 rows x 64 accumulator columns (SiLU*up: 32 gate + 32 up) with
//                 one wait and releases the accumulator at once (the next
//                 tile's MMAs wait for the slowest warp), then scales /
//                 applies SiLU*up / converts and stores through a 32 x 64-byte
//                 staging block per warp with TMA bulk-tensor stores
template <bool SILU> struct PairRoles {
  static constexpr int kCpWarps = 6;
  static constexpr int kEpiWarp0 = 2 + kCpWarps;
  static constexpr int kThreads = 32 * (kEpiWarp0 + 16);
};
struct PairCfg {
  static constexpr int kABytes = 128 * 128;
  static constexpr int kBBytes = 128 * 128;
  static constexpr int kSfaBytes = 4 * 512;
  static constexpr int kSfbBytes = 2 * 4 * 512;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;   // 38 KB
  static constexpr int kStages = 5;
  static constexpr int kSfCols = 16 + 32;
  static constexpr int kEpiWarps = 16;
  static constexpr int kEpiScratch = 2048;                                          // 32 rows x 64 bytes
  static constexpr int kRopeGainBytes = 1024;                                      // fused RoPE: Q, K gains
  static constexpr int kSmem = kStages * kStageBytes + kEpiWarps * kEpiScratch + 1024 + 512;
  static constexpr int kSmemRope = kSmem + kRopeGainBytes;
  static constexpr int kTmemCols = 512;
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert(256 + kStages * kSfCols <= kTmemCols, "TMEM budget");
  static_assert(kSmemRope <= 232448, "shared memory budget");
};

// silu(g) * u with g = scale * acc_gate, u = scale * acc_up (fast exp and divide;
// for very negative g the quotient underflows to 0, the limit of g / (1 + e^-g)).
// TWO: each of g and u is then multiplied by post (epi_scale's second factor).
template <bool TWO>
__device__ __forceinline__ float silu_mul_fast(float scale, float post, uint32_t acc_g, uint32_t acc_u) {
  float g = __fmul_rn(scale, __uint_as_float(acc_g));
  float u = __fmul_rn(scale, __uint_as_float(acc_u));
  if (TWO) {
    g = __fmul_rn(g, post);
    u = __fmul_rn(u, post);
  }
  return __fmul_rn(__fdividef(g, 1.0f + __expf(-g)), u);
}
// The same for two adjacent columns, the multiplies paired (identical results;
// the epilogue's instruction count shows up in the MMA issue rate).
template <bool TWO>
__device__ __forceinline__ uint32_t silu_mul2_bf16(float scale, float post, uint32_t g0, uint32_t g1, uint32_t u0,
                                                   uint32_t u1) {
  float ga, gb, ua, ub, oa, ob;
  fmul2_rn(__uint_as_float(g0), __uint_as_float(g1), scale, scale, ga, gb);
  fmul2_rn(__uint_as_float(u0), __uint_as_float(u1), scale, scale, ua, ub);
  if (TWO) {
    fmul2_rn(ga, gb, post, post, ga, gb);
    fmul2_rn(ua, ub, post, post, ua, ub);
  }
  fmul2_rn(__fdividef(ga, 1.0f + __expf(-ga)), __fdividef(gb, 1.0f + __expf(-gb)), ua, ub, oa, ob);
  return pack_bf16x2(oa, ob);
}

// One staging row's worth (16 words) of a pair-epilogue warp's output from its
// accumulator columns a (0..31) and b (32..63, or the up half for SiLU*up).
template <bool SILU, bool F32OUT, bool TWO>
__device__ __forceinline__ void epi_convert(float scale, float post, const uint32_t (&a)[32], const uint32_t (&b)[32],
                                            int rd, uint32_t (&w)[16]) {
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    if (F32OUT) {
      const int c = rd * 16 + k;   // output column of this warp
      if (SILU) {
        w[k] = __float_as_uint(silu_mul_fast<TWO>(scale, post, a[c], b[c]));
      } else {
        float y = __fmul_rn(scale, __uint_as_float(c < 32 ? a[c] : b[c - 32]));
        if (TWO) y = __fmul_rn(y, post);
        w[k] = __float_as_uint(y);
      }
    } else if (SILU) {
      w[k] = silu_mul2_bf16<TWO>(scale, post, a[2 * k], a[2 * k + 1], b[2 * k], b[2 * k + 1]);
    } else {
      const int c = rd * 32 + 2 * k;
      const uint32_t lo = c < 32 ? a[c] : b[c - 32], hi = c < 32 ? a[c + 1] : b[c - 31];
      float ylo, yhi;
      fmul2_rn(__uint_as_float(lo), __uint_as_float(hi), scale, scale, ylo, yhi);
      if (TWO) fmul2_rn(ylo, yhi, post, post, ylo, yhi);
      w[k] = pack_bf16x2(ylo, yhi);
    }
  }
}

// The warp's staging block (32 rows x 64 bytes, 16-byte chunks placed as the
// 64-byte TMA swizzle lays them out) -> global through the TMA engine; rows
// >= M are clipped by the tensor map.
__device__ __forceinline__ void epi_store(const CUtensorMap* tm_out, const uint8_t* scratch, int col, int row0,
                                          int lane) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tm_out, scratch, col, row0);
    bulk_commit_group();
  }
}
// Before rewriting the scratch: the previous TMA store has finished reading it.
__device__ __forceinline__ void epi_scratch_ready(int lane) {
  if (lane == 0) bulk_wait_group_read0();
  __syncwarp();
}

// Fused Q/K RMSNorm + split-half RoPE: one warp's part of a Q or K tile, one
// head (the 128 accumulator columns at tq's column) x 16 rows (the 16 TMEM
// lanes at tq's lane), bf16 output.  With the 16-lane x 2 TMEM load shape lane l holds row
// l % 16 and, by half h = l / 16, 64 of the head's dimensions in three runs
// ("slots"):
//   slots  0..31   h = 0: dims 16..47    h = 1: dims 64..95
//   slots 32..47   h = 0: dims  0..15    h = 1: dims 96..111
//   slots 48..63   h = 0: dims 48..63    h = 1: dims 112..127
// The rotation partner (d +- 48) of slot s < 32 is slot s of lane l ^ 16; on
// h = 0 slots 32 + k and 48 + k are each other's partners; h = 1's slots from
// 32 on are not rotated.  Every value is the float k_qk_norm_rope computes
// from the stored bf16 output: the same bf16 rounding of the scaled
// accumulator, the sum of squares as the same tree (8-dimension fma chains,
// then chunks 8, 4, 2 and 1 apart; the other half's chunks one shuffle away),
// the same normalisation and rotation expressions.  Stores: slots 0..31 go
// straight to global memory (16 bytes a lane), slots 32..63 through the
// warp's staging block as four 16-row x 16-column TMA boxes (tm16).
__device__ __forceinline__ void rope_head_epilogue(uint32_t tq, uint32_t leader_tmem_empty, float scale, float post,
                                                   const float* gain, const float4* __restrict__ cs, int row, int M,
                                                   __nv_bfloat16* __restrict__ out, int col0, int ldo, float eps,
                                                   int lane, uint32_t* status, uint8_t* scratch,
                                                   const CUtensorMap* tm16, int row0) {
  const int h = lane >> 4;
  epi_scratch_ready(lane);   // a V tile's TMA store may still be reading the staging block
  uint32_t v[32];   // the bf16 output values, slot order, two per word
  float sm[8];      // sums of squares of the 8-dimension slot chunks
  {
    uint32_t a[32], b[16], c[16];
    tmem_ld16x2_x32<48>(tq + 16, a);   // slots 0..31
    tmem_ld16x2_x16<96>(tq + 0, b);    // slots 32..47
    tmem_ld16x2_x16<64>(tq + 48, c);   // slots 48..63
    tmem_ld_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(leader_tmem_empty);
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const uint32_t lo = k < 16 ? a[2 * k] : (k < 24 ? b[2 * k - 32] : c[2 * k - 48]);
      const uint32_t hi = k < 16 ? a[2 * k + 1] : (k < 24 ? b[2 * k - 31] : c[2 * k - 47]);
      float ylo, yhi;
      fmul2_rn(__uint_as_float(lo), __uint_as_float(hi), scale, scale, ylo, yhi);
      fmul2_rn(ylo, yhi, post, post, ylo, yhi);   // post = 1 but for tiny tensor scales: exact then
      v[k] = pack_bf16x2(ylo, yhi);
      float ss = (k & 3) ? sm[k >> 2] : 0.0f;
      ss = fmaf(bf16lo(v[k]), bf16lo(v[k]), ss);
      sm[k >> 2] = fmaf(bf16hi(v[k]), bf16hi(v[k]), ss);
    }
  }
  // the sum of squares over the head: the tree over its 16 chunks in
  // dimension order (h = 0 holds chunks 0..7 in slot-chunk order 2 3 4 5 0 1
  // 6 7, h = 1 chunks 8..15 in order), each add's operands the same floats
  constexpr int kChunkOfSlot0[8] = {4, 5, 0, 1, 2, 3, 6, 7};   // h = 0: slot chunk holding dimension chunk j
  float t1[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float g = h ? sm[j] : sm[kChunkOfSlot0[j]];
    t1[j] = g + __shfl_xor_sync(0xFFFFFFFFu, g, 16);
  }
  const float ss = ((t1[0] + t1[4]) + (t1[2] + t1[6])) + ((t1[1] + t1[5]) + (t1[3] + t1[7]));
  const float r = rsqrtf(fmaf(ss, 1.0f / 128.0f, eps));

  // slots 32..63 wait in the warp's staging block (free in this path) while
  // slots 0..31 are rotated: 16 registers fewer in flight
  {
    uint4* st4 = reinterpret_cast<uint4*>(scratch) + lane * 4;
#pragma unroll
    for (int c = 0; c < 4; ++c)
      st4[c ^ ((lane >> 1) & 3)] = make_uint4(v[16 + 4 * c], v[17 + 4 * c], v[18 + 4 * c], v[19 + 4 * c]);
  }
  const bool live = row < M;
  const int trow = live ? row : M - 1;   // the warp's 16 rows read one 256-byte run per float4
  const float4* csr = cs + int64_t(trow >> 4) * (16 * kRopePairs / 2) + (trow & 15);
  const float2* g2 = reinterpret_cast<const float2*>(gain);
  __nv_bfloat16* orow = out + int64_t(live ? row : 0) * ldo + col0;
  // slots 0..31: rotation with the other half's slot (angles 16..47); h = 0
  // subtracts the partner's sine term, h = 1 adds it
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int d = h ? 64 + 8 * m : 16 + 8 * m;
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 t = __ldg(csr + 16 * (8 + 4 * m + k));   // (cos, sin) of angles 16 + 8m + 2k, + 1
      const float2 g = g2[(d >> 1) + k];
      const uint32_t w = v[4 * m + k];
      const float y0 = bf16lo(w) * r * g.x, y1 = bf16hi(w) * r * g.y;
      const float p0 = __shfl_xor_sync(0xFFFFFFFFu, y0, 16), p1 = __shfl_xor_sync(0xFFFFFFFFu, y1, 16);
      o[k] = pack_bf16x2(fmaf(p0, h ? t.y : -t.y, y0 * t.x), fmaf(p1, h ? t.w : -t.w, y1 * t.z));
    }
    if (live && in_bounds(col0 + d + 8 <= ldo, status))
      *reinterpret_cast<uint4*>(orow + d) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  {
    const uint4* st4 = reinterpret_cast<const uint4*>(scratch) + lane * 4;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 w4 = st4[c ^ ((lane >> 1) & 3)];
      v[16 + 4 * c] = w4.x;
      v[17 + 4 * c] = w4.y;
      v[18 + 4 * c] = w4.z;
      v[19 + 4 * c] = w4.w;
    }
  }
  __syncwarp();   // every lane has its slots back before the block holds outputs
  // slots 32..63: h = 0 rotates dims j and j + 48 (angles 0..15) with each
  // other; h = 1's dims 96..127 keep y (cos 1, sin +0, partner itself)
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const int da = h ? 96 + 8 * m : 8 * m, db = h ? 112 + 8 * m : 48 + 8 * m;
    uint32_t oa[4], ob[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float4 t = h ? make_float4(1.0f, 0.0f, 1.0f, 0.0f) : __ldg(csr + 16 * (4 * m + k));
      const float2 ga = g2[(da >> 1) + k], gb = g2[(db >> 1) + k];
      const uint32_t wa = v[16 + 4 * m + k], wb = v[24 + 4 * m + k];
      const float ya0 = bf16lo(wa) * r * ga.x, ya1 = bf16hi(wa) * r * ga.y;
      const float yb0 = bf16lo(wb) * r * gb.x, yb1 = bf16hi(wb) * r * gb.y;
      oa[k] = pack_bf16x2(fmaf(h ? ya0 : yb0, h ? 0.0f : -t.y, ya0 * t.x),
                          fmaf(h ? ya1 : yb1, h ? 0.0f : -t.w, ya1 * t.z));
      ob[k] = pack_bf16x2(fmaf(h ? yb0 : ya0, h ? 0.0f : t.y, yb0 * t.x),
                          fmaf(h ? yb1 : ya1, h ? 0.0f : t.w, yb1 * t.z));
    }
    // boxes of 16 rows x 32 bytes (a: dims 0.. or 96.., b: 48.. or 112..), 32-byte swizzle
    const int rr = lane & 15;
    const int sw = (m ^ ((rr >> 2) & 1)) << 4;
    *reinterpret_cast<uint4*>(scratch + (h ? 2 : 0) * 512 + rr * 32 + sw) = make_uint4(oa[0], oa[1], oa[2], oa[3]);
    *reinterpret_cast<uint4*>(scratch + (h ? 3 : 1) * 512 + rr * 32 + sw) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tm16, scratch, col0 + 0, row0);
    tma_store_2d(tm16, scratch + 512, col0 + 48, row0);
    tma_store_2d(tm16, scratch + 1024, col0 + 96, row0);
    tma_store_2d(tm16, scratch + 1536, col0 + 112, row0);
    bulk_commit_group();
  }
}

// AMAX (SiLU*up with a bf16 output only): the epilogue also reduces
// max |float(h) * s_next| over the tile's valid rows, h the bf16 value it
// stores and s_next the per-channel pre_quant_scale of the projection that
// consumes h (null = 1); each CTA writes its maximum to amax_out[blockIdx.x]
// and CTA 0 the count gridDim.x to *amax_count.  The consumer's quantiser
// then needs no amax pass over h.
//
// ROPE (bf16 output of a fused QKV projection without SiLU*up): the tiles of
// Q and K heads take rope_head_epilogue; V tiles are stored as usual.
template <bool SILU, bool LORA, bool F32OUT, bool AMAX, bool ROPE>
__global__ void __launch_bounds__(PairRoles<SILU>::kThreads, 1) k_fp4gemm_pair(
    const __grid_constant__ CUtensorMap tm_xq, const __grid_constant__ CUtensorMap tm_wq,
    const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_b,
    const __grid_constant__ CUtensorMap tm_xs, const __grid_constant__ CUtensorMap tm_ws,
    const __grid_constant__ CUtensorMap tm_out, const __grid_constant__ CUtensorMap tm_out16,
    const float* __restrict__ ts_x, const float* __restrict__ ts_w, void* __restrict__ out, int M, int N, int K,
    int rank, int ldo, int group_m, uint32_t* __restrict__ status, const float* __restrict__ amax_s,
    float* __restrict__ amax_out, int* __restrict__ amax_count, const RopeEpi rope) {
  static_assert(!AMAX || (SILU && !F32OUT), "the fused amax serves the bf16 SiLU*up output");
  static_assert(!ROPE || (!SILU && !F32OUT && !AMAX), "the fused RoPE serves the bf16 QKV output");
  using C = PairCfg;
  constexpr int kPairCpWarps = PairRoles<SILU>::kCpWarps;
  constexpr int kPairEpiWarp0 = PairRoles<SILU>::kEpiWarp0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* epi_scratch = smem + C::kStages * C::kStageBytes;
  float* rope_gain = reinterpret_cast<float*>(epi_scratch + C::kEpiWarps * C::kEpiScratch);   // ROPE: Q, K gains
  uint64_t* full = reinterpret_cast<uint64_t*>(epi_scratch + C::kEpiWarps * C::kEpiScratch +
                                               (ROPE ? C::kRopeGainBytes : 0));
  uint64_t* empty = full + C::kStages;
  uint64_t* sf_full = empty + C::kStages;
  uint64_t* tmem_full = sf_full + C::kStages;
  uint64_t* tmem_empty = tmem_full + 1;
  uint64_t* drain_bar = tmem_empty + 1;
  uint64_t* drain_cp = drain_bar + 1;   // one per copy warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_cp + kPairCpWarps);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  float* amax_red = reinterpret_cast<float*>(abort_flag + 1);   // one per epilogue warp (AMAX)
  float* epi_post = amax_red + C::kEpiWarps;                     // epi_scale's second factor (1 normally)

  const int warp = warp_id(), lane = lane_id();
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_full[s], kPairCpWarps);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, 2 * C::kEpiWarps);
    mbar_init(drain_bar, 1);
    for (int w = 0; w < kPairCpWarps; ++w) mbar_init(&drain_cp[w], 1);
    *abort_flag = 0;
    *epi_post = epi_scale(*ts_x, *ts_w).b;
    fence_mbar_init();
    tma_prefetch_desc(&tm_xq);
    tma_prefetch_desc(&tm_wq);
    tma_prefetch_desc(&tm_xs);
    tma_prefetch_desc(&tm_ws);
    if (LORA) {
      tma_prefetch_desc(&tm_u);
      tma_prefetch_desc(&tm_b);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::kTmemCols);
    tmem_relinquish_pair();
  }
  if (ROPE && threadIdx.x < 256)
    rope_gain[threadIdx.x] = threadIdx.x < 128 ? rope.q_gain[threadIdx.x] : rope.k_gain[threadIdx.x - 128];
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag, status};

  const int tiles_m = (M + 255) >> 8;
  const int tiles_n = SILU ? (N / 2) / 128 : N / 256;
  const int num_tiles = tiles_m * tiles_n;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int nk = (K + 255) >> 8;
  const int nr = LORA ? (rank + 63) >> 6 : 0;
  const int k_atoms = K >> 6;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0;
      uint32_t filled = 0, fill_par = 0;   // leader: slots with a fill expected on full[], and its phase
      for (int t = pair; t < num_tiles; t += npairs) {
        int tm, tn;
        tile_coords(t, tiles_m, tiles_n, group_m, tm, tn);
        const int m0 = tm * 256 + 128 * static_cast<int>(crank);
        const int h0 = SILU ? tn * 128 : tn * 256;              // B rows of the tile's two halves
        const int h1 = SILU ? N / 2 + tn * 128 : tn * 256 + 128;
        const int brow = crank ? h1 : h0;                        // this CTA's half
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait(&empty[st], ph ^ 1, ab)) goto producer_done;
          uint8_t* base = smem + st * C::kStageBytes;
          const uint32_t lbar = cluster_addr(&full[st], 0);
          if (leader) {
            mbar_arrive_expect_tx(&full[st], 2 * C::kStageBytes);
            filled |= 1u << st;
            fill_par = (fill_par & ~(1u << st)) | (ph << st);
          }
          tma_load_2d_pair(base, &tm_xq, lbar, kc * 128, m0);
          tma_load_2d_pair(base + C::kABytes, &tm_wq, lbar, kc * 128, brow);
          tma_load_2d_pair(base + C::kABytes + C::kBBytes, &tm_xs, lbar, 0, 2 * ((m0 >> 7) * k_atoms + kc * 4));
          tma_load_2d_pair(base + C::kABytes + C::kBBytes + C::kSfaBytes, &tm_ws, lbar, 0,
                           2 * ((h0 >> 7) * k_atoms + kc * 4));
          tma_load_2d_pair(base + C::kABytes + C::kBBytes + C::kSfaBytes + 2048, &tm_ws, lbar, 0,
                           2 * ((h1 >> 7) * k_atoms + kc * 4));
          if (++st == C::kStages) { st = 0; ph ^= 1; }
        }
        for (int rc = 0; rc < nr; ++rc) {
          if (!mbar_wait(&empty[st], ph ^ 1, ab)) goto producer_done;
          uint8_t* base = smem + st * C::kStageBytes;
          const uint32_t lbar = cluster_addr(&full[st], 0);
          if (leader) {
            mbar_arrive_expect_tx(&full[st], 2 * (C::kABytes + C::kBBytes));
            filled |= 1u << st;
            fill_par = (fill_par & ~(1u << st)) | (ph << st);
          }
          tma_load_2d_pair(base, &tm_u, lbar, rc * 64, m0);
          tma_load_2d_pair(base + C::kABytes, &tm_b, lbar, rc * 64, brow);
          if (++st == C::kStages) { st = 0; ph ^= 1; }
        }
      }
    producer_done:
      // Both CTAs' loads of a stage complete on the leader's full barrier: before
      // this CTA pair can exit (after an abort, too) the leader waits, bounded,
      // for every fill it expected.  After a normal run these have all completed.
      if (leader)
        for (int s2 = 0; s2 < C::kStages; ++s2)
          if (filled & (1u << s2)) mbar_drain(&full[s2], (fill_par >> s2) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // A tcgen05.mma is accepted only about when the previous one starts, so every
    // instruction between two MMAs idles the tensor pipe: the loop waits on one
    // barrier per stage (sf_full: the copy warps commit it only after they saw
    // the stage's TMA data land, so it implies full) and issues the stage's MMAs
    // back to back from precomputed descriptors.
    if (lane == 0 && leader) {
      int st = 0;
      uint32_t ph = 0, acc_ph = 0;
      const uint32_t idesc_f4 = idesc_nvfp4_m256(256);
      const uint32_t idesc_bf = idesc_bf16_m256(256);
      const uint32_t smem0 = smem_u32(smem);
      const bool k_full = (K & 255) == 0;
      for (int t = pair; t < num_tiles; t += npairs) {
        // the tile's first stage is waited for while the epilogue still drains
        // the accumulator, so the first MMA follows the release directly
        if (!mbar_wait(&sf_full[st], ph, ab) || !mbar_wait(tmem_empty, acc_ph ^ 1, ab)) goto mma_done;
        tc_fence_after();
        for (int kc = 0; kc < nk; ++kc) {
          if (kc > 0 && !mbar_wait(&sf_full[st], ph, ab)) goto mma_done;
          tc_fence_after();
          const uint32_t a_addr = smem0 + st * C::kStageBytes;
          // +32 bytes along K = +2 in a descriptor's start-address field
          const uint64_t ad = sdesc_kmajor_sw128(a_addr), bd = sdesc_kmajor_sw128(a_addr + C::kABytes);
          const uint32_t sf = tmem + 256 + st * C::kSfCols;
          if (k_full) {
            mma_nvfp4_pair(tmem, ad, bd, idesc_f4, sf, sf + 16, kc != 0);
            mma_nvfp4_pair(tmem, ad + 2, bd + 2, idesc_f4, sf + 4, sf + 24, 1u);
            mma_nvfp4_pair(tmem, ad + 4, bd + 4, idesc_f4, sf + 8, sf + 32, 1u);
            mma_nvfp4_pair(tmem, ad + 6, bd + 6, idesc_f4, sf + 12, sf + 40, 1u);
          } else {
            const int nsub = min(4, (K - kc * 256) >> 6);
            for (int j = 0; j < nsub; ++j)
              mma_nvfp4_pair(tmem, ad + 2 * j, bd + 2 * j, idesc_f4, sf + 4 * j, sf + 16 + 8 * j, (kc | j) != 0);
          }
          tc_commit_pair_mc(&empty[st]);
          if (++st == C::kStages) { st = 0; ph ^= 1; }
        }
        for (int rc = 0; rc < nr; ++rc) {
          if (!mbar_wait(&sf_full[st], ph, ab)) goto mma_done;
          tc_fence_after();
          const uint32_t a_addr = smem0 + st * C::kStageBytes;
          const uint64_t ad = sdesc_kmajor_sw128(a_addr), bd = sdesc_kmajor_sw128(a_addr + C::kABytes);
          const int nk16 = min(4, (rank - rc * 64) >> 4);
          for (int j = 0; j < nk16; ++j) mma_bf16_pair(tmem, ad + 2 * j, bd + 2 * j, idesc_bf, 1u);
          tc_commit_pair_mc(&empty[st]);
          if (++st == C::kStages) { st = 0; ph ^= 1; }
        }
        tc_commit_pair_mc(tmem_full);
        acc_ph ^= 1;
      }
    mma_done:
      tc_commit_pair(drain_bar);
      mbar_drain(drain_bar, 0);
    }
  } else if (warp < kPairEpiWarp0) {
    // ------------------------------------------------- scale atoms -> TMEM
    // Copy i (0..11) of a stage: K step j = i / 3; kind i % 3 = A rows, B half 0, B half 1.
    const int cw = warp - 2;
    if (lane == 0 && leader) {
      int st = 0;
      uint32_t ph = 0;
      for (int t = pair; t < num_tiles; t += npairs) {
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait(&full[st], ph, ab)) goto cp_done;
          tc_fence_after();
          const int nsub = min(4, (K - kc * 256) >> 6);
          const uint32_t sfa_addr = smem_u32(smem + st * C::kStageBytes) + C::kABytes + C::kBBytes;
          const uint32_t sf_col = tmem + 256 + st * C::kSfCols;
          for (int i = cw; i < 12; i += kPairCpWarps) {
            const int j = i / 3, kind = i - 3 * j;
            if (j >= nsub) continue;
            if (kind == 0)
              tmem_cp_sf_atom_pair(sf_col + 4 * j, sdesc_sf_atom(sfa_addr + j * 512));
            else
              tmem_cp_sf_atom_pair(sf_col + 16 + 8 * j + 4 * (kind - 1),
                                   sdesc_sf_atom(sfa_addr + C::kSfaBytes + (kind - 1) * 2048 + j * 512));
          }
          tc_commit_pair(&sf_full[st]);
          if (++st == C::kStages) { st = 0; ph ^= 1; }
        }
        for (int rc = 0; rc < nr; ++rc) {   // LoRA stages carry no scales
          if (!mbar_wait(&full[st], ph, ab)) goto cp_done;
          tc_commit_pair(&sf_full[st]);
          if (++st == C::kStages) { st = 0; ph ^= 1; }
        }
      }
    cp_done:
      tc_commit_pair(&drain_cp[cw]);
      mbar_drain(&drain_cp[cw], 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                  // TMEM lane quarter of this warp
    const int e = warp - kPairEpiWarp0;
    const int c4 = e >> 2;                   // which quarter of the tile's columns
    uint8_t* scratch = epi_scratch + e * C::kEpiScratch;
    const float scale = epi_scale(*ts_x, *ts_w).a;
    const uint32_t leader_tmem_empty = cluster_addr(tmem_empty, 0);
    constexpr int kEsize = F32OUT ? 4 : 2;
    constexpr int kRoundCols = 64 / kEsize;          // output columns per 64-byte staging row
    constexpr int kRounds = (SILU ? 32 : 64) / kRoundCols;
    uint32_t acc_ph = 0;
    float am = 0.0f;                         // AMAX: running max of |h * s_next|
    for (int t = pair; t < num_tiles; t += npairs) {
      int tm, tn;
      tile_coords(t, tiles_m, tiles_n, group_m, tm, tn);
      if (!mbar_wait(tmem_full, acc_ph, ab)) break;
      tc_fence_after();
      if (ROPE && tn < rope.heads) {   // the tile's two heads are both Q or both K heads
        const int hs = c4 >> 1, rh = c4 & 1;   // head of the tile, half of the quarter's rows
        const int head = 2 * tn + hs;
        rope_head_epilogue(tmem + (static_cast<uint32_t>(32 * q + 16 * rh) << 16) + 128 * hs, leader_tmem_empty,
                           scale, *epi_post, rope_gain + (head < rope.heads ? 0 : 128), rope.cs,
                           tm * 256 + 128 * static_cast<int>(crank) + 32 * q + 16 * rh + (lane & 15), M,
                           static_cast<__nv_bfloat16*>(out), 128 * head, ldo, rope.eps, lane, status, scratch,
                           &tm_out16, tm * 256 + 128 * static_cast<int>(crank) + 32 * q + 16 * rh);
        acc_ph ^= 1;
        continue;
      }
      const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16);
      const int row0 = tm * 256 + 128 * static_cast<int>(crank) + 32 * q;   // first row of this warp
      const int col0 = SILU ? tn * 128 + c4 * 32 : tn * 256 + c4 * 64;
      // SiLU*up: a = gate columns c4*32.., b = the matching up columns 128 + c4*32..
      // otherwise: a, b = accumulator columns c4*64 .. c4*64 + 63
      uint32_t a[32], b[32];
      tmem_ld32(taddr + (SILU ? c4 * 32 : c4 * 64), a);
      tmem_ld32(taddr + (SILU ? 128 + c4 * 32 : c4 * 64 + 32), b);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(leader_tmem_empty);
#pragma unroll
      for (int rd = 0; rd < kRounds; ++rd) {
        uint32_t w[16];
        const float post = *epi_post;   // != 1 for tiny tensor scales only
        if (post != 1.0f)
          epi_convert<SILU, F32OUT, true>(scale, post, a, b, rd, w);
        else
          epi_convert<SILU, F32OUT, false>(scale, 1.0f, a, b, rd, w);
        if (AMAX && row0 + lane < M && in_bounds(col0 + rd * kRoundCols + kRoundCols <= ldo, status)) {
          // per element: |fl(h * s)| with h the stored bf16 value (the lanes'
          // loads of s are broadcasts: all lanes read the same 32 columns)
          const int cb = col0 + rd * kRoundCols;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 sv = amax_s ? __ldg(reinterpret_cast<const float2*>(amax_s + cb) + k) : make_float2(1.0f, 1.0f);
            am = fmaxf(am, fabsf(__fmul_rn(bf16lo(w[k]), sv.x)));
            am = fmaxf(am, fabsf(__fmul_rn(bf16hi(w[k]), sv.y)));
          }
        }
        epi_scratch_ready(lane);
        // row = lane, 64 bytes; 16-byte chunks placed as the 64-byte TMA swizzle expects
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
          *reinterpret_cast<uint4*>(scratch + lane * 64 + ((ch ^ ((lane >> 1) & 3)) << 4)) =
              make_uint4(w[4 * ch], w[4 * ch + 1], w[4 * ch + 2], w[4 * ch + 3]);
        epi_store(&tm_out, scratch, col0 + rd * kRoundCols, row0, lane);
      }
      acc_ph ^= 1;
    }
    if (lane == 0) bulk_wait_group0();   // this warp's output stores are complete
    __syncwarp();
    if (AMAX) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
      if (lane == 0) amax_red[e] = am;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (AMAX && threadIdx.x == 0) {
    float m = amax_red[0];
    for (int i = 1; i < C::kEpiWarps; ++i) m = fmaxf(m, amax_red[i]);
    if (in_bounds(blockIdx.x < static_cast<unsigned>(kMaxPartials), status)) amax_out[blockIdx.x] = m;
    if (blockIdx.x == 0) *amax_count = static_cast<int>(gridDim.x);
  }
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
}

template <bool SILU, bool LORA, bool F32OUT, bool AMAX = false, bool ROPE = false>
static cudaError_t launch_pair_variant(const GemmArgs& a, int sm_count, cudaStream_t st) {
  auto kern = k_fp4gemm_pair<SILU, LORA, F32OUT, AMAX, ROPE>;
  const int smem = ROPE ? PairCfg::kSmemRope : PairCfg::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int tiles_m = (a.M + 255) / 256;
  const int tiles_n = SILU ? (a.N / 2) / 128 : a.N / 256;
  const int tiles = tiles_m * tiles_n;
  const int max_pairs = sm_count / 2;
  const int grid = 2 * (tiles < max_pairs ? tiles : max_pairs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(PairRoles<SILU>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  trace_launch("k_fp4gemm_pair", grid, 2, PairRoles<SILU>::kThreads, smem,
               "silu=%d lora=%d f32out=%d amax=%d rope=%d M=%d N=%d K=%d rank=%d tiles=%d raster_group=%d",
               int(SILU), int(LORA), int(F32OUT), int(AMAX), int(ROPE), a.M, a.N, a.K, a.rank, tiles, a.group_m);
  return cudaLaunchKernelEx(&cfg, kern, a.tm_xq, a.tm_wq, a.tm_u, a.tm_b, a.tm_xs, a.tm_ws, a.tm_out, a.tm_out16,
                            a.ts_x, a.ts_w,
                            a.out, a.M, a.N, a.K, a.rank, a.ldo, a.group_m, a.status, a.amax_s, a.amax_out,
                            a.amax_count, a.rope);
}

template <bool F32OUT>
static cudaError_t launch_pair_dtype(const GemmArgs& a, int sm_count, cudaStream_t st) {
  if (!F32OUT && !a.silu && a.rope.cs) {
    return a.lora ? launch_pair_variant<false, true, false, false, true>(a, sm_count, st)
                  : launch_pair_variant<false, false, false, false, true>(a, sm_count, st);
  }
  if (!F32OUT && a.silu && a.amax_out) {
    return a.lora ? launch_pair_variant<true, true, false, true>(a, sm_count, st)
                  : launch_pair_variant<true, false, false, true>(a, sm_count, st);
  }
  if (a.silu) {
    return a.lora ? launch_pair_variant<true, true, F32OUT>(a, sm_count, st)
                  : launch_pair_variant<true, false, F32OUT>(a, sm_count, st);
  }
  return a.lora ? launch_pair_variant<false, true, F32OUT>(a, sm_count, st)
                : launch_pair_variant<false, false, F32OUT>(a, sm_count, st);
}

template <bool F32OUT>
static cudaError_t launch_dtype(const GemmArgs& a, int sm_count, cudaStream_t st) {
  if (a.silu) {
    return a.lora ? launch_variant<256, true, true, F32OUT>(a, sm_count, st)
                  : launch_variant<256, true, false, F32OUT>(a, sm_count, st);
  }
  if (a.N % 256 == 0) {
    return a.lora ? launch_variant<256, false, true, F32OUT>(a, sm_count, st)
                  : launch_variant<256, false, false, F32OUT>(a, sm_count, st);
  }
  return a.lora ? launch_variant<128, false, true, F32OUT>(a, sm_count, st)
                : launch_variant<128, false, false, F32OUT>(a, sm_count, st);
}

// M-tiles per raster group of the GEMM.  A narrow weight (N <= 8192, packed
// codes and scales <= 48 MB) stays resident in L2 while its few N tiles are
// swept, so the raster runs N-fastest and every x panel is read from HBM once
// (measured on the block: attn-out and down GEMM reads drop from 0.21 and 1.79
// GB to 0.13 and 0.54 GB).  A wide weight (QKV, gate/up) is evicted by the
// output streaming through L2 between its reuses; there a group keeps about
// 24 MB of x panels in L2 while the weight panels pass.
int raster_group(int64_t N, int64_t K, int tile_rows) {
  const int64_t weight_bytes = N * (K / 2) + N * (K / 16);
  if (N <= 8192 && weight_bytes <= (int64_t(48) << 20)) return 1;
  const int64_t panel = int64_t(tile_rows) * (K / 2);
  int64_t g = (int64_t(24) << 20) / (panel > 0 ? panel : 1);
  if (g < 1) g = 1;
  if (g > 32) g = 32;
  return int(g);
}

cudaError_t launch_fp4gemm(const GemmArgs& a, int sm_count, cudaStream_t st) {
  if (a.pair) return a.f32out ? launch_pair_dtype<true>(a, sm_count, st) : launch_pair_dtype<false>(a, sm_count, st);
  return a.f32out ? launch_dtype<true>(a, sm_count, st) : launch_dtype<false>(a, sm_count, st);
}

}  // namespace h3lin
