// Activation side of the dynamic-LoRA NVFP4 linear (TURBO.md,
// h3-blackwell-runtime, "Implementation"; MiniMax-H3 Ultra Fast README,
// "Kernel path", item 1: dynamic NVFP4 activation quantisation):
//
//   k_amax       amax |x * s| over the tensor -> one partial per CTA
//   k_amax_lora  the same pass with TMA-staged tiles, fused with the LoRA
//                down projection u = A(x) on the BF16 tensor cores (tcgen05,
//                accumulator in TMEM); the LoRA branch sees the original x
//   k_quant      reduces the partials to the tensor scale, quantises x * s to
//                E2M1 codes + E4M3 block scales (bit-exact rules below), and
//                optionally writes B' = B * strength * (alpha/rank) / (ts_x ts_w)
//                so that the GEMM can accumulate B'(u) into the FP4 tile
//                (for tiny tensor scales a power of two moves from B' to u).
//   k_amax_lora<QUANT>  when a producer GEMM's epilogue already reduced the
//                amax of x (the gate/up output feeding down): the TMA-staged
//                pass quantises x and computes u = A(x) in one read of x.
//
// Quantisation rules (float32, round to nearest even at every step):
//   v = x * s;  ts = amax / 2688 (0 -> 1);  per 16 elements:
//   sb = E4M3_sat(blockamax / (6 ts));  d = E4M3(sb) * ts;
//   code = E2M1_sat(v / d) with the sign of v kept;  d == 0 -> all codes 0.
#include "h3lin_device.cuh"

namespace h3lin {

// ----------------------------------------------------------------- helpers
__device__ __forceinline__ void load_scale8(const float* __restrict__ pqs, int c, float (&s)[8]) {
  if (pqs == nullptr) {
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = 1.0f;
  } else {
    const float4 a = __ldg(reinterpret_cast<const float4*>(pqs) + 2 * c);
    const float4 b = __ldg(reinterpret_cast<const float4*>(pqs) + 2 * c + 1);
    s[0] = a.x; s[1] = a.y; s[2] = a.z; s[3] = a.w;
    s[4] = b.x; s[5] = b.y; s[6] = b.z; s[7] = b.w;
  }
}

__device__ __forceinline__ void prescale8(const uint4& w, const float (&s)[8], float (&v)[8]) {
  fmul2_rn(bf16lo(w.x), bf16hi(w.x), s[0], s[1], v[0], v[1]);
  fmul2_rn(bf16lo(w.y), bf16hi(w.y), s[2], s[3], v[2], v[3]);
  fmul2_rn(bf16lo(w.z), bf16hi(w.z), s[4], s[5], v[4], v[5]);
  fmul2_rn(bf16lo(w.w), bf16hi(w.w), s[6], s[7], v[6], v[7]);
}

// max |x * s| over rows, without a multiply per element: rounding is monotone,
// so max_r |fl(x_r * s)| = fl(max_r |x_r| * |s|) exactly.  The column-wise
// max |x| is kept as four bf16 pairs (NaN operands are skipped, as fmaxf
// skips them), and scaled once per column.
struct ColMax8 {
  __nv_bfloat162 h[4];
  __device__ __forceinline__ ColMax8() {
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __float2bfloat162_rn(0.0f);
  }
  __device__ __forceinline__ void add(const uint4& w) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __hmax2(h[i], __habs2(*reinterpret_cast<const __nv_bfloat162*>(&u[i])));
  }
  // max over the 8 columns of |colmax * s| (a tree of maxima: short dependency chains)
  __device__ __forceinline__ float scaled_max(const float (&s)[8]) const {
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t u = *reinterpret_cast<const uint32_t*>(&h[i]);
      v[2 * i] = __fmul_rn(bf16lo(u), fabsf(s[2 * i]));
      v[2 * i + 1] = __fmul_rn(bf16hi(u), fabsf(s[2 * i + 1]));
    }
    return fmaxf(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])), fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7])));
  }
};

// Block-wide max; every thread gets the result.
__device__ __forceinline__ float block_max(float m, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  const int nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = red[0];
  for (int i = 1; i < nw; ++i) m = fmaxf(m, red[i]);
  return m;
}

// ----------------------------------------------------------------- k_amax
// Thread t owns 16-byte column chunk c = t % kc of rows r0, r0 + R, ... with
// r0 = t / kc (R = rows_step).  The 8 per-channel scales live in registers.
__global__ void __launch_bounds__(kQuantThreads) k_amax(const uint4* __restrict__ x, int M, int kc,
                                                       const float* __restrict__ pqs,
                                                       float* __restrict__ partials, int rows_step,
                                                       int* __restrict__ count_out, uint32_t* status) {
  __shared__ float red[kQuantThreads / 32];
  const int tid = blockIdx.x * kQuantThreads + threadIdx.x;
  const int c = tid % kc;
  const int r0 = tid / kc;
  float m = 0.0f;
  if (r0 < rows_step) {
    ColMax8 cm;
    int row = r0;
    const int64_t x_chunks = static_cast<int64_t>(M) * kc;
    for (; row + rows_step < M; row += 2 * rows_step) {
      const int64_t ia = static_cast<int64_t>(row) * kc + c, ib = static_cast<int64_t>(row + rows_step) * kc + c;
      if (!in_bounds(ia < x_chunks && ib < x_chunks, status)) break;
      const uint4 a = x[ia];
      const uint4 b = x[ib];
      cm.add(a);
      cm.add(b);
    }
    if (row < M && in_bounds(static_cast<int64_t>(row) * kc + c < x_chunks, status))
      cm.add(x[static_cast<int64_t>(row) * kc + c]);
    float s[8];
    load_scale8(pqs, c, s);
    m = cm.scaled_max(s);
  }
  m = block_max(m, red);
  if (threadIdx.x == 0 && in_bounds(blockIdx.x < static_cast<unsigned>(kMaxPartials), status)) {
    partials[blockIdx.x] = m;
    if (count_out && blockIdx.x == 0) *count_out = static_cast<int>(gridDim.x);
  }
}

// ---------------------------------------------------------------- k_quant
// Thread t owns 16-element block b = t % (K/16) of rows r0, r0 + R, ... with
// r0 = t / (K/16): its 16 per-channel scales stay in registers, the block
// scale is computed once per block, and each thread stores its own scale byte.
struct QuantCtx {
  float ts, six_ts;
  float rcp_six_ts;       // fl(1 / six_ts)
  const float2* yt;       // bracket of 1 / d for every scale byte (shared memory, bracket_entry)
};
__device__ __forceinline__ QuantCtx make_quant_ctx(float ts, const float2* yt) {
  const float six_ts = __fmul_rn(6.0f, ts);
  return QuantCtx{ts, six_ts, __frcp_rn(six_ts), yt};
}

// sb = E4M3_sat(fl(bm / (6 ts))), mostly without the division: p = fl(bm *
// fl(1 / (6 ts))) lies within 2.5 ulp of the exact quotient, so p and the
// IEEE quotient are at most 2 ulp apart and round to the same E4M3 value
// unless an E4M3 rounding midpoint (float mantissa bit 19 set, bits 18-0
// clear) is within 3 ulp of p, or p is below 2^-6 (E4M3's subnormal range,
// where the midpoints sit elsewhere).  Only those cases take the division.
__device__ __forceinline__ uint32_t block_scale_byte(float bm, const QuantCtx& q) {
  const float p = __fmul_rn(bm, q.rcp_six_ts);
  const uint32_t low = __float_as_uint(p) & 0xFFFFFu;
  if (p < 0x1p-6f || low - (0x80000u - 3u) <= 6u) return e4m3_rn_satfinite(__fdiv_rn(bm, q.six_ts));
  return e4m3_rn_satfinite(p);
}

// Element codes are E2M1(fl(v / d)), the IEEE quotient rounded once.  The
// quotient is not taken per element: with y = fl(1 / d), the products
// q_lo = fl(v fl(y (1 - 2^-21))) and q_hi = fl(v fl(y (1 + 2^-21))) lie
// strictly on either side of fl(v / d) (each is at least 5 * 2^-24 away from
// v / d in relative terms, the rounded quotient at most 2^-24, while all
// values are normal floats, which d > 2^-100 ensures for any value that can
// reach an E2M1 midpoint), and the E2M1 value is monotone in its argument,
// so where q_lo and q_hi give the same code that is the quotient's code.
// They differ only for a quotient within about 2^-21 (relative) of an E2M1
// rounding midpoint: there, element by element, the IEEE division decides.
// Such quotients are frequent on bf16 data (short mantissas make exact
// midpoints of v / d common: a few elements in 10^4), so only the differing
// elements divide.  A block with d <= 2^-100 divides every element.
// bracket_entry(ts, sb) = (fl(y (1 - 2^-21)), fl(y (1 + 2^-21))), tabulated
// once per CTA for the 256 scale bytes (y = inf for d == 0).
__device__ __forceinline__ float2 bracket_entry(float ts, uint32_t sb) {
  const float y = __frcp_rn(__fmul_rn(e4m3_to_float(sb), ts));
  return make_float2(__fmul_rn(y, 1.0f - 0x1p-21f), __fmul_rn(y, 1.0f + 0x1p-21f));
}
__device__ __forceinline__ void build_bracket_table(float2* yt, float ts) {
  for (int i = threadIdx.x; i < 256; i += blockDim.x) yt[i] = bracket_entry(ts, i);
}

// The slow path of block_codes, out of line so that the hot loop stays small:
// element i takes the IEEE division where its two bracket codes differ (bit i
// of `which`), or every element when `which` is all ones.
__device__ __noinline__ uint2 block_codes_slow(const float* v, float d, uint32_t which, uint2 c) {
  if (d == 0.0f) return make_uint2(0u, 0u);
#pragma unroll 1
  for (int i = 0; i < 16; ++i) {
    if (!((which >> i) & 1u)) continue;
    const float q[8] = {__fdiv_rn(v[i], d), 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    const uint32_t code = e2m1x8(q) & 0xFu;
    const int sh = 4 * (i & 7);
    if (i < 8)
      c.x = (c.x & ~(0xFu << sh)) | (code << sh);
    else
      c.y = (c.y & ~(0xFu << sh)) | (code << sh);
  }
  return c;
}

// One bit per element whose 4-bit codes in a and b differ.
__device__ __forceinline__ uint32_t nibble_mask(uint32_t x) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m |= ((x >> (4 * i)) & 0xFu) != 0u ? (1u << i) : 0u;
  return m;
}

__device__ __forceinline__ uint2 block_codes(const float (&v)[16], float2 y, float ts, uint32_t sb) {
  float la[8], lb[8], ha[8], hb[8];
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    fmul2_rn(v[i], v[i + 1], y.x, y.x, la[i], la[i + 1]);
    fmul2_rn(v[8 + i], v[9 + i], y.x, y.x, lb[i], lb[i + 1]);
    fmul2_rn(v[i], v[i + 1], y.y, y.y, ha[i], ha[i + 1]);
    fmul2_rn(v[8 + i], v[9 + i], y.y, y.y, hb[i], hb[i + 1]);
  }
  const uint2 c = make_uint2(e2m1x8(la), e2m1x8(lb));
  const uint32_t dx = c.x ^ e2m1x8(ha), dy = c.y ^ e2m1x8(hb);
  const bool bracket_ok = y.y < 0x1p100f;
  if (bracket_ok && (dx | dy) == 0u) return c;
  float vv[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) vv[i] = v[i];
  const uint32_t which = bracket_ok ? (nibble_mask(dx) | (nibble_mask(dy) << 8)) : 0xFFFFu;
  return block_codes_slow(vv, __fmul_rn(e4m3_to_float(sb), ts), which, c);
}

__device__ __forceinline__ void load_scale16(const float* __restrict__ pqs, int b, float (&s)[16]) {
  if (pqs == nullptr) {
#pragma unroll
    for (int i = 0; i < 16; ++i) s[i] = 1.0f;
  } else {
    const float4* p = reinterpret_cast<const float4*>(pqs) + 4 * b;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 a = __ldg(p + i);
      s[4 * i] = a.x; s[4 * i + 1] = a.y; s[4 * i + 2] = a.z; s[4 * i + 3] = a.w;
    }
  }
}

// Quantise one 16-element block (two 16-byte halves): its 16 codes go to
// *code (skipped when code is null: rows >= M have none) and its scale byte
// to *sf (each thread writes its own byte of the row's 4-byte scale word).
__device__ __forceinline__ void quant_block(const QuantCtx& q, uint2* code, uint8_t* sf, const uint4& w0,
                                            const uint4& w1, const float (&s)[16]) {
  float v[16];
  {
    float h0[8], h1[8], s0[8], s1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { s0[i] = s[i]; s1[i] = s[8 + i]; }
    prescale8(w0, s0, h0);
    prescale8(w1, s1, h1);
#pragma unroll
    for (int i = 0; i < 8; ++i) { v[i] = h0[i]; v[8 + i] = h1[i]; }
  }
  float bm = fabsf(v[0]);
#pragma unroll
  for (int i = 1; i < 16; ++i) bm = fmaxf(bm, fabsf(v[i]));
  const uint32_t sb = block_scale_byte(bm, q);
  const uint2 cw = block_codes(v, q.yt[sb], q.ts, sb);
  if (code) *code = cw;
  *sf = static_cast<uint8_t>(sb);
}

// B' = bf16(B * c) over [b_chunks] 16-byte chunks, grid-strided from `first`
// by `stride`; and, when the LoRA scale moved a power of two to u (u_mul != 1),
// u *= u_mul in place over [u_chunks] chunks (u was written by the amax pass).
__device__ __forceinline__ void scale_lora_operands(const LoraScale& ls, const uint4* __restrict__ b_src,
                                                    uint4* __restrict__ b_dst, int64_t b_chunks, uint4* u,
                                                    int64_t u_chunks, int64_t first, int64_t stride) {
  for (int64_t i = first; i < b_chunks; i += stride) {
    const uint4 w = __ldg(b_src + i);
    uint4 o;
    o.x = pack_bf16x2(__fmul_rn(bf16lo(w.x), ls.c), __fmul_rn(bf16hi(w.x), ls.c));
    o.y = pack_bf16x2(__fmul_rn(bf16lo(w.y), ls.c), __fmul_rn(bf16hi(w.y), ls.c));
    o.z = pack_bf16x2(__fmul_rn(bf16lo(w.z), ls.c), __fmul_rn(bf16hi(w.z), ls.c));
    o.w = pack_bf16x2(__fmul_rn(bf16lo(w.w), ls.c), __fmul_rn(bf16hi(w.w), ls.c));
    b_dst[i] = o;
  }
  if (ls.u_mul != 1.0f && u != nullptr) {
    for (int64_t i = first; i < u_chunks; i += stride) {
      const uint4 w = u[i];
      uint4 o;
      o.x = pack_bf16x2(__fmul_rn(bf16lo(w.x), ls.u_mul), __fmul_rn(bf16hi(w.x), ls.u_mul));
      o.y = pack_bf16x2(__fmul_rn(bf16lo(w.y), ls.u_mul), __fmul_rn(bf16hi(w.y), ls.u_mul));
      o.z = pack_bf16x2(__fmul_rn(bf16lo(w.z), ls.u_mul), __fmul_rn(bf16hi(w.z), ls.u_mul));
      o.w = pack_bf16x2(__fmul_rn(bf16lo(w.w), ls.u_mul), __fmul_rn(bf16hi(w.w), ls.u_mul));
      u[i] = o;
    }
  }
}

// Rows are visited from the last to the first: the amax pass streamed them
// in ascending order, so the tail of x is still in L2 when this pass starts.
__global__ void __launch_bounds__(kQuantThreads, 4) k_quant(
    const uint4* __restrict__ x, int M, int Mpad, int K, const float* __restrict__ pqs,
    const float* __restrict__ partials, int nparts, const int* __restrict__ nparts_dev, uint2* __restrict__ codes,
    uint8_t* __restrict__ scales, float* __restrict__ ts_out, int rows_step, const uint4* __restrict__ b_src,
    uint4* __restrict__ b_dst, int64_t b_chunks, float lora_k, const float* __restrict__ ts_w, uint4* u,
    int64_t u_chunks, uint32_t* status) {
  __shared__ float red[kQuantThreads / 32];
  __shared__ float2 yt[256];
  float m = 0.0f;
  if (nparts_dev) nparts = min(max(*nparts_dev, 0), kMaxPartials);   // never read past the partials
  for (int i = threadIdx.x; i < nparts; i += kQuantThreads)
    if (in_bounds(i < kMaxPartials, status)) m = fmaxf(m, partials[i]);
  const float amax = block_max(m, red);
  float ts = __fdiv_rn(amax, 2688.0f);
  if (ts == 0.0f) ts = 1.0f;
  if (blockIdx.x == 0 && threadIdx.x == 0) *ts_out = ts;
  const int kb = K >> 4;
  build_bracket_table(yt, ts);
  __syncthreads();
  const QuantCtx q = make_quant_ctx(ts, yt);

  const int tid = blockIdx.x * kQuantThreads + threadIdx.x;
  const int b = tid % kb;
  const int r0 = tid / kb;
  const int kc = K >> 3;   // 16-byte chunks per row
  if (r0 < rows_step) {
    float s[16];
    load_scale16(pqs, b, s);
    for (int i = r0; i < Mpad; i += 2 * rows_step) {
      const int ra = Mpad - 1 - i;
      const bool has_b = i + rows_step < Mpad;
      const int rb = Mpad - 1 - (i + rows_step);
      uint4 a0 = make_uint4(0, 0, 0, 0), a1 = a0, c0 = a0, c1 = a0;
      // bounds build: x chunks, code words and scale bytes against their buffers
      const int64_t x_chunks = static_cast<int64_t>(M) * kc, code_words = static_cast<int64_t>(M) * kb;
      const int64_t sf_bytes = static_cast<int64_t>(Mpad) * kb;
      if (ra < M && in_bounds(static_cast<int64_t>(ra) * kc + 2 * b + 1 < x_chunks, status)) {
        const uint4* p = x + static_cast<int64_t>(ra) * kc + 2 * b;
        a0 = __ldcs(p);
        a1 = __ldcs(p + 1);
      }
      if (has_b && rb < M && in_bounds(static_cast<int64_t>(rb) * kc + 2 * b + 1 < x_chunks, status)) {
        const uint4* p = x + static_cast<int64_t>(rb) * kc + 2 * b;
        c0 = __ldcs(p);
        c1 = __ldcs(p + 1);
      }
      if (in_bounds(ra >= 0 && sf_offset(ra, b, K) < sf_bytes && (ra >= M || static_cast<int64_t>(ra) * kb + b < code_words),
                    status)) {
        if (ra < M) quant_block(q, codes + static_cast<int64_t>(ra) * kb + b, scales + sf_offset(ra, b, K), a0, a1, s);
        else scales[sf_offset(ra, b, K)] = 0;
      }
      if (has_b && in_bounds(rb >= 0 && sf_offset(rb, b, K) < sf_bytes &&
                             (rb >= M || static_cast<int64_t>(rb) * kb + b < code_words), status)) {
        if (rb < M) quant_block(q, codes + static_cast<int64_t>(rb) * kb + b, scales + sf_offset(rb, b, K), c0, c1, s);
        else scales[sf_offset(rb, b, K)] = 0;
      }
    }
  }
  if (b_chunks > 0) {
    const LoraScale ls = lora_scale(lora_k, ts, *ts_w);
    scale_lora_operands(ls, b_src, b_dst, b_chunks, u, u_chunks, tid,
                        static_cast<int64_t>(gridDim.x) * kQuantThreads);
  }
}

// ------------------------------------------------------------- k_amax_lora
// Warp 0: TMA producer.  Warp 1: TMEM owner + MMA issuer.  Warps 2-9: amax of
// |x * s| read from the staged tile, then the epilogue u = bf16(TMEM).
// One 128-row tile of x per CTA iteration; K in 64-column stages (x tile
// 128 x 64 bf16 = 16 KB, A tile rank x 64 bf16), 128-byte swizzle.
// Amax thread a owns the 16-byte column chunk a % 8 of rows a / 8 + R i
// (R = 32 * warps / 8) of every stage, so its 8 per-channel scales are two
// loads per stage.
constexpr int kLoraAmaxWarps = 8;   // per 128 rows of the tile
// Worker warps per CTA of the quantising variant.  Two CTAs share an SM when
// the TMEM accumulator and the ring fit twice (rank <= 256): each CTA's
// pipeline (ring fill, tile epilogue, stalls) then overlaps the other's, which
// measured faster than one CTA with twice the workers.
constexpr int kLoraQuantWarps = 8;   // per 128 rows of the tile
constexpr bool kLoraAmaxTwoCtas = true;   // the amax pass takes two CTAs per SM as well
// ROWS: rows of x per tile, 128 or 256.  A 256-row tile (one CTA per SM, two
// 128-row accumulators, twice the workers) stages 32 KB of x against one
// A slice per K step, so an SM holds a third more of x in flight than two
// CTAs of 128-row tiles; it needs 2 * (rank / parts) <= 256 TMEM columns.
template <bool QUANT, int ROWS> constexpr int lora_workers() {
  return (QUANT ? kLoraQuantWarps : kLoraAmaxWarps) * (ROWS / 128);
}
template <bool QUANT, int ROWS> constexpr int lora_threads() { return 64 + 32 * lora_workers<QUANT, ROWS>(); }

// QUANT: the amax is known (partials_in, *nparts_dev of them, left by a
// producer GEMM), so warps 2-17 quantise the staged tile instead: thread a
// owns 16-element block a % 4 of the stage's 64 columns in row a / 4 (the
// four threads of a row assemble its 32-bit scale word).
struct QuantPassOut {
  const float* partials_in;
  const int* nparts_dev;
  uint2* codes;
  uint8_t* scales;
  float* ts_out;
  const uint4* b_src;   // optional B' = bf16(B * lora_k / (ts * ts_w)), as k_quant
  uint4* b_dst;
  int64_t b_chunks;
  float lora_k;
  const float* ts_w;
};

template <bool QUANT, int ROWS>
__global__ void __launch_bounds__(lora_threads<QUANT, ROWS>(), ROWS == 128 ? 2 : 1) k_amax_lora(
    const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_a, int M, int K,
    int rank, int parts, int a_box_rows, const float* __restrict__ pqs, float* __restrict__ partials,
    __nv_bfloat16* __restrict__ u, uint32_t* __restrict__ status, int stages, int tmem_cols, QuantPassOut qo) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  static_assert(ROWS == 128 || ROWS == 256, "tile rows");
  constexpr int kXBytes = ROWS * 128;   // x tile of a stage: ROWS x 64 bf16
  const int pr = rank / parts;   // rank columns of u one work item computes
  const int stage_bytes = kXBytes + pr * 128;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + stages * stage_bytes);
  uint64_t* empty = full + stages;
  uint64_t* tmem_full = empty + stages;
  uint64_t* tmem_empty = tmem_full + 1;
  uint64_t* drain_bar = tmem_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(abort_flag + 1);
  float2* yt = reinterpret_cast<float2*>(smem + stages * stage_bytes + 256);   // QUANT: 256 brackets of 1 / d

  constexpr int kWorkers = lora_workers<QUANT, ROWS>();
  constexpr int kThreads = lora_threads<QUANT, ROWS>();
  const int warp = warp_id(), lane = lane_id();
  if (QUANT) {   // tensor amax from the producer's partials (every CTA, deterministic)
    const int n = min(max(*qo.nparts_dev, 0), kMaxPartials);   // never read past the partials
    float m = 0.0f;
    for (int i = threadIdx.x; i < n; i += kThreads)
      if (in_bounds(i < kMaxPartials, status)) m = fmaxf(m, qo.partials_in[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) red[warp] = m;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1 + kWorkers);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, kWorkers);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_a);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Abort ab{abort_flag, status};
  const int tiles = (M + ROWS - 1) / ROWS;
  const int items = tiles * parts;   // work item w: row tile w / parts, rank part w % parts
  const int nk = K >> 6;
  float ts = 1.0f;
  if (QUANT) {
    float m = red[0];
    for (int i = 1; i < kThreads / 32; ++i) m = fmaxf(m, red[i]);
    ts = __fdiv_rn(m, 2688.0f);
    if (ts == 0.0f) ts = 1.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *qo.ts_out = ts;
    build_bracket_table(yt, ts);
    __syncthreads();
  }
  // QUANT: B' multiplier, and the power of two u carries when the tensor
  // scales are tiny (u is written below, after ts is known)
  const LoraScale ls = (QUANT && qo.b_chunks > 0) ? lora_scale(qo.lora_k, ts, *qo.ts_w) : LoraScale{1.0f, 1.0f};

  if (warp == 0) {
    if (lane == 0) {
      uint32_t filled = 0, fill_par = 0;
      int st = 0;
      uint32_t ph = 0;
      const uint32_t tx = static_cast<uint32_t>(kXBytes) + static_cast<uint32_t>(pr) * 128u;
      for (int w = blockIdx.x; w < items; w += gridDim.x) {
        const int t = w / parts, rpart = w - t * parts;
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait(&empty[st], ph ^ 1, ab)) goto producer_done;
          uint8_t* base = smem + st * stage_bytes;
          mbar_arrive_expect_tx(&full[st], tx);
#pragma unroll
          for (int hh = 0; hh < ROWS / 128; ++hh)
            tma_load_2d(base + hh * 16384, &tm_x, &full[st], kc * 64, t * ROWS + hh * 128);
          for (int rb = 0; rb < pr; rb += a_box_rows)
            tma_load_2d(base + kXBytes + rb * 128, &tm_a, &full[st], kc * 64, rpart * pr + rb);
          filled |= 1u << st;
          fill_par = (fill_par & ~(1u << st)) | (ph << st);
          if (++st == stages) { st = 0; ph ^= 1; }
        }
      }
    producer_done:
      for (int s = 0; s < stages; ++s)
        if (filled & (1u << s)) mbar_drain(&full[s], (fill_par >> s) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int st = 0;
      uint32_t ph = 0, acc_ph = 0;
      const int n_pieces = pr <= 256 ? 1 : 2;
      const int piece_n = pr / n_pieces;
      const uint32_t idesc = idesc_bf16(static_cast<uint32_t>(piece_n));
      for (int w = blockIdx.x; w < items; w += gridDim.x) {
        if (!mbar_wait(tmem_empty, acc_ph ^ 1, ab)) goto mma_done;
        tc_fence_after();
        for (int kc = 0; kc < nk; ++kc) {
          if (!mbar_wait(&full[st], ph, ab)) goto mma_done;
          tc_fence_after();
          const uint32_t xa = smem_u32(smem + st * stage_bytes);
          const uint32_t aa = xa + static_cast<uint32_t>(kXBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int hh = 0; hh < ROWS / 128; ++hh) {   // rows 128 hh ..: accumulator at column hh * pr
              const uint64_t adesc = sdesc_kmajor_sw128(xa + hh * 16384 + kk * 32);
              for (int p = 0; p < n_pieces; ++p) {
                const uint64_t bdesc = sdesc_kmajor_sw128(aa + p * piece_n * 128 + kk * 32);
                mma_bf16(tmem + hh * pr + p * piece_n, adesc, bdesc, idesc, (kc | kk) != 0);
              }
            }
          }
          tc_commit(&empty[st]);
          if (++st == stages) { st = 0; ph ^= 1; }
        }
        tc_commit(tmem_full);
        acc_ph ^= 1;
      }
    mma_done:
      tc_commit(drain_bar);
      mbar_drain(drain_bar, 0);
    }
  } else {
    // amax + epilogue warps.  TMEM access: warp w reads lanes 32 * (w % 4) ..;
    // the warps of a lane quarter take interleaved 32-column chunks of u.
    const int aw = warp - 2;                 // 0 .. kWorkers - 1
    const int at = threadIdx.x - 64;         // amax thread
    const int ch = at & 7;                   // 16-byte column chunk
    const int rb = at >> 3;                  // first row
    const int q = warp & 3;
    const int cpart = aw >> 2;               // 0 .. kWorkers / 4 - 1: this warp's u column chunks
    constexpr int kCParts = kWorkers / 4;
    float m = 0.0f;
    int st = 0;
    uint32_t ph = 0, acc_ph = 0;
    // QUANT: block qj of rows qr + kQuantRowStep h of each stage; its 16
    // scales are loaded one stage ahead
    const int qj = at & 3, qr = at >> 2;
    const QuantCtx qc = make_quant_ctx(ts, yt);
    constexpr int kQuantRowStep = 8 * kWorkers;        // rows covered by the workers at once
    constexpr int kQuantRows = ROWS / kQuantRowStep;   // rows of a tile per thread
    static_assert(kQuantRows * kQuantRowStep == ROWS, "rows of a tile per quantising thread");
    constexpr int kRowStride = 32 * kWorkers / 8;      // amax: rows between a thread's rows
    static_assert(ROWS % kRowStride == 0, "rows of a tile per amax thread");
    float qs_next[16];
    if (QUANT) load_scale16(pqs, qj, qs_next);
    // The per-channel scales of a stage are loaded two stages ahead: the
    // shared-memory ring leaves little L1, so these loads go to L2.
    float s0[8], s1[8];
    if (!QUANT) {
      load_scale8(pqs, ch, s0);
      load_scale8(pqs, (nk > 1 ? 1 : 0) * 8 + ch, s1);
    }
    for (int w = blockIdx.x; w < items; w += gridDim.x) {
      const int t = w / parts, rpart = w - t * parts;
      const bool first = rpart == 0;   // the amax / quantisation of a tile is done by its first rank part only
      // QUANT: row h's scale byte of the stage's first 64 columns at sf_row[h]
      // (the native layout: 512-byte atoms of 128 rows x 64 columns ordered
      // [rows / 128][K / 64], (r % 32) * 16 + (r % 128 / 32) * 4 + j inside;
      // null past the scales' 128-row padding), its codes at code_row[h]
      // (null past M: rows >= M get no codes)
      uint8_t* sf_row[kQuantRows];
      uint2* code_row[kQuantRows];
      if (QUANT) {
#pragma unroll
        for (int h = 0; h < kQuantRows; ++h) {
          const int row = t * ROWS + qr + kQuantRowStep * h;
          sf_row[h] = row < ((M + 127) & ~127)
                          ? qo.scales + static_cast<int64_t>(row >> 7) * (K >> 6) * 512 + (row & 31) * 16 +
                                ((row & 127) >> 5) * 4 + qj
                          : nullptr;
          code_row[h] = row < M ? qo.codes + static_cast<int64_t>(row) * (K >> 4) + qj : nullptr;
        }
      }
      // unrolled by two, which lets the scale prefetch of one stage and the
      // work of the next interleave (measured: -8 us per block)
#pragma unroll 2
      for (int kc = 0; kc < nk; ++kc) {
        if (QUANT) {
          float qs[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) qs[i] = qs_next[i];
          const int kn = kc + 1 < nk ? kc + 1 : 0;
          load_scale16(pqs, 4 * kn + qj, qs_next);
          if (!mbar_wait(&full[st], ph, ab)) goto amax_done;
          const uint8_t* tile = smem + st * stage_bytes;
#pragma unroll
          for (int h = 0; h < kQuantRows; ++h) {
            const int r = qr + kQuantRowStep * h;
            const uint4 w0 = *reinterpret_cast<const uint4*>(tile + r * 128 + (((2 * qj) ^ (r & 7)) << 4));
            const uint4 w1 = *reinterpret_cast<const uint4*>(tile + r * 128 + (((2 * qj + 1) ^ (r & 7)) << 4));
            // rows >= M were filled with zeros by the TMA load: scale 0, no codes
            if (first && sf_row[h] && in_bounds(4 * kc + 3 < (K >> 4), status))
              quant_block(qc, code_row[h] ? code_row[h] + 4 * kc : nullptr, sf_row[h] + kc * 512, w0, w1, qs);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);
          if (++st == stages) { st = 0; ph ^= 1; }
          continue;
        }
        float s[8], s2[8];
        int k2 = kc + 2;
        while (k2 >= nk) k2 -= nk;
        load_scale8(pqs, k2 * 8 + ch, s2);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          s[i] = s0[i];
          s0[i] = s1[i];
          s1[i] = s2[i];
        }
        if (!mbar_wait(&full[st], ph, ab)) goto amax_done;
        if (first) {
          const uint8_t* tile = smem + st * stage_bytes;
          ColMax8 cm;
#pragma unroll
          for (int i = 0; i < ROWS / kRowStride; ++i) {
            const int r = rb + kRowStride * i;
            cm.add(*reinterpret_cast<const uint4*>(tile + r * 128 + ((ch ^ (r & 7)) << 4)));
          }
          m = fmaxf(m, cm.scaled_max(s));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (++st == stages) { st = 0; ph ^= 1; }
      }
      // epilogue: u[row, :] = bf16(acc * u_mul) (u_mul = 1 but for tiny tensor scales)
      if (!mbar_wait(tmem_full, acc_ph, ab)) goto amax_done;
      tc_fence_after();
#pragma unroll 1
      for (int hh = 0; hh < ROWS / 128; ++hh) {   // rows 128 hh ..: accumulator at column hh * pr
        const int row = t * ROWS + hh * 128 + 32 * q + lane;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + hh * pr;
        for (int c0 = 32 * cpart; c0 < pr; c0 += 32 * kCParts) {
          uint32_t r[32];
          tmem_ld32(taddr + c0, r);
          tmem_ld_wait();
          const int nvec = (pr - c0) >= 32 ? 4 : 2;
          if (row < M && in_bounds(row >= 0 && rpart * pr + c0 + 8 * nvec <= rank, status)) {
            uint4* dst = reinterpret_cast<uint4*>(u + static_cast<int64_t>(row) * rank + rpart * pr + c0);
            for (int v = 0; v < nvec; ++v) {
              float f[8];
#pragma unroll
              for (int i = 0; i < 8; ++i)
                f[i] = QUANT ? __fmul_rn(__uint_as_float(r[8 * v + i]), ls.u_mul) : __uint_as_float(r[8 * v + i]);
              uint4 o;
              o.x = pack_bf16x2(f[0], f[1]);
              o.y = pack_bf16x2(f[2], f[3]);
              o.z = pack_bf16x2(f[4], f[5]);
              o.w = pack_bf16x2(f[6], f[7]);
              dst[v] = o;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty);
      acc_ph ^= 1;
    }
    if (QUANT && qo.b_chunks > 0)   // B' only: u already carries its power of two
      scale_lora_operands(LoraScale{ls.c, 1.0f}, qo.b_src, qo.b_dst, qo.b_chunks, nullptr, 0,
                          static_cast<int64_t>(blockIdx.x) * (32 * kWorkers) + at,
                          static_cast<int64_t>(gridDim.x) * (32 * kWorkers));
  amax_done:
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (!QUANT && lane == 0) red[aw] = m;
  }
  tc_fence_before();
  __syncthreads();
  if (!QUANT && threadIdx.x == 0 && in_bounds(blockIdx.x < static_cast<unsigned>(kMaxPartials), status)) {
    float m = red[0];
    for (int i = 1; i < kWorkers; ++i) m = fmaxf(m, red[i]);
    partials[blockIdx.x] = m;
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// --------------------------------------------------------------- launchers
RowPlan plan_rows(int64_t M, int64_t K, int sm_count) {
  const int64_t kc = K / 8;
  int64_t target = static_cast<int64_t>(sm_count) * 2048;
  int64_t rows_step = target / kc;
  if (rows_step < 1) rows_step = 1;
  const int64_t mpad = ((M + 127) / 128) * 128;
  if (rows_step > mpad) rows_step = mpad;
  int64_t blocks = (kc * rows_step + kQuantThreads - 1) / kQuantThreads;
  while (blocks > kMaxPartials && rows_step > 1) {
    rows_step /= 2;
    blocks = (kc * rows_step + kQuantThreads - 1) / kQuantThreads;
  }
  return RowPlan{static_cast<int>(blocks), static_cast<int>(rows_step)};
}

cudaError_t launch_amax(const void* x, int M, int K, const float* pqs, float* partials, const RowPlan& p,
                        int* count_out, uint32_t* status, cudaStream_t st) {
  trace_launch("k_amax", p.blocks, 1, kQuantThreads, 0, "M=%d K=%d rows_step=%d", M, K, p.rows_step);
  k_amax<<<p.blocks, kQuantThreads, 0, st>>>(static_cast<const uint4*>(x), M, K / 8, pqs, partials, p.rows_step,
                                             count_out, status);
  return cudaGetLastError();
}

// One wave of k_quant: as many 256-thread blocks as fit on the device at once;
// each thread owns one 16-element block column of K / 16.
static RowPlan plan_quant(int64_t M, int64_t K, int sm_count) {
  static int per_sm = 0;
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_quant, kQuantThreads, 0) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 4;
    }
    per_sm = n;
  }
  const int64_t kb = K / 16;
  const int64_t threads = static_cast<int64_t>(sm_count) * per_sm * kQuantThreads;
  int64_t rows_step = threads / kb;
  if (rows_step < 1) rows_step = 1;
  const int64_t mpad = ((M + 127) / 128) * 128;
  if (rows_step > mpad) rows_step = mpad;
  const int64_t blocks = (kb * rows_step + kQuantThreads - 1) / kQuantThreads;
  return RowPlan{static_cast<int>(blocks), static_cast<int>(rows_step)};
}

cudaError_t launch_quant(const void* x, int M, int K, const float* pqs, const float* partials, int nparts,
                         const int* nparts_dev, void* codes, void* scales, float* ts_out, const RowPlan& /*amax plan*/,
                         const void* b_src, void* b_dst, int64_t b_elems, float lora_k, const float* ts_w,
                         void* u, int64_t u_elems, uint32_t* status, int sm_count, cudaStream_t st) {
  const int Mpad = ((M + 127) / 128) * 128;
  const RowPlan p = plan_quant(M, K, sm_count);
  trace_launch("k_quant", p.blocks, 1, kQuantThreads, 0, "M=%d K=%d rows_step=%d lora_b=%lld", M, K, p.rows_step,
               static_cast<long long>(b_elems));
  k_quant<<<p.blocks, kQuantThreads, 0, st>>>(
      static_cast<const uint4*>(x), M, Mpad, K, pqs, partials, nparts, nparts_dev, static_cast<uint2*>(codes),
      static_cast<uint8_t*>(scales), ts_out, p.rows_step, static_cast<const uint4*>(b_src),
      static_cast<uint4*>(b_dst), b_elems / 8, lora_k, ts_w, static_cast<uint4*>(u), u_elems / 8, status);
  return cudaGetLastError();
}

// Rank parts of the LoRA-down passes: a row tile's u = A(x) is split into
// `parts` column ranges computed by separate CTAs, each staging the same x
// tile (each element's sum over K runs as before, so u is the same bit for
// bit), so that small M still fills the GPU.  Only below half a tile per SM:
// each part re-reads x, which costs more than it gains once the tiles alone
// come near one per SM (measured at M = 16384, 128 tiles: 0.114 -> 0.133 ms
// for rank 384 in two parts).  Then the smallest split whose work items
// reach one per SM, each part a multiple of 16 columns and at least 32.
int lora_rank_parts(int64_t M, int rank, int sm_count) {
  const int64_t tiles = (M + 127) / 128;
  if (2 * tiles > sm_count) return 1;
  int best = 1;
  for (int p : {1, 2, 3, 4, 6}) {
    if (rank % p != 0 || (rank / p) % 16 != 0 || rank / p < 32) continue;
    best = p;
    if (tiles * p >= sm_count) break;
  }
  return best;
}
int lora_a_box_rows(int rank, int parts) {
  const int pr = rank / parts;
  return pr <= 256 ? pr : pr / 2;
}

template <bool QUANT, int ROWS>
static cudaError_t launch_lora_pass(const CUtensorMap& tm_x, const CUtensorMap& tm_a, int M, int K, int rank,
                                    int parts, int a_box_rows, const float* pqs, float* partials, void* u,
                                    uint32_t* status, int sm_count, const QuantPassOut& qo, int* grid_out,
                                    cudaStream_t st) {
  const int pr = rank / parts;
  const int stage_bytes = ROWS * 128 + pr * 128;
  constexpr int kSmemLimit = 232448;     // per CTA, one CTA per SM
  constexpr int kSmemPerSm = 233472;     // shared memory of an SM (228 KB), 1 KB of it reserved per CTA
  const int tail = 256 + (QUANT ? 2048 : 0);   // barriers, flags, partial maxima (+ bracket table)
  int tmem_cols = 32;
  while (tmem_cols < (ROWS / 128) * pr) tmem_cols <<= 1;
  // 128-row tiles: two CTAs per SM when their accumulators fit TMEM together
  // and each gets a ring of at least 3 stages; else (and for 256-row tiles)
  // one CTA with up to 8 stages
  const int two_stages = (kSmemPerSm / 2 - 1024 - 1024 - tail) / stage_bytes;
  const bool two = ROWS == 128 && (QUANT || kLoraAmaxTwoCtas) && 2 * tmem_cols <= 512 && two_stages >= 3;
  int stages = two ? two_stages : (kSmemLimit - 1024 - tail) / stage_bytes;
  if (stages > 8) stages = 8;
  if (stages < 2) return cudaErrorInvalidValue;
  const int smem = stages * stage_bytes + 1024 + tail;
  const int items = (M + ROWS - 1) / ROWS * parts;
  const int slots = (two ? 2 : 1) * sm_count;
  int grid = items < slots ? items : slots;
  if (grid > kMaxPartials) grid = kMaxPartials;
  auto kern = k_amax_lora<QUANT, ROWS>;
  constexpr int kThreads = lora_threads<QUANT, ROWS>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  trace_launch(QUANT ? "k_amax_lora<quant>" : "k_amax_lora<amax>", grid, 1, kThreads, smem,
               "M=%d K=%d rank=%d rank_parts=%d tile_rows=%d stages=%d ctas_per_sm=%d tmem_cols=%d", M, K, rank,
               parts, ROWS, stages, two ? 2 : 1, tmem_cols);
  kern<<<grid, kThreads, smem, st>>>(tm_x, tm_a, M, K, rank, parts, a_box_rows, pqs, partials,
                                     static_cast<__nv_bfloat16*>(u), status, stages, tmem_cols, qo);
  if (grid_out) *grid_out = grid;
  return cudaGetLastError();
}

// Tile rows of the LoRA-down passes.  The quantising pass takes 256 when two
// 128-row accumulators of rank / parts columns fit TMEM and the 256-row tiles
// still give about one per SM (down at S = 37726: 358 -> 284 us); the amax
// pass keeps 128 (its two CTAs per SM already stream x at 86 % of HBM, and
// 256-row tiles measured 66 -> 76 us there).
static int lora_tile_rows(bool quant, int64_t M, int rank, int parts, int sm_count) {
  const int64_t tiles256 = (M + 255) / 256 * parts;
  return (quant && rank / parts <= 128 && 4 * tiles256 >= 3 * int64_t(sm_count)) ? 256 : 128;
}

cudaError_t launch_amax_lora(const CUtensorMap& tm_x, const CUtensorMap& tm_a, int M, int K, int rank, int parts,
                             int a_box_rows, const float* pqs, float* partials, void* u, uint32_t* status,
                             int sm_count, int* nparts, cudaStream_t st) {
  QuantPassOut qo{};
  return launch_lora_pass<false, 128>(tm_x, tm_a, M, K, rank, parts, a_box_rows, pqs, partials, u, status, sm_count,
                                      qo, nparts, st);
}

cudaError_t launch_quant_lora(const CUtensorMap& tm_x, const CUtensorMap& tm_a, int M, int K, int rank, int parts,
                              int a_box_rows, const float* pqs, const float* partials, const int* nparts_dev,
                              void* codes, void* scales, float* ts_out, void* u, uint32_t* status,
                              const void* b_src, void* b_dst, int64_t b_elems, float lora_k, const float* ts_w,
                              int sm_count, cudaStream_t st) {
  QuantPassOut qo{partials, nparts_dev, static_cast<uint2*>(codes), static_cast<uint8_t*>(scales), ts_out,
                  static_cast<const uint4*>(b_src), static_cast<uint4*>(b_dst), b_elems / 8, lora_k, ts_w};
  if (lora_tile_rows(true, M, rank, parts, sm_count) == 256)
    return launch_lora_pass<true, 256>(tm_x, tm_a, M, K, rank, parts, a_box_rows, pqs, nullptr, u, status, sm_count,
                                       qo, nullptr, st);
  return launch_lora_pass<true, 128>(tm_x, tm_a, M, K, rank, parts, a_box_rows, pqs, nullptr, u, status, sm_count,
                                     qo, nullptr, st);
}

}  // namespace h3lin
