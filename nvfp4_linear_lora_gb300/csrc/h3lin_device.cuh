// Device-side building blocks for the sm_103a kernels: mbarriers with bounded
// waits, TMA (tiled tensor and plain bulk copies), and tcgen05 (TMEM
// allocation, UMMA descriptors, MMA issue, TMEM loads).  Inline PTX only.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "h3lin_internal.h"

namespace h3lin {

// ------------------------------------------------------------------ basics
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31; }
__device__ __forceinline__ uint32_t warp_id() { return threadIdx.x >> 5; }

// ------------------------------------------------------------ error record
// Kernels never trap.  A wait that exceeds kWaitLimitCycles records
// H3LIN_E_TIMEOUT in the workspace status word (first error wins) and raises
// the CTA-wide abort flag; every other waiter of the CTA then gives up too.
constexpr long long kWaitLimitCycles = 1ll << 31;  // ~1 s at 2 GHz

struct Abort {
  int* cta_flag;         // shared memory
  uint32_t* status;      // global, workspace status word
  __device__ __forceinline__ bool raised() const {
    return *reinterpret_cast<volatile int*>(cta_flag) != 0;
  }
  __device__ __forceinline__ void raise(uint32_t code) const {
    atomicCAS(status, 0u, code);
    *reinterpret_cast<volatile int*>(cta_flag) = 1;
  }
};

// ------------------------------------------------------------- bounds build
// Built with -DH3LIN_BOUNDS (libh3lin_bounds.so), the kernels check the
// index of every plain global access whose extent no TMA tensor map enforces:
// an index outside its buffer records H3LIN_E_BOUNDS in the status word
// (first error wins) and the access is skipped; nothing traps.  In the normal
// build the check is the constant true and compiles away.
#ifdef H3LIN_BOUNDS
__device__ __forceinline__ bool in_bounds(bool ok, uint32_t* status) {
  if (!ok && status != nullptr) atomicCAS(status, 0u, static_cast<uint32_t>(H3LIN_E_BOUNDS));
  return ok;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(bool, uint32_t*) { return true; }
#endif

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test: has the phase of parity `parity` completed?  Never
// suspends the thread (for a thread that must keep issuing work).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of parity `parity` to complete.  Returns false
// (without completing) when the CTA aborted or `limit` cycles expired.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const Abort& ab,
                                          long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (ab.raised()) return false;
    if (clock64() - t0 > limit) {
      ab.raise(H3LIN_E_TIMEOUT);
      return false;
    }
  }
  return true;
}
// Teardown variant: bounded, ignores the abort flag (used to drain copies
// still in flight before the CTA exits).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) return;
  }
}

// --------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2-D tiled load; x = innermost coordinate (elements), y = row.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// Plain bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {  // whole warp
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive (once) on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Shared-memory matrix descriptor, K-major operand in the canonical
// 128-byte-swizzled layout: rows of 128 bytes, 8-row atoms of 1024 bytes
// (SBO = 1024), atom base 1024-aligned.  Advancing along K inside the
// 128-byte row is done by adding the byte offset to the start address.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address  [0,14)
  d |= static_cast<uint64_t>(1) << 16;                    // LBO (unused)   [16,30)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;            // SBO            [32,46)
  d |= static_cast<uint64_t>(1) << 46;                    // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
  return d;
}
// Descriptor of a 32-row x 16-byte block-scale atom chunk (no swizzle, core
// matrices of 8 rows x 16 bytes stacked 128 bytes apart) for tcgen05.cp.
__device__ __forceinline__ uint64_t sdesc_sf_atom(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(128 >> 4) << 32;             // SBO = 128 bytes
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptors (dense, K-major A and B, M = 128).
// kind::f16 with BF16 inputs and FP32 accumulation.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t n) {
  return (1u << 4)              // D format: F32
         | (1u << 7)            // A format: BF16
         | (1u << 10)           // B format: BF16
         | ((n >> 3) << 17)     // N / 8
         | ((128u >> 4) << 24); // M / 16
}
// kind::mxf4nvf4 with E2M1 inputs and UE4M3 block scales (16 elements each).
__host__ __device__ constexpr uint32_t idesc_nvfp4(uint32_t n) {
  return (1u << 7)              // A format: E2M1
         | (1u << 10)           // B format: E2M1
         | ((n >> 3) << 17)     // N / 8
         | (0u << 23)           // scale format: UE4M3
         | ((128u >> 4) << 24); // M / 16
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_nvfp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Copy one 512-byte scale atom (32 rows x 128 bits, replicated to the four
// 32-lane quarters) from shared memory to 4 TMEM columns.
__device__ __forceinline__ void tmem_cp_sf_atom(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Load 32 consecutive FP32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 16 TMEM lanes, two column groups: thread t reads lane L + t % 16 (L = the
// lane field of taddr, a multiple of 16 inside the warp's 32-lane quarter) and
// the columns C + (t / 16) * SPLIT .. + 31 (x32) or .. + 15 (x16), C = the
// column field of taddr.
template <int SPLIT>
__device__ __forceinline__ void tmem_ld16x2_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32], %33;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr), "n"(SPLIT));
}
template <int SPLIT>
__device__ __forceinline__ void tmem_ld16x2_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16], %17;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr), "n"(SPLIT));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// --------------------------------------------------------------- numerics
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// bf16 pair (as packed in memory: element 0 in the low half) -> two floats.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// E4M3, round to nearest even, saturate to +-448.
__device__ __forceinline__ uint32_t e4m3_rn_satfinite(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}
__device__ __forceinline__ float e4m3_to_float(uint32_t b) {
  uint32_t h2;
  uint16_t in = static_cast<uint16_t>(b);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}
// Eight floats -> eight E2M1 codes (round to nearest even, saturate to 6,
// sign kept), element i in bits [4i, 4i+4).
__device__ __forceinline__ uint32_t e2m1x8(const float (&q)[8]) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return out;
}

// (r0, r1) = (a0 * b0, a1 * b1), each rounded to nearest even: one packed
// f32x2 multiply on sm_100+ (the same results as two __fmul_rn).
__device__ __forceinline__ void fmul2_rn(float a0, float a1, float b0, float b1, float& r0, float& r1) {
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// (r0, r1) = (fma(a0, b0, c0), fma(a1, b1, c1)), each rounded once to
// nearest even: one packed f32x2 fma (the same results as two fmaf).
__device__ __forceinline__ void ffma2_rn(float a0, float a1, float b0, float b1, float c0, float c1, float& r0,
                                         float& r1) {
  asm("{\n\t.reg .b64 a, b, c, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// ------------------------------------------- LoRA operand and epilogue scales
// The GEMM accumulates the base products and u.B' in one FP32 tile and
// multiplies the sum by ts_x * ts_w in its epilogue, so B' = B * c with
// c = lora_k / (ts_x * ts_w).  For tiny tensor scales c leaves the bf16 range
// although the LoRA product itself is representable; then a power of two 2^E
// moves from B' to u (u' = u * 2^E exactly, B' = B * c * 2^-E: the same
// product, both operands in range).  E = 0, and c = fl(lora_k / fl(ts_x ts_w))
// bit for bit, whenever those values are normal floats with c below 2^64.
struct LoraScale {
  float c;       // multiplier of B
  float u_mul;   // 2^E, multiplier of u (1 normally)
};
__device__ __forceinline__ LoraScale lora_scale(float lora_k, float ts_x, float ts_w) {
  const int ex = ilogbf(ts_x), ew = ilogbf(ts_w);
  const float m = __fmul_rn(scalbnf(ts_x, -ex), scalbnf(ts_w, -ew));   // in [1, 4)
  const float cm = __fdiv_rn(lora_k, m);
  const int e = -(ex + ew);                                            // c = cm * 2^e
  int E = 0;
  if (cm != 0.0f) E = min(max(e + ilogbf(cm) - 64, 0), 126);
  return LoraScale{scalbnf(cm, e - E), scalbnf(1.0f, E)};
}

// The epilogue's y = ts_x * ts_w * acc as fl(fl(acc * a) * b): (a, b) =
// (fl(ts_x ts_w), 1) while that product is at least 2^-100; below, a is the
// product scaled up by 2^k (exactly) and b = 2^-k, so outputs in the normal
// float range keep full precision however small the two tensor scales are.
struct EpiScale {
  float a, b;
};
__device__ __forceinline__ EpiScale epi_scale(float ts_x, float ts_w) {
  const float p = __fmul_rn(ts_x, ts_w);
  if (p >= 0x1p-100f) return EpiScale{p, 1.0f};
  const int ex = ilogbf(ts_x), ew = ilogbf(ts_w);
  const float m = __fmul_rn(scalbnf(ts_x, -ex), scalbnf(ts_w, -ew));   // in [1, 4); product = m * 2^(ex + ew)
  const int k = min(-(ex + ew), 126);
  return EpiScale{scalbnf(m, ex + ew + k), scalbnf(1.0f, -k)};
}

// Byte offset of the scale of (row, 16-block j) in the native scale layout.
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t row, int64_t j, int64_t K) {
  const int64_t atom = (row >> 7) * (K >> 6) + (j >> 2);
  const int64_t r = row & 127;
  return atom * 512 + (r & 31) * 16 + (r >> 5) * 4 + (j & 3);
}

}  // namespace h3lin

// ------------------------------------------------------ CTA pairs (cluster of 2)
// A CTA pair shares one tcgen05 MMA of M = 256 (cta_group::2): each CTA holds
// its own 128 rows of A and 128 of the 256 B rows; the leader (cluster rank 0)
// issues the MMAs, and every pair-wide tcgen05 op uses .cta_group::2.
namespace h3lin {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Shared-memory address of the same object in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t o;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(o) : "r"(smem_u32(p)), "r"(rank));
  return o;
}
// Arrive on a barrier of any CTA of the cluster with the default (CTA-scope)
// release.  Enough for handing a TMEM accumulator back to the pair leader
// (the tcgen05 loads have completed before the arrive); a cluster-scope
// release here costs over a thousand cycles per arrival.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 2-D tiled load into this CTA's shared memory whose completion is counted on
// the pair leader's barrier (`leader_bar` from cluster_addr(bar, 0)).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t leader_bar, int32_t x,
                                                 int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(leader_bar)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {  // one warp in each CTA
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Arrive on the barrier at the same offset in both CTAs of the pair.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}
// Arrive on this CTA's barrier when this thread's pair-wide tcgen05 ops complete.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// One scale atom from each CTA's shared memory into its own TMEM (4 columns).
__device__ __forceinline__ void tmem_cp_sf_atom_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__host__ __device__ constexpr uint32_t idesc_nvfp4_m256(uint32_t n) {
  return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | (0u << 23) | ((256u >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16_m256(uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((256u >> 4) << 24);
}
__device__ __forceinline__ void mma_nvfp4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

}  // namespace h3lin

namespace h3lin {
// ---------------------------------------------------------------- TMA store
// Make this thread's generic-proxy shared-memory writes visible to the TMA.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 2-D tiled store shared -> global (rows/columns outside the tensor are clipped).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until every committed bulk store of this thread is complete.
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
}  // namespace h3lin
