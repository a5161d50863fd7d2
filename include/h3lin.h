/*
 * h3lin — dynamic-LoRA NVFP4 linear for GB300 (sm_103a): the C ABI.
 *
 * The operation (TURBO.md, h3-blackwell-runtime, section "Implementation"):
 *
 *     out = NVFP4_base(x * pre_quant_scale) + strength * (alpha / rank) * B(A(x))
 *
 * The NVFP4 base branch quantises the pre-scaled activation at run time
 * ("dynamic NVFP4 activation quantization", MiniMax-H3 Ultra Fast README,
 * section "Kernel path", item 1) and multiplies it with the packed NVFP4
 * weight on the FP4 tensor cores.  The BF16 LoRA branch receives the ORIGINAL
 * activation and is never merged into the packed weight (TURBO.md,
 * "Implementation").  The fused gate/up projection applies silu(gate) * up in
 * place (Ultra Fast README, table "Active optimization stack", row MLP).
 *
 * NVFP4 encoding used throughout (the format's public definition):
 *   codes   E2M1, two per byte, element 2j in bits 0-3, element 2j+1 in 4-7,
 *           row-major [rows, K/2];
 *   scales  one E4M3 scale per 16 elements along K, stored in the NATIVE
 *           layout: 512-byte atoms covering 128 rows x 64 columns, atoms
 *           ordered [rows/128][K/64]; inside an atom the scale of row r,
 *           16-block j sits at byte (r % 32) * 16 + (r / 32) * 4 + j
 *           (rows padded to a multiple of 128; padded rows hold scale 0);
 *   tensor  one FP32 scale per tensor, amax / 2688 (1 when that is zero),
 *           kept in device memory.
 *
 * Conventions (all entry points):
 *   - Pointers marked "device" are CUDA device pointers; the library never
 *     allocates or frees memory.  The caller owns every buffer.
 *   - Work is enqueued asynchronously on `stream` (0 = legacy default stream);
 *     no call synchronises except h3lin_read_status.
 *   - Arguments are validated on the host BEFORE anything is enqueued; on any
 *     error the call returns a non-zero status and enqueues nothing.
 *   - Calls keep no state between them (no caches keyed by pointer); the
 *     adapter is chosen per call.  A workspace must not be used by two calls
 *     that may run concurrently.
 *   - Kernels never trap: every device-side wait is bounded; on expiry the
 *     kernel records H3LIN_E_TIMEOUT in the workspace status word and returns.
 *
 * Shape rules: M >= 0; K % 64 == 0; N % 128 == 0 (SiLU*up: N % 256 == 0);
 * an activation of M = 0 rows is a valid call of h3lin_forward (and its two
 * stages) or h3lin_quantize_act that enqueues nothing and touches no buffer
 * (x, out, codes, scales and the workspace may then be NULL); a weight needs
 * N >= 1;
 * rank % 16 == 0 and 16 <= rank <= 256, or rank % 32 == 0 and rank <= 512;
 * x, codes, scales, out, A, B 16-byte aligned; rows and K below 2^31.
 */
#ifndef H3LIN_H
#define H3LIN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define H3LIN_ABI_VERSION 1

typedef int32_t h3lin_status;
#define H3LIN_OK            0
#define H3LIN_E_INVALID     1  /* null pointer, unknown enum, non-finite scalar      */
#define H3LIN_E_SHAPE       2  /* a shape rule above is violated                      */
#define H3LIN_E_ALIGN       3  /* a pointer is not 16-byte aligned                    */
#define H3LIN_E_WORKSPACE   4  /* workspace too small                                 */
#define H3LIN_E_CUDA        5  /* CUDA runtime error while enqueueing / no device     */
#define H3LIN_E_TIMEOUT     6  /* device-side bounded wait expired (device status)    */
#define H3LIN_E_UNSUPPORTED 7  /* device is not compute capability 10.x (tcgen05)     */
#define H3LIN_E_BOUNDS      8  /* (device status, bounds build only) an index left its
                                  buffer; the access was skipped                     */

/* Output element types of h3lin_forward. */
#define H3LIN_OUT_BF16      0  /* bf16, round to nearest even (the model's dtype)         */
#define H3LIN_OUT_F32       1  /* fp32: the epilogue value before the bf16 rounding       */

/* Epilogues of h3lin_forward. */
#define H3LIN_EPI_NONE      0  /* out[M, N] = y                                       */
#define H3LIN_EPI_SILU_MUL  1  /* y = [gate | up] (N = 2 * Nh); out[M, Nh] = silu(gate) * up */

/* A packed NVFP4 weight W[N, K] (as written by h3lin_pack_weight).  POD,
 * caller-owned; all three pointers are device pointers. */
typedef struct {
    const void*  codes;         /* u8 [N, K/2]                                      */
    const void*  scales;        /* u8, native layout, h3lin_scales_bytes(N, K) bytes */
    const float* tensor_scale;  /* 1 float                                           */
    int64_t      N, K;
} h3lin_weight;

/* One resident LoRA adapter for one projection.  POD, caller-owned; A and B
 * are device pointers to row-major bf16. */
typedef struct {
    const void* A;      /* bf16 [rank, K]: down projection, applied to the original x */
    const void* B;      /* bf16 [N, rank]: up projection (gate/up: rows [gate; up])   */
    int32_t     rank;
    float       alpha;  /* the adapter's alpha; the branch is scaled by alpha / rank  */
} h3lin_adapter;

/* ------------------------------------------------------------------ sizes */
/* Bytes of the packed codes / native scales of a [rows, K] NVFP4 tensor
 * (0 when the shape is invalid). */
size_t h3lin_codes_bytes(int64_t rows, int64_t K);
size_t h3lin_scales_bytes(int64_t rows, int64_t K);
/* Workspace of h3lin_quantize_act / h3lin_pack_weight (status word, tensor
 * scale, per-CTA amax partials). */
size_t h3lin_quant_workspace_bytes(void);
/* Workspace of h3lin_forward for activations of up to M rows, in-features K,
 * out-features N (before the epilogue) and adapters of rank up to max_rank
 * (0 = no adapter will ever be passed).  Holds the quantised activation, the
 * LoRA intermediate A(x), the scaled copy of B and the quantiser header. */
size_t h3lin_forward_workspace_bytes(int64_t M, int64_t K, int64_t N, int32_t max_rank);

/* Byte offsets of the regions inside a forward workspace for (M, K, N, rank),
 * for inspection (the kernels' intermediates are not part of the output):
 *   offsets[0]  quantised activation codes, u8 [M, K/2]
 *   offsets[1]  its E4M3 scales, native layout (h3lin_scales_bytes(M, K) bytes)
 *   offsets[2]  u = A(x), bf16 [M, rank] row-major
 *   offsets[3]  B' = bf16(B * strength * (alpha / rank) / (ts_x * ts_w)), [N, rank]
 *   offsets[4]  ts_x, the activation's tensor scale (fp32)
 *   offsets[5]  the device status word (u32)
 * When ts_x * ts_w is so small that B' would leave the bf16 range, a power
 * of two 2^E moves from B' to u (u holds A(x) * 2^E); the product u B', which
 * is all the GEMM uses, is the same.  Returns H3LIN_E_SHAPE for shapes
 * h3lin_forward_workspace_bytes rejects, H3LIN_E_INVALID for a null array. */
h3lin_status h3lin_forward_workspace_regions(int64_t M, int64_t K, int64_t N, int32_t rank, size_t* offsets);

/* Zero the status word and header of a workspace (enqueued on `stream`).
 * Call once after allocating a workspace, and after reading an error. */
h3lin_status h3lin_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* --------------------------------------------------------------- quantiser */
/* Dynamic NVFP4 quantisation of an activation (Ultra Fast README, "Kernel
 * path", item 1) with the checkpoint's per-input-channel pre_quant_scale
 * (TURBO.md, "Implementation"):  v = x * s in FP32, ts = amax|v| / 2688,
 * per-16 E4M3 scale = RNE_sat(blockamax / (6 ts)), codes = RNE_sat(v / (scale ts)),
 * every step in float32 with round to nearest even (the code from the IEEE
 * quotient; a block whose scale * ts is 0 gets all-zero codes).
 *   x                device bf16 [M, K] row-major
 *   pre_quant_scale  device fp32 [K], or NULL for all ones
 *   codes            device u8 [M, K/2]                (output)
 *   scales           device u8 h3lin_scales_bytes(M,K) (output, native layout)
 *   tensor_scale     device fp32 [1]                   (output)
 *   workspace        device, >= h3lin_quant_workspace_bytes(), initialised once
 * Two kernels: an amax pass and the quantise pass. */
h3lin_status h3lin_quantize_act(const void* x, int64_t M, int64_t K, const float* pre_quant_scale,
                                void* codes, void* scales, float* tensor_scale,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* One-time packing of a bf16 weight W[N, K] (row-major) into NVFP4: the same
 * rules with s = 1 (TURBO.md, "Implementation": the packed NVFP4 base).  For
 * the fused gate/up projection pass W = [gate; up] (N = 2 * Nh rows). */
h3lin_status h3lin_pack_weight(const void* w, int64_t N, int64_t K,
                               void* codes, void* scales, float* tensor_scale,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ----------------------------------------------------------------- forward */
/* One projection:  out = NVFP4_base(x * s) + strength * (alpha/rank) * B(A(x)),
 * followed by the epilogue.
 *   x                device bf16 [M, K] row-major (M ragged: no padding needed)
 *   pre_quant_scale  device fp32 [K] or NULL
 *   weight           packed weight with weight->K == K
 *   epilogue         H3LIN_EPI_NONE or H3LIN_EPI_SILU_MUL
 *   adapter          NULL selects the base path; otherwise A [rank, K],
 *                    B [weight->N, rank].  strength == 0 also selects the base
 *                    path, whose output is bit-identical to adapter == NULL
 *                    (TURBO.md, "Validation": disabled exactness).
 *   strength         finite float
 *   out              device [M, N] (SiLU*up: [M, N/2]) of type out_dtype, row-major;
 *                    rows >= M are never touched
 *   out_dtype        H3LIN_OUT_BF16 or H3LIN_OUT_F32 (the bf16 output is exactly
 *                    the round-to-nearest-even of the fp32 one)
 *   workspace        device, >= h3lin_forward_workspace_bytes(M, K, N, rank),
 *                    initialised once with h3lin_workspace_init
 * Kernels (stream order): amax pass (fused with A(x) when the adapter is
 * active), quantise pass (also writes the scaled copy of B), then the FP4
 * GEMM whose TMEM accumulator also receives B(A(x)) before the epilogue. */
h3lin_status h3lin_forward(const void* x, int64_t M, const float* pre_quant_scale,
                           const h3lin_weight* weight, int32_t epilogue,
                           const h3lin_adapter* adapter, float strength,
                           void* out, int32_t out_dtype, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/* The two stages of h3lin_forward, for callers that schedule them apart
 * (h3lin_forward == h3lin_forward_prepare followed by h3lin_forward_gemm on
 * the same stream).  Both must be given the same M, weight, adapter, strength
 * and workspace; the GEMM stage reads what the prepare stage left in the
 * workspace (quantised activation, tensor scale, A(x), scaled B).
 *   prepare  amax pass (+ A(x) when the adapter is active) and quantise pass
 *   gemm     FP4 GEMM + B(A(x)) into the same accumulator + epilogue */
h3lin_status h3lin_forward_prepare(const void* x, int64_t M, const float* pre_quant_scale,
                                   const h3lin_weight* weight, const h3lin_adapter* adapter, float strength,
                                   void* workspace, size_t workspace_bytes, cudaStream_t stream);
h3lin_status h3lin_forward_gemm(int64_t M, const h3lin_weight* weight, int32_t epilogue,
                                const h3lin_adapter* adapter, float strength, void* out, int32_t out_dtype,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------- producer fusion */
/* The MLP's down projection consumes gate/up's SiLU*up output h (MiniMax-H3
 * Ultra Fast README, "Active optimization stack", row "MLP": fused gate/up,
 * in-place SiLU*up, NVFP4 down projection).  TURBO.md (h3-blackwell-runtime,
 * "Implementation") describes the SwiGLU producer packing NVFP4 for the next
 * projection while it emits the exact BF16 LoRA input.  With a dynamic
 * per-tensor scale the packing needs amax(h * s_down) over the whole tensor
 * first, so here the fusion has two phases: the gate/up epilogue reduces the
 * amax while it stores h, and the down projection's prepare stage then makes
 * ONE pass over h (quantise + A(h)) instead of two.  Every value is
 * bit-identical to the unfused chain (h3lin_forward on gate/up, then on down).
 *
 * h3lin_forward_gemm_produce: h3lin_forward_gemm with a bf16 output that is
 * also left, as amax partials, for the consuming projection:
 *   next_pre_quant_scale  the consumer's pre_quant_scale, device fp32 [N_out] or
 *                         NULL (N_out = N, or N/2 for SiLU*up); 16-byte aligned
 *   next_workspace        the consumer's workspace (may be `workspace` itself);
 *                         its header receives the partials; >= header size
 *                         (h3lin_quant_workspace_bytes()), 16-byte aligned
 * The amax is reduced inside the CTA-pair kernel's SiLU*up epilogue; other
 * shapes get an amax pass over the output instead (same result).
 *
 * h3lin_forward_prepare_produced: h3lin_forward_prepare for an x that a
 * producer GEMM wrote, with the same pre_quant_scale and workspace given to
 * that producer, on the same stream after it: no amax pass; with an active
 * adapter a single TMA-staged pass quantises x and computes A(x).  Calling it
 * without such a producer quantises with stale or zero partials (documented
 * misuse, not detected). */
h3lin_status h3lin_forward_gemm_produce(int64_t M, const h3lin_weight* weight, int32_t epilogue,
                                        const h3lin_adapter* adapter, float strength, void* out,
                                        void* workspace, size_t workspace_bytes,
                                        const float* next_pre_quant_scale, void* next_workspace,
                                        size_t next_workspace_bytes, cudaStream_t stream);
h3lin_status h3lin_forward_prepare_produced(const void* x, int64_t M, const float* pre_quant_scale,
                                            const h3lin_weight* weight, const h3lin_adapter* adapter,
                                            float strength, void* workspace, size_t workspace_bytes,
                                            cudaStream_t stream);

/* The whole MLP on one stream and one workspace:
 *   h   = silu(gate(x)) * up(x)   (h3lin_forward with H3LIN_EPI_SILU_MUL, bf16)
 *   out = down(h)                 (h3lin_forward, out_dtype)
 * through the producer fusion above.
 *   x         device bf16 [M, K]
 *   gate_up   packed [gate; up] weight, N_gu rows (N_gu % 256 == 0), K columns
 *   down      packed weight with down->K == N_gu / 2
 *   h         device bf16 [M, N_gu / 2], written (the down projection's input
 *             and its LoRA input)
 *   out       device [M, down->N] of out_dtype
 *   workspace >= h3lin_mlp_workspace_bytes(M, K, N_gu, down->N, max rank)
 * Each pre_quant_scale / adapter / strength as for h3lin_forward; M == 0 is
 * a no-op.  Errors are those of h3lin_forward, checked for both projections
 * before anything is enqueued, plus H3LIN_E_SHAPE when down->K != N_gu / 2. */
size_t h3lin_mlp_workspace_bytes(int64_t M, int64_t K, int64_t N_gate_up, int64_t N_down, int32_t max_rank);
h3lin_status h3lin_mlp_forward(const void* x, int64_t M,
                               const float* gate_up_pre_quant_scale, const h3lin_weight* gate_up,
                               const h3lin_adapter* gate_up_adapter, float gate_up_strength,
                               const float* down_pre_quant_scale, const h3lin_weight* down,
                               const h3lin_adapter* down_adapter, float down_strength,
                               void* h, void* out, int32_t out_dtype,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------ merged-LoRA weights */
/* Comparison mode of the dynamic path: the LoRA update folded into the
 * weight before it is packed (MiniMax-H3 Turbo — one file, no Python, "What
 * the conversion did", list "The rest.", item "Backbone": the LoRA update is
 * merged before quantizing).
 *
 *   w_out[n, k] = bf16_rn( w[n, k] + strength * (alpha / rank) * (sum_j B[n, j] * A[j, k]) / s[k] )
 *
 * with FP32 fused multiply-adds over j in ascending order and one rounding to
 * bf16 at the end.  s is the pre_quant_scale the forward will be called with
 * (1 when NULL): the base branch quantises x * s while the LoRA branch sees x
 * (TURBO.md, h3-blackwell-runtime, "Implementation"), so the folded update is
 * divided by s.  Pack the result with h3lin_pack_weight and run
 * h3lin_forward with adapter == NULL: that forward costs only the base path,
 * the speed bound of the dynamic one, at the price of re-packing the weight
 * for every adapter or strength.
 *   w        device bf16 [N, K], row-major; 8-byte aligned
 *   pre_quant_scale  device fp32 [K] or NULL; 16-byte aligned
 *   adapter  the adapter (A bf16 [rank, K], B bf16 [N, rank]); rank rule as
 *            for h3lin_forward
 *   w_out    device bf16 [N, K], 8-byte aligned; may equal w (in place)
 * K must be a multiple of 64.  Errors: H3LIN_E_INVALID (null pointers,
 * non-finite alpha or strength), H3LIN_E_SHAPE (N, K or rank),
 * H3LIN_E_ALIGN, H3LIN_E_UNSUPPORTED, H3LIN_E_CUDA; nothing is enqueued on
 * error.  Allocates nothing. */
h3lin_status h3lin_merge_lora(const void* w, int64_t N, int64_t K, const float* pre_quant_scale,
                              const h3lin_adapter* adapter, float strength, void* w_out, cudaStream_t stream);

/* ------------------------------------------------ modulation producer */
/* The input of the QKV and gate/up projections: the residual stream
 * normalised and modulated by the AdaLN table, one table row per distinct
 * timestep gathered segment-wise over the packed sequence (MiniMax-H3 Ultra
 * Fast README, "Active optimization stack", row "AdaLN"), emitted as the
 * exact BF16 LoRA input while the NVFP4 packing's amax is reduced on the way
 * (TURBO.md, h3-blackwell-runtime, "Implementation": modulation producer):
 *
 *   y     = (x - mean) / sqrt(var + eps)   per row over K, population variance, fp32
 *   x_mod = bf16(y * (1 + scale[t]) + shift[t]),  t = row_table[row]
 *
 * and, in the consuming projection's workspace, the amax partials of
 * |x_mod * next_pre_quant_scale| that h3lin_forward_prepare_produced reads
 * (one pass over x_mod instead of two; the result is bit-identical to
 * h3lin_forward on x_mod).
 *   x          device bf16 [M, K], 16-byte aligned
 *   table      device fp32 [table_rows, 2, K]: (shift, scale) per row, 16-byte aligned
 *   row_table  device int32 [M]: table row of every row; an entry outside
 *              [0, table_rows) records H3LIN_E_INVALID in next_workspace's
 *              status word and that row is written as zeros
 *   x_mod      device bf16 [M, K] (output), 16-byte aligned
 *   next_pre_quant_scale  the consumer's pre_quant_scale, fp32 [K] or NULL
 *   next_workspace        the consumer's workspace (>= header size, 16-byte aligned)
 * Rules: K % 64 == 0, 64 <= K <= 8192; table_rows >= 1; eps >= 0 finite;
 * M >= 0 (0: no-op).  Errors: H3LIN_E_SHAPE, H3LIN_E_INVALID, H3LIN_E_ALIGN,
 * H3LIN_E_WORKSPACE, H3LIN_E_UNSUPPORTED, H3LIN_E_CUDA; nothing is enqueued
 * on error.  Allocates nothing. */
h3lin_status h3lin_modulate_produce(const void* x, int64_t M, int64_t K, const float* table, int32_t table_rows,
                                    const int32_t* row_table, float eps, void* x_mod,
                                    const float* next_pre_quant_scale, void* next_workspace,
                                    size_t next_workspace_bytes, cudaStream_t stream);

/* ------------------------------------- Q/K RMSNorm + split-half RoPE step */
/* The step after the fused QKV projection (MiniMax-H3 Ultra Fast README,
 * "Active optimization stack", row "Attention projections": one fused in-place
 * Q/K RMSNorm + partial split-half RoPE kernel per block; "Kernel path", item
 * 2: three-axis split-half rotary embedding; head size 128 with 96 rotated
 * dimensions: MiniMax-H3 Turbo — one file, no Python, the list of conventions
 * before "Two clocks").  In place on the projection's bf16 output
 * qkv [M, 3 * heads * head_dim] = [Q | K | V] (head-major), for every row m
 * and every head of Q (gain q_gain) and of K (gain k_gain):
 *
 *   y[d]   = x[d] / sqrt(mean_d(x^2) + eps) * gain[d]            (fp32)
 *   pair i < rot/2 of axis a (t, h, w: pairs concatenated in that order,
 *   axis_dims[a] / 2 each; j = i minus the pairs of the earlier axes):
 *     angle  = float(positions[m, a]) * theta^(-2 j / axis_dims[a])
 *     out[i]         = y[i] cos(angle) - y[i + rot/2] sin(angle)
 *     out[i + rot/2] = y[i + rot/2] cos(angle) + y[i] sin(angle)
 *   out[d] = y[d] for rot <= d < head_dim;  stored as bf16 (round to nearest)
 *
 * V is not touched.  The frequencies are computed on the host in double and
 * rounded to float; angles in float, then sincosf.
 *   qkv        device bf16, 16-byte aligned; rows >= M never touched
 *   q_gain, k_gain  device fp32 [head_dim], 16-byte aligned
 *   positions  device int32 [M, 3] (t, h, w), 4-byte aligned
 *   workspace  >= h3lin_quant_workspace_bytes(), initialised once; only its
 *              status word is used (a timed-out device wait records
 *              H3LIN_E_TIMEOUT there, read with h3lin_read_status)
 * Rules: head_dim == 128; rot_dims % 16 == 0, 16 <= rot_dims <= head_dim;
 * axis_dims even, >= 0, summing to rot_dims; heads >= 1; theta > 0 and eps
 * >= 0 finite; M >= 0 (M == 0: no-op).  Errors: H3LIN_E_INVALID (null
 * pointer or parameter), H3LIN_E_SHAPE, H3LIN_E_ALIGN, H3LIN_E_UNSUPPORTED,
 * H3LIN_E_CUDA; nothing is enqueued on error.  Allocates nothing. */
typedef struct {
  int32_t heads;        /* heads of Q and of K */
  int32_t head_dim;     /* 128 */
  int32_t rot_dims;     /* rotated dimensions per head (96) */
  int32_t axis_dims[3]; /* rotated dimensions per position axis t, h, w */
  float theta;          /* frequency base (10000) */
  float eps;            /* RMSNorm epsilon (1e-6) */
} h3lin_rope_params;

h3lin_status h3lin_qk_norm_rope(void* qkv, int64_t M, const h3lin_rope_params* params, const float* q_gain,
                                const float* k_gain, const int32_t* positions, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/* ------------------- QKV projection with Q/K RMSNorm + RoPE in its epilogue */
/* The fused QKV projection and the Q/K RMSNorm + split-half RoPE step in one
 * GEMM (MiniMax-H3 Ultra Fast README, "Active optimization stack", row
 * "Attention projections"; "Kernel path", item 2): the GEMM's epilogue
 * normalises and rotates every Q and K head of its tile before the single
 * bf16 store, so Q and K are not read back and written again.  The result is
 * bit-identical to
 *     h3lin_forward(x, M, pre_quant_scale, weight, H3LIN_EPI_NONE, adapter,
 *                   strength, out, H3LIN_OUT_BF16, ...)
 *     h3lin_qk_norm_rope(out, M, params, q_gain, k_gain, positions, ...)
 * and out holds the same [Q | K | V] rows; the arguments mean what they mean
 * there.  A small pass first writes the (cos, sin) of every row's 48 rotation
 * pairs into the workspace (angles as h3lin_qk_norm_rope computes them).
 *   workspace  >= h3lin_forward_qk_rope_workspace_bytes(M, K, N, rank):
 *              h3lin_forward's regions plus M * 384 bytes of angles;
 *              initialised once (h3lin_workspace_init); its status word
 *              records a timed-out device wait
 * Rules: those of h3lin_forward and of h3lin_qk_norm_rope, and weight->N ==
 * 3 * heads * head_dim.  Only the shape the fused epilogue serves is
 * accepted: rot_dims == 96 (head_dim 128), an even head count (N % 256 == 0)
 * and a GPU with at least two SMs; any other valid parameters return
 * H3LIN_E_UNSUPPORTED (use the two calls above).  Errors: as h3lin_forward,
 * plus those of h3lin_qk_norm_rope's parameters; nothing is enqueued on
 * error.  M == 0: no-op.  Allocates nothing.
 *
 * h3lin_forward_gemm_qk_rope is its GEMM stage alone, after
 * h3lin_forward_prepare or h3lin_forward_prepare_produced on the same
 * workspace (as h3lin_forward_gemm). */
size_t       h3lin_forward_qk_rope_workspace_bytes(int64_t M, int64_t K, int64_t N, int32_t max_rank);
h3lin_status h3lin_forward_qk_rope(const void* x, int64_t M, const float* pre_quant_scale,
                                   const h3lin_weight* weight, const h3lin_adapter* adapter, float strength,
                                   const h3lin_rope_params* params, const float* q_gain, const float* k_gain,
                                   const int32_t* positions, void* out, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream);
h3lin_status h3lin_forward_gemm_qk_rope(int64_t M, const h3lin_weight* weight, const h3lin_adapter* adapter,
                                        float strength, const h3lin_rope_params* params, const float* q_gain,
                                        const float* k_gain, const int32_t* positions, void* out,
                                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------- failure self-test */
/* Exercises the kernels' failure path on the device without any fault: a
 * kernel waits, with a bound of `wait_cycles` SM clock cycles (1 .. 2^31), on
 * an mbarrier that nothing ever arrives on.  The wait runs out, the kernel
 * records H3LIN_E_TIMEOUT in the workspace status word (read it with
 * h3lin_read_status, clear it with h3lin_workspace_init), stops its other
 * waiter through the CTA abort flag and returns; the context stays usable.
 * Every wait in the production kernels is bounded the same way (about 2^31
 * cycles).  No counterpart in the paper: part of the library's failure
 * detection. */
h3lin_status h3lin_selftest_wait_timeout(void* workspace, size_t workspace_bytes, int64_t wait_cycles,
                                         cudaStream_t stream);

/* ------------------------------------------------------- bounds self-test */
/* The bounds build of this library (libh3lin_bounds.so, compiled with
 * -DH3LIN_BOUNDS) checks in its kernels the index of every plain global
 * access that no TMA tensor map bounds; an index outside its buffer records
 * H3LIN_E_BOUNDS in the workspace status word and the access is skipped, so
 * a bad index is reported instead of corrupting memory or faulting.  This
 * entry point proves the check is live: a kernel stores through an index
 * past the end of a 16-byte window inside the workspace header (the store's
 * address is still inside the workspace); the check must record
 * H3LIN_E_BOUNDS and skip it.  In the normal build it returns
 * H3LIN_E_UNSUPPORTED and enqueues nothing.  No counterpart in the paper:
 * part of the library's memory-safety checks.
 *   workspace  >= h3lin_quant_workspace_bytes(), initialised */
h3lin_status h3lin_selftest_bounds(void* workspace, size_t workspace_bytes, cudaStream_t stream);
int32_t      h3lin_bounds_build(void);   /* 1 in the bounds build, else 0 */

/* ----------------------------------------------- forward without allocation */
/* No counterpart in the paper: a library-level addition.
 *
 * h3lin_forward for callers that cannot allocate device memory at all (for
 * example a plugin inside a host application that owns every allocation and
 * gives plugins no allocator, or a latency-bound loop where cudaMalloc and
 * cudaFree are forbidden because they can block on the device).  Same
 * arguments and results as h3lin_forward, minus the workspace: the scratch
 * is a fixed H3LIN_NOALLOC_SCRATCH_BYTES array inside the library, one per
 * CUDA context the library's module is loaded into, held until that context
 * is destroyed (the primary context: process exit or cudaDeviceReset).
 * Nothing is allocated.
 *   - Calls whose scratch need (h3lin_forward_workspace_bytes) exceeds
 *     H3LIN_NOALLOC_SCRATCH_BYTES return H3LIN_E_WORKSPACE, enqueueing nothing.
 *   - All calls in a context share the array; calls that may overlap on the
 *     GPU race on it.  Order them on one stream.
 *   - The array's device address is looked up on the first call made in each
 *     context (the current one) and again whenever a call finds a context it
 *     has not seen before, e.g. after cudaDeviceReset or when the caller makes
 *     its own driver context current.  Make the first call in each context
 *     before any stream capture begins.
 *   - A timed-out device wait is recorded in a status word inside the array,
 *     not returned by this call (which only enqueues): read it, and clear it,
 *     with h3lin_noalloc_read_status. */
#define H3LIN_NOALLOC_SCRATCH_BYTES (64u << 20)
h3lin_status h3lin_forward_noalloc(const void* x, int64_t M, const float* pre_quant_scale,
                                   const h3lin_weight* weight, int32_t epilogue,
                                   const h3lin_adapter* adapter, float strength, void* out,
                                   int32_t out_dtype, cudaStream_t stream);
/* Synchronises `stream`, reads the status word of the current context's
 * allocation-free scratch into *device_status (H3LIN_OK or H3LIN_E_TIMEOUT)
 * and, when it is set, clears it so that later calls start clean.  No
 * counterpart in the paper.  Allocates nothing. */
h3lin_status h3lin_noalloc_read_status(cudaStream_t stream, int32_t* device_status);

/* ------------------------------------------------------------------ status */
/* Synchronises `stream`, then reads the workspace's sticky device status word
 * (H3LIN_OK or H3LIN_E_TIMEOUT) into *device_status.  Returns H3LIN_E_CUDA if
 * the stream reported an error. */
h3lin_status h3lin_read_status(const void* workspace, cudaStream_t stream, int32_t* device_status);
const char*  h3lin_status_string(h3lin_status status);
int32_t      h3lin_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* H3LIN_H */
