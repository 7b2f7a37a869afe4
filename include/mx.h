/*
 * mx.h -- C ABI of the GB300 (sm_103a) microscaled (OCP MX) quantized linear.
 *
 * Weights are OCP e4m3 (MXFP8) bytes or packed e2m1 (MXFP4, fp4x2, low nibble
 * first) with one E8M0 power-of-two scale code per 32-element K block; code c
 * stands for 2^(c - 127).  Sources, cited by page title and section:
 *
 *   weights942  = vllm.models.deepseek_v41.amd.mono.weights942
 *   rocm_native = vllm.model_executor.kernels.linear.mxfp8.rocm_native
 *   a16w4       = vllm.models.minimax_m3.amd.specialized_decode.mono.a16w4
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller, 16-byte aligned,
 *     row-major and dense.  The library allocates no memory.  bf16 tensors are
 *     passed as void*.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work and return; only mx_pack_weights and mx_check_device_errors
 *     synchronise the stream.
 *   - The return value is an MX_* status.  On failure nothing was enqueued and
 *     mx_last_error() returns a message (per host thread).  Conditions only the
 *     device can see (bad expert ids) are written to a caller-provided device
 *     int (`dev_status`) instead; no kernel ever traps.
 *   - All calls require the current device to be an sm_103 GPU.
 */
#ifndef MX_GB300_H
#define MX_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
enum {
  MX_OK = 0,
  MX_ERR_SHAPE = 1,        /* a size is out of range or inconsistent          */
  MX_ERR_ALIGN = 2,        /* a pointer is not 16-byte aligned                 */
  MX_ERR_ARG = 3,          /* NULL pointer, unknown format / mode / flag       */
  MX_ERR_NOT_BLOCK32 = 4,  /* 32x32 block codes required, rows disagree       */
  MX_ERR_SCALE = 5,        /* an E8M0 weight code is 255 (NaN)                */
  MX_ERR_WORKSPACE = 6,    /* workspace missing or smaller than required      */
  MX_ERR_EXPERT_ID = 7,    /* (device status) an expert id outside [-1, E)     */
  MX_ERR_CUDA = 8,         /* a CUDA runtime call failed                      */
  MX_ERR_UNSUPPORTED = 9,  /* device is not sm_103, or a size beyond a limit  */
  MX_ERR_TIMEOUT = 10,     /* (device flag) a bounded wait inside a kernel ran out */
  MX_ERR_INEXACT = 11      /* a bf16 weight is not e4m3 x its scale (weights942,
                              ocp_from_dequant refuses it)                      */
};

enum { MX_FMT_E4M3 = 0, MX_FMT_E2M1 = 1 };
enum { MX_SCALE_BLOCK32X32 = 0, MX_SCALE_ROW1X32 = 1 };

/* mx_pack_weights flags */
#define MX_PACK_FOLD 1u          /* fold [N, K/32] row codes into [N/32, K/32] blocks when
                                    every 32 rows agree (rocm_native, _as_block32_scale)   */
#define MX_PACK_REQUIRE_BLOCK 2u /* fail with MX_ERR_NOT_BLOCK32 when they do not
                                    (weights942, linear_copy)                              */
#define MX_PACK_GATE_UP 4u       /* E2M1 only: the weight is a gate / up expert tensor
                                    [E, 2 I, K/2] with the I gate rows first, then the I up
                                    rows (weights942, moe_copies); pack it with the halves
                                    interleaved in 8-row groups (layout MX_LAYOUT_GATE_UP).
                                    Needs N = 2 I a multiple of 16.                        */

/* mx_packed_weight.layout */
#define MX_LAYOUT_PLAIN 0
#define MX_LAYOUT_GATE_UP 1      /* packed row 16 q + i = gate row 8 q + i (i < 8), else
                                    up row 8 q + i - 8; codes alike                         */

/* mxfp8_linear flags */
#define MX_LINEAR_NO_FUSED_QUANT 1u /* M <= 32: always quantize x in a separate launch into
                                       the workspace (the pages' kill switch of the fused
                                       quant, rocm_native, apply_weights); same bits      */
#define MX_LINEAR_CLUSTER_GEMV (1u << 14) /* M <= 32: run the CUDA-core-scaled mma.sync GEMV
                                       with cluster split-K (fused quant for M <= 8)
                                       instead of the tensor-core GEMV                      */

/* Largest token count the GEMV path serves; larger M runs the block-scaled GEMM. */
#define MX_GEMV_MAX_M 32
/* Largest expert count mx_route_experts / mxfp4_moe_linear accept. */
#define MX_MAX_EXPERTS 512

/*
 * A packed weight, filled by mx_pack_weights.  All pointers are device
 * pointers into the caller's pack buffer; the struct itself is plain host
 * memory the caller keeps and passes back by pointer.
 *
 * E4M3 (dense MXFP8), K padded to Kp = roundup(K, 128) with zero bytes and
 * code 128 (weights942, dense_copy):
 *   bytes  [E, N, Kp]          row-major e4m3
 *   codes  [E, N/32, Kp/32]    (scale_mode BLOCK32X32) or [E, N, Kp/32] (ROW1X32)
 *   sf     [E, ceil(N/128), Kp/128, 512]  per-row codes in 512-byte atoms: row
 *          n = 128 rt + m and K block j = 4 kt + kb at byte
 *          (m % 32) * 16 + (m / 32) * 4 + kb of atom (rt, kt); 127 past N.
 * E2M1 (MXFP4 experts):
 *   bytes  [E, ceil(N/128), Kp/128, 128, 64]  128-row x 128-value tiles, each
 *          a contiguous 8 KB block: tile (rt, kt) row m holds values
 *          128 kt .. 128 kt + 127 of row 128 rt + m as 64 fp4x2 bytes in the
 *          input order (element 2i in the low nibble of byte i); zero past K
 *          and past N; -0 nibbles rewritten to +0 (weights942,
 *          fp4_drop_negative_zero_)
 *   codes  [E, N, Kp/32] per-row codes, 128 past K
 *   sf     [E, ceil(N/128), Kp/128, 512]  the per-row codes in 512-byte atoms
 *          as for E4M3 (127 past N)
 *   With MX_PACK_GATE_UP the rows of bytes, codes and sf are interleaved in
 *   8-row groups: packed row 16 q + i holds gate row 8 q + i (i < 8) or up row
 *   8 q + i - 8 (i >= 8) of the gate-then-up tensor (layout MX_LAYOUT_GATE_UP).
 */
typedef struct mx_packed_weight {
  int32_t fmt;         /* MX_FMT_*                                 */
  int32_t scale_mode;  /* MX_SCALE_*                               */
  int32_t E, N, K, Kp; /* experts, rows, logical K, padded K       */
  uint8_t* bytes;
  uint8_t* codes;
  uint8_t* sf;
  int64_t neg_zero_count; /* -0 nibbles rewritten (E2M1), else 0   */
  int32_t layout;         /* MX_LAYOUT_* (row order of the packed rows) */
} mx_packed_weight;

/* Message of the last failed call on this host thread ("" if none). */
const char* mx_last_error(void);

/*
 * Reads and clears the library's device error flags on the current device
 * (synchronises the device).  Returns MX_OK, or MX_ERR_TIMEOUT when a bounded
 * in-kernel wait gave up since the last check.
 */
int mx_check_device_errors(void);

/* ------------------------------------------------------------------ packing */

/* Bytes the pack buffer needs for a weight of this format and shape
 * (0 if the shape is invalid). */
size_t mx_pack_size(int fmt, int E, int N, int K);

/*
 * Load-time repack of MX weights into the layout above (one device pass).
 *   bytes       E4M3: [E, N, K] e4m3;  E2M1: [E, N, K/2] fp4x2, low nibble first
 *               (weights942, moe_copies: w13 [E, 2Np, K/2])
 *   codes       [E, codes_rows, K/32] E8M0, codes_rows = N (1x32 rows) or
 *               N/32 (32x32 blocks, weights942 dense_copy: [N/32, K/32])
 *   flags       MX_PACK_FOLD / MX_PACK_REQUIRE_BLOCK (E4M3; E2M1 always keeps
 *               per-row codes), MX_PACK_GATE_UP (E2M1)
 *   dst/dst_bytes  caller buffer of at least mx_pack_size() bytes, 256-byte aligned
 *   out         filled on success
 * Requirements: K % 32 == 0, N >= 1, E >= 1; codes_rows = N/32 needs N % 32 == 0.
 * Errors: MX_ERR_SCALE if a code is 255; MX_ERR_NOT_BLOCK32 if REQUIRE_BLOCK and
 * the rows of some 32-row group disagree.  The call synchronises `stream` (it
 * returns the fold decision and the -0 count, as the pages' host functions do).
 */
int mx_pack_weights(const uint8_t* bytes, const uint8_t* codes, int fmt, int E, int N,
                    int K, int codes_rows, unsigned flags, void* dst, size_t dst_bytes,
                    mx_packed_weight* out, void* stream);

/* ------------------------------------------------------------- activations */

/*
 * Per-token MXFP8 quantization of a bf16 activation (rocm_native,
 * _quant_mxfp8_tile): per row and 32-wide K block, amax = max(max|x|, 2^-126),
 * code = clamp(ceil(log2(amax / 448)) + 127, 0, 254), q = e4m3_rne(x * 2^(127 - code)).
 * A block holding NaN or inf gets code 255 and bytes 0x7F.
 *   x [M, K] bf16;  q [M, K] e4m3;  codes [M, K/32] E8M0, row-major
 *   (rocm_native, input_quant_key).  K % 32 == 0; M == 0 is a no-op.
 */
int mx_quantize_act(const void* x, int M, int K, uint8_t* q, uint8_t* codes, void* stream);

/*
 * The OCP e4m3 bytes behind a bf16 weight that was dequantized at load
 * (weights942, ocp_from_dequant: w = e4m3 value x 2^(code - 127)), so such a
 * weight can be packed and served as MXFP8.  Each value is scaled by
 * 2^(127 - code) and rounded to e4m3; the call refuses the weight unless every
 * byte gives its value back (dequant rounded to bf16; -0 equals +0, NaN never).
 *   w        [N, K] bf16 (16-byte aligned), K a multiple of 32
 *   codes    [N/32, K/32] (scale_mode BLOCK32X32) or [N, K/32] (ROW1X32)
 *   out      [N, K] e4m3 bytes (16-byte aligned)
 *   scratch  8 bytes of device memory the call may overwrite
 *   *mismatches  (host, may be NULL) the number of values not given back
 * Returns MX_ERR_INEXACT when that number is not 0.  Synchronises the stream.
 */
int mx_e4m3_from_dequant(const void* w, const uint8_t* codes, int scale_mode, int N, int K, uint8_t* out,
                         void* scratch, int64_t* mismatches, void* stream);

/*
 * Dequantize MX weights to bf16: out = bf16_rne(value(byte) * 2^(code - 127))
 * (weights942, ocp_from_dequant; rocm_native names it dequant_mxfp8_to_bf16).
 *   bytes  E4M3: [N, K];  E2M1: [N, K/2] fp4x2, low nibble first (unpacked order)
 *   codes  BLOCK32X32: [N/32, K/32]  or  ROW1X32: [N, K/32]
 *   out    [N, K] bf16.   Code 255 gives NaN.
 */
int mx_dequant(const uint8_t* bytes, const uint8_t* codes, int fmt, int scale_mode, int N,
               int K, void* out, void* stream);

/* ------------------------------------------------------------- MXFP8 linear */

/* Workspace bytes mxfp8_linear needs for M tokens on weight w: the size of the
 * quantized activation and its codes (used by the GEMM for M > 32, by the
 * MX_LINEAR_CLUSTER_GEMV path and with MX_LINEAR_NO_FUSED_QUANT; the default
 * decode GEMV uses none of it), plus,
 * for M > 32 when the GEMM's output tiles would leave more than half the SMs
 * of the current device idle, room for f32 partial sums of up to 8 K ranges
 * ([ranges, M, N], at most 64 MB; the size depends on the current device's SM
 * count, 152 assumed when there is no device).  That room is optional: a
 * workspace holding only the quantized activation and codes is accepted and
 * the GEMM then splits K into as many ranges as the bytes past them hold. */
size_t mxfp8_linear_workspace_size(int M, const mx_packed_weight* w);

/*
 * out = x @ w^T (+ bias) with the bf16 activation MXFP8-quantized per token
 * inside the call (rocm_native, apply_weights / _launch):
 *   y[m, n] = sum_b 2^(cw[n,b]-127) 2^(cx[m,b]-127) sum_{k in b} W[n,k] xq[m,k]
 * accumulated in fp32, bias added in fp32, rounded once to bf16.
 *   x     [M, K] bf16           w     packed E4M3 weight with E == 1
 *   bias  [N] bf16 or NULL      out   [M, N] bf16
 *   workspace  device scratch of mxfp8_linear_workspace_size(M, w) bytes
 * M <= MX_GEMV_MAX_M runs the split-K decode GEMV on the tensor cores (block
 * scales applied by tcgen05, activation quantized inside the kernel), larger M
 * the block-scaled GEMM (which, when its tiles would leave SMs idle, splits K
 * into ranges and adds their f32 sums in range order before the bias and the
 * one rounding).  Within the decode range a token's result does not depend on
 * M; above it, the K split (and so the f32 summation order) depends on M, the
 * device's SM count and the workspace's size.
 * The kernels start streaming w's buffers before the previous kernel on the
 * stream has finished (programmatic dependent launch): w must not be written
 * by the kernel launched just before on the same stream (mx_pack_weights
 * returns only once its writes are complete).  x, bias and out are ordered
 * with earlier work as usual.
 */
int mxfp8_linear(const void* x, int M, const mx_packed_weight* w, const void* bias, void* out,
                 unsigned flags, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes mxfp8_linear_q needs for M tokens on weight w (the
 * activation's scale-factor atoms for the GEMM when M > MX_GEMV_MAX_M, then
 * the optional room for the GEMM's K-range partial sums as in
 * mxfp8_linear_workspace_size; 0 for M <= MX_GEMV_MAX_M). */
size_t mxfp8_linear_q_workspace_size(int M, const mx_packed_weight* w);

/*
 * mxfp8_linear on an activation that arrives already MXFP8-quantized
 * (rocm_native, apply_weights / input_quant_key: a QuantizedActivation with
 * row-major, not swizzled, [M, K/32] E8M0 scales):
 *   y[m, n] = sum_b 2^(cw[n,b]-127) 2^(cx[m,b]-127) sum_{k in b} W[n,k] xq[m,k]
 * accumulated in fp32, bias added in fp32, rounded once to bf16.
 *   xq     [M, K] e4m3 bytes row-major (16-byte aligned)
 *   xcodes [M, K/32] E8M0 codes row-major
 *   w, bias, out as in mxfp8_linear; flags must be 0;
 *   workspace of mxfp8_linear_q_workspace_size(M, w) bytes (16-byte aligned).
 * Given (xq, xcodes) = mx_quantize_act(x), the result is bit-identical to
 * mxfp8_linear(x).  M <= MX_GEMV_MAX_M runs the decode GEMV, larger M the GEMM
 * reading xq in place.
 */
int mxfp8_linear_q(const uint8_t* xq, const uint8_t* xcodes, int M, const mx_packed_weight* w, const void* bias,
                   void* out, unsigned flags, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Scratch-free decode linear.  The source pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory or pass a
 * workspace -- engines that plan all device memory before serving and forbid
 * allocation on the request path, and plugin / callback code that receives
 * only its input and output buffers from a framework owning the allocator.
 *
 * Computes exactly what mxfp8_linear computes for M <= MX_GEMV_MAX_M with
 * flags MX_LINEAR_CLUSTER_GEMV | MX_LINEAR_NO_FUSED_QUANT, but keeps the quantized
 * activation and its codes in a fixed library-owned device array of
 * MX_NOALLOC_SCRATCH_BYTES, present on every GPU that loads the library until
 * the process exits.  It calls no allocator.
 *   - Limits: 1 <= M <= MX_GEMV_MAX_M and M*Kp + M*Kp/32 (+ 256-byte alignment)
 *     <= MX_NOALLOC_SCRATCH_BYTES (e.g. M = 32 up to K = 31744); otherwise
 *     MX_ERR_UNSUPPORTED with a message.  M == 0 is a no-op.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is kept per device together with the id of the context it
 *     belongs to; after a device reset (a new context) the next call looks it
 *     up again, so make that call outside a stream capture too.
 *   - All calls share the array: calls that overlap on the GPU (e.g. on two
 *     streams at once) race and must be serialised by the caller.  Each call
 *     writes every scratch byte it reads, so stale contents are harmless.
 */
#define MX_NOALLOC_SCRATCH_BYTES (1u << 20)
int mxfp8_linear_noalloc(const void* x, int M, const mx_packed_weight* w, const void* bias, void* out,
                         void* stream);

/* ------------------------------------------------------------------ MXFP4 MoE */

/*
 * Token -> expert grouping (the plainest reading of routed experts; the pages
 * show no router).  Pairs p = t * topk + j are grouped by id in increasing p.
 *   topk_ids [T, topk] int32; ids of -1 are skipped; ids outside [-1, E) are
 *            skipped and set *dev_status = MX_ERR_EXPERT_ID (else it is set to 0)
 *   counts [E], offsets [E + 1], pairs [T * topk] (first offsets[E] valid),
 *   active [E] (experts with a pair, ascending; first *n_active valid),
 *   n_active [1]: all int32 device outputs.   E <= MX_MAX_EXPERTS.
 */
int mx_route_experts(const int32_t* topk_ids, int T, int topk, int E, int32_t* counts,
                     int32_t* offsets, int32_t* pairs, int32_t* active, int32_t* n_active,
                     int* dev_status, void* stream);

/* Workspace bytes mxfp4_moe_linear needs for T tokens, top-k slots, E experts
 * of N output rows and activations of K values (0 for a shape it refuses).
 * It holds the routing, the activation pieces and, at decode sizes (T * topk
 * <= 64), f32 partial sums for splitting K when the few touched experts would
 * leave SMs idle. */
size_t mxfp4_moe_workspace_size(int T, int topk, int E, int N, int K);

/*
 * Routed A16W4 expert GEMM (a16w4 module text, dequant / step_mfma): for every
 * pair (t, j) with e = topk_ids[t, j] in [0, E),
 *   out[t, j, n] = sum_k bf16(e2m1(W_e[n,k]) * 2^(c_e[n,k/32] - 127)) * x[t, k]
 * in fp32, rounded to bf16; pairs with an invalid id get zeros.
 *   x [T, K] bf16; topk_ids [T, topk] int32; w packed E2M1 weight [E, N, K];
 *   out [T, topk, N] bf16; workspace of mxfp4_moe_workspace_size bytes;
 *   dev_status as in mx_route_experts.
 */
int mxfp4_moe_linear(const void* x, const int32_t* topk_ids, int T, int topk,
                     const mx_packed_weight* w, void* out, void* workspace,
                     size_t workspace_bytes, int* dev_status, void* stream);

/*
 * The routed expert GEMM with MXFP8 activations (MXFP4 x MXFP8, the prefill
 * form of the layer): x is quantized per token inside the call exactly as
 * mx_quantize_act does (rocm_native, _quant_mxfp8_tile), then for every pair
 * (t, j) with e = topk_ids[t, j] in [0, E)
 *   out[t, j, n] = sum_k e2m1(W_e[n,k]) 2^(c_e[n,k/32] - 127)
 *                        e4m3(q[t,k]) 2^(cx[t,k/32] - 127)
 * in fp32 on the tensor cores (kind::mxf8f6f4, both scales applied by the
 * MMA), rounded to bf16; pairs with an invalid id get zeros.  Arguments,
 * workspace (mxfp4_moe_workspace_size) and errors as mxfp4_moe_linear.
 */
int mxfp4_moe_linear_w4a8(const void* x, const int32_t* topk_ids, int T, int topk,
                          const mx_packed_weight* w, void* out, void* workspace,
                          size_t workspace_bytes, int* dev_status, void* stream);

/* Workspace bytes mxfp4_moe_expert needs for x [T, K], w13 [E, 2 I, K] and
 * w2 [E, H, I] (routing, the activation pieces, the activation [T*topk, I]
 * bf16 and the down projection [T*topk, H] f32). */
size_t mxfp4_moe_expert_workspace_size(int T, int topk, int E, int K, int I, int H);

/*
 * The routed expert MLP (A16W4 throughout), from the tensors weights942
 * moe_copies describes -- w13 [E, 2 I, K/2] gate rows then up rows, w2
 * [E, H, I/2]:
 *   g, u   = w13_e[:I] x_t, w13_e[I:] x_t        (as mxfp4_moe_linear)
 *   act    = bf16(silu(g) * u),  silu(v) = v / (1 + e^-v)   (f32, fused into
 *            the gate/up kernel's epilogue)
 *   y2     = w2_e act                              (f32, kept in the workspace)
 *   out[t] = bf16(sum_j topk_weights[t, j] * y2[t, j])  in increasing j, f32;
 *            slots whose id is not in [0, E) are skipped.
 * The activation and the combine are not printed on the pages (SiLU-and-mul
 * and a weighted sum over the top-k slots are the plain reading).
 *   x [T, K] bf16; topk_ids [T, topk] int32; topk_weights [T, topk] f32;
 *   w13 packed E2M1 with MX_PACK_GATE_UP (N = 2 I, K = x's K);
 *   w2 packed E2M1 plain (E alike, N = H, K = I; H a multiple of 4);
 *   out [T, H] bf16; workspace of mxfp4_moe_expert_workspace_size bytes
 *   (16-byte aligned); dev_status as in mx_route_experts.
 */
int mxfp4_moe_expert(const void* x, const int32_t* topk_ids, const float* topk_weights, int T, int topk,
                     const mx_packed_weight* w13, const mx_packed_weight* w2, void* out, void* workspace,
                     size_t workspace_bytes, int* dev_status, void* stream);

/* ------------------------------------------------------------------ self-test */

/*
 * Exercises the failure path of the library's bounded waits (no counterpart on
 * the source pages): one GPU thread waits on an mbarrier that nothing arrives
 * on, gives up after limit_us microseconds (1..100000), writes 1 to the device
 * int *waited_out, and raises the device timeout flag, so that the next
 * mx_check_device_errors() returns MX_ERR_TIMEOUT.  Nothing faults or traps.
 */
int mx_selftest_bounded_wait(int limit_us, int* waited_out, void* stream);

/* --------------------------------------------------------------- measurement */

/*
 * Measures the dense MXFP8 tensor throughput of the current device (no
 * counterpart on the source pages; the denominator of the block-scaled GEMM's
 * roofline fraction): every SM runs `iters` rounds of 8 block-scaled
 * tcgen05.mma kind::mxf8f6f4 (M = 128, N = 224, K = 32, e4m3 operands already
 * in shared memory, UE8M0 scales in tensor memory) from two issuing threads,
 * `reps` launches back to back on `stream` after one warm-up launch, timed with
 * CUDA events.  Writes TFLOP/s (2 flops a multiply-add) to *tflops.
 * Synchronizes the stream; allocates nothing.  1 <= iters <= 65536 (about
 * 2000 runs 1 ms), 1 <= reps <= 1000.  Errors: MX_ERR_ARG, MX_ERR_UNSUPPORTED
 * (not sm_103), MX_ERR_CUDA, MX_ERR_TIMEOUT (a bounded wait ran out or an
 * accumulator did not hold the expected sum).
 */
int mx_measure_mxf8_peak(int iters, int reps, double* tflops, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MX_GB300_H */
