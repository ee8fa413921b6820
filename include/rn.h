/*
 * rn.h — C ABI of a GB300 (sm_103a) library of fused LayerNorm / RMSNorm
 * kernels with FP8 (E4M3), MXFP8 and NVFP4 output quantization, and of the
 * scaled activations (SReLU, SwiGLU, clamped SwiGLU) with the same
 * quantized outputs.
 *
 * What is computed follows the page "Implementation:NVIDIA TransformerEngine
 * PyTorch Ext Normalization": forward functions normalize each row of x and
 * optionally quantize the output, choosing between an unfused path, a fully
 * fused kernel (delayed-scaling FP8, MXFP8) and a norm+amax-then-quantize
 * path (current-scaling FP8, and the same for NVFP4) (section "Description");
 * they return the output,
 * mu (LayerNorm only) and rsigma (section "I/O Contract"); backward functions
 * return dx, dgamma and dbeta; gamma may be zero-centered; sm_margin leaves
 * SMs free; calls that need scratch memory follow a two-step protocol (query
 * the workspace size, allocate, execute).
 *
 * Arithmetic (the page gives no formula; standard readings):
 *   LayerNorm  mu = mean(x), var = mean((x-mu)^2), rsigma = 1/sqrt(var+eps),
 *              y = (x-mu)*rsigma*g + beta
 *   RMSNorm    rsigma = 1/sqrt(mean(x^2)+eps), y = x*rsigma*g
 *   g = 1 + gamma when zero_centered_gamma, else gamma.
 *   Statistics are accumulated in fp32; y is formed in fp32 ("y32").
 *   FP8_DELAYED  code = E4M3(fp32(y32*scale)), amax = max|y32| (whole tensor)
 *   FP8_CURRENT  amax = max|y32|, scale = 448/amax (1 if amax == 0), then as
 *                FP8_DELAYED; x is read twice (norm+amax pass, quantize pass)
 *   MXFP8        per block of 32 (1x32 along rows and 32x1 down columns):
 *                e = floor(log2(max|y32|)) - 8 clamped to [-127,127], stored
 *                as the E8M0 byte e+127; code = E4M3(y32 * 2^-e)
 *   NVFP4        (the page names the path only; NVIDIA's published NVFP4
 *                layout is taken): amax = max|y32|, S = 448*6/amax (fp32
 *                division, capped at the largest finite fp32; 1 if amax ==
 *                0); per block of 16 along a row A = max|y32|, scale code
 *                sc = E4M3(fp32(A * fp32(S/6))), element code
 *                E2M1(fp32(y32 * fp32(S / value(sc)))) (0 when value(sc)
 *                == 0); x is read twice as for FP8_CURRENT.  The value an
 *                element stands for is E2M1 value * value(sc) / S.
 *   E4M3 conversion: round to nearest even, saturate to +-448, NaN -> 0x7F.
 *   E2M1 conversion: round to nearest even, saturate to +-6; the sign bit
 *                follows the input (negative values that round to 0 give
 *                0x8).  NVFP4 output of non-finite inputs is unspecified.
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers, row-major, owned by the
 *     caller; the library allocates no memory and keeps no state apart from
 *     per-device attribute caches and a device-side error word.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and never synchronizes.
 *   - x is [N, H]; gamma, beta are fp32 [H]; mu, rsigma are fp32 [N].
 *   - Pointers must be 16-byte aligned; H must be a multiple of 8 for bf16
 *     and of 4 for fp32.  MXFP8 additionally needs H % 32 == 0 and
 *     N % 32 == 0; NVFP4 needs H % 16 == 0.  Violations return
 *     RN_ERR_UNSUPPORTED (shape/alignment) or RN_ERR_INVALID (missing
 *     pointer, bad enum, negative size) before anything is launched.
 *   - Row widths (with 227 KB of shared memory per block, as on GB300):
 *     every forward mode but two-direction MXFP8 takes H up to 32768 bf16 /
 *     16384 fp32 columns; the backward H up to 16384 bf16 / 8192 fp32.
 *     MXFP8 with the columnwise copy: bf16 rows with H % 64 == 0 and every
 *     fp32 row take a kernel that holds no whole 32-row tile, up to
 *     H = 41216 bf16 / 20608 fp32 (its per-tile statistics partials must
 *     fit beside 4 copy slots); bf16 rows with
 *     H % 64 == 32 take a kernel that holds a 32-row tile plus look-ahead,
 *     up to H = 3104 (LayerNorm) / 3296 (RMSNorm).  Wider rows return
 *     RN_ERR_UNSUPPORTED.
 *   - 0 <= sm_margin < number of SMs; the persistent grid uses
 *     (SMs - sm_margin) CTAs.  No result depends on sm_margin.
 *   - N == 0 is valid and launches nothing (the backward then writes zeros
 *     to dgamma/dbeta).
 *   - RN_ERR_CUDA reports a failed launch (cudaGetLastError) or a failed
 *     device query.
 */
#ifndef RN_H_
#define RN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RN_QUANT_NONE = 0,        /* unquantized output in out_dtype */
  RN_QUANT_FP8_DELAYED = 1, /* E4M3 with a caller-given scale */
  RN_QUANT_FP8_CURRENT = 2, /* E4M3 with scale = 448 / amax of this tensor */
  RN_QUANT_MXFP8 = 3,       /* E4M3 with E8M0 scales per 1x32 and 32x1 block */
  RN_QUANT_NVFP4 = 4        /* E2M1 with an E4M3 scale per 1x16 block and an
                               fp32 tensor scale 448*6/amax */
} rn_quant_mode;

typedef enum { RN_BF16 = 0, RN_F32 = 1 } rn_dtype;

typedef enum {
  RN_OK = 0,
  RN_ERR_INVALID = 1,     /* bad argument (NULL where required, bad enum) */
  RN_ERR_UNSUPPORTED = 2, /* valid request this library does not run */
  RN_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
  RN_ERR_CUDA = 4         /* CUDA runtime error */
} rn_status;

/*
 * Output descriptor of the forward calls and rn_quantize_only.  Fields a
 * mode does not use must be NULL.
 *   data        NONE: [N, H] in out_dtype.  FP8_*: uint8 E4M3 codes [N, H].
 *               MXFP8: rowwise uint8 E4M3 codes [N, H].
 *   row_scales  MXFP8: E8M0 bytes [N, H/32] (scale of data[i, 32b:32b+32]).
 *   col_data    MXFP8: columnwise codes stored TRANSPOSED, uint8 [H, N]:
 *               col_data[j, i] is the code of y[i, j] in its 32x1 block.
 *   col_scales  MXFP8: E8M0 bytes [H, N/32] (scale of col_data[j, 32b:32b+32]).
 *   NVFP4:      data = E2M1 codes packed two per byte, uint8 [N, H/2]
 *               (byte j of row i: element 2j in bits 0-3, 2j+1 in bits
 *               4-7); row_scales = E4M3 scale codes [N, H/16] (scale of
 *               elements 16b .. 16b+15 of a row); scale_out = S;
 *               scale_inv = fp32(1/S); amax as for FP8_CURRENT.
 *   scale       FP8_DELAYED: input, device fp32 scalar.
 *   scale_out   FP8_CURRENT: output, device fp32 scalar (448 / amax).
 *   scale_inv   FP8_*, NVFP4: output, device fp32 scalar 1/scale (IEEE division).
 *   amax        FP8_*, NVFP4: output, device fp32 scalar max|y32|; the library
 *               zeroes it on `stream` before reducing into it.
 *   out_dtype   NONE only: RN_BF16 or RN_F32 (fp32 returns y32 itself).
 * MXFP8 may skip either direction: data == NULL skips the rowwise output
 * (row_scales must then be NULL too), col_data == NULL the columnwise one.
 */
typedef struct {
  void* data;
  uint8_t* row_scales;
  uint8_t* col_data;
  uint8_t* col_scales;
  const float* scale;
  float* scale_out;
  float* scale_inv;
  float* amax;
  rn_dtype out_dtype;
} rn_output;

/*
 * LayerNorm forward (page section "Signature": layernorm_fwd(input, weight,
 * bias, eps, quantizer, sm_margin, zero_centered_gamma) -> (output, mu,
 * rsigma)).  x: [N, H] in x_dtype; gamma, beta: fp32 [H]; writes *out per
 * `mode`, mu and rsigma (fp32 [N]).  No scratch memory is used in any mode,
 * so the forward takes no workspace.
 */
rn_status rn_layernorm_fwd(const void* x, rn_dtype x_dtype, const float* gamma,
                           const float* beta, int64_t N, int64_t H, float eps,
                           int zero_centered_gamma, int sm_margin,
                           rn_quant_mode mode, const rn_output* out, float* mu,
                           float* rsigma, void* stream);

/*
 * RMSNorm forward (page: rmsnorm_fwd(input, weight, eps, quantizer,
 * sm_margin, zero_centered_gamma); mu is "LayerNorm only").  As
 * rn_layernorm_fwd without beta and mu.
 */
rn_status rn_rmsnorm_fwd(const void* x, rn_dtype x_dtype, const float* gamma,
                         int64_t N, int64_t H, float eps,
                         int zero_centered_gamma, int sm_margin,
                         rn_quant_mode mode, const rn_output* out,
                         float* rsigma, void* stream);

/*
 * Residual add + LayerNorm / RMSNorm forward: the single-GPU core of the
 * fused "reduce-scatter + residual add + RMSNorm + all-gather" named on the
 * page "NVIDIA Megatron-Core ... core.tensor_parallel.inference_layers"
 * (the collectives are not part of this library).
 *   h = x + residual, each element rounded once (to nearest even) to the
 *       dtype of x — the new residual stream, written to residual_out;
 *   then exactly rn_layernorm_fwd / rn_rmsnorm_fwd of h (mu, rsigma, output
 *   per `mode`).
 * x, residual, residual_out: [N, H] in `dtype`, 16-byte aligned;
 * residual_out may not alias x or residual.  Every mode: FP8_CURRENT and
 * NVFP4 read residual_out in their second pass; MXFP8 with the rowwise
 * blocks only is one pass, and with the columnwise copy two kernels (the
 * first forms h, the rowwise blocks when asked for and mu / rsigma, the
 * second reads residual_out back for the columnwise blocks and writes mu /
 * rsigma again from the same h), both planned before either is launched,
 * with the width limits of the plain forward's two-direction MXFP8.  Other
 * arguments, errors and conventions as in the plain forward.
 */
rn_status rn_layernorm_add_fwd(const void* x, const void* residual, rn_dtype dtype,
                               const float* gamma, const float* beta, int64_t N, int64_t H,
                               float eps, int zero_centered_gamma, int sm_margin,
                               rn_quant_mode mode, const rn_output* out, void* residual_out,
                               float* mu, float* rsigma, void* stream);

rn_status rn_rmsnorm_add_fwd(const void* x, const void* residual, rn_dtype dtype,
                             const float* gamma, int64_t N, int64_t H, float eps,
                             int zero_centered_gamma, int sm_margin, rn_quant_mode mode,
                             const rn_output* out, void* residual_out, float* rsigma,
                             void* stream);

/*
 * LayerNorm backward (page: layernorm_bwd(dz, x, mu, rsigma, gamma,
 * sm_margin, zero_centered_gamma) -> (dx, dgamma, dbeta)).
 *   dz, x, dx: [N, H] in `dtype`; mu, rsigma: the forward's fp32 [N];
 *   gamma: fp32 [H] (stored value; zero_centered_gamma as in the forward);
 *   dgamma, dbeta: fp32 [H], overwritten.
 * dgamma/dbeta are reduced in two deterministic stages: fixed row chunks
 * (their size depends on N, H and the device's SM count, never on
 * sm_margin) write fp32 partial sums, each in row order, into the
 * workspace, then a second kernel adds the chunks of every column in a
 * fixed order that depends on the chunk count and H only.  Results are
 * bitwise reproducible and independent of sm_margin.  The size the query
 * reports depends on N, H and dtype only (it covers every chunking).
 * Workspace protocol: with workspace == NULL the call only stores the
 * required byte count in *workspace_bytes and returns RN_OK; otherwise
 * *workspace_bytes must hold the size of `workspace` (16-byte aligned,
 * caller-owned, contents need not be initialized); too small ->
 * RN_ERR_WORKSPACE.  The workspace must not be shared by calls that may run
 * concurrently.
 */
rn_status rn_layernorm_bwd(const void* dz, const void* x, rn_dtype dtype,
                           const float* mu, const float* rsigma,
                           const float* gamma, int64_t N, int64_t H,
                           int zero_centered_gamma, int sm_margin, void* dx,
                           float* dgamma, float* dbeta, void* workspace,
                           size_t* workspace_bytes, void* stream);

/*
 * RMSNorm backward (page: rmsnorm_bwd(dz, x, rsigma, gamma, sm_margin,
 * zero_centered_gamma) -> (dx, dgamma)).  As rn_layernorm_bwd without mu
 * and dbeta.
 */
rn_status rn_rmsnorm_bwd(const void* dz, const void* x, rn_dtype dtype,
                         const float* rsigma, const float* gamma, int64_t N,
                         int64_t H, int zero_centered_gamma, int sm_margin,
                         void* dx, float* dgamma, void* workspace,
                         size_t* workspace_bytes, void* stream);

/*
 * LayerNorm backward that allocates nothing (the pages have no counterpart:
 * this is an addition for callers that cannot allocate device memory where
 * they run the backward, e.g. code that must not call cudaMalloc because it
 * may synchronize the device, or that runs without an allocator of its own).
 * Same arguments, arithmetic and results as rn_layernorm_bwd, minus the
 * workspace: the dgamma/dbeta partial sums go to a fixed 16 MiB array that
 * the library image places in the memory of every device that loads it and
 * that stays there until the process exits.
 *   - Limit: problems whose partials exceed 16 MiB (chunks * 2 * H * 4 bytes;
 *     e.g. N = 3000, H = 5120 fits, N = 8192, H = 4096 does not) return
 *     RN_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on each device looks up the array's device address
 *     (with that device current); make that first call before any stream
 *     capture.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents; nothing in it needs to start at zero (each call
 *     overwrites every partial it reads).  Calls whose kernels may overlap on
 *     the GPU (different streams, or host threads without ordering) race on
 *     the array and must be serialized by the caller.
 * No cudaMalloc / cudaFree or other allocating call is made.
 */
rn_status rn_layernorm_bwd_noalloc(const void* dz, const void* x, rn_dtype dtype,
                                   const float* mu, const float* rsigma,
                                   const float* gamma, int64_t N, int64_t H,
                                   int zero_centered_gamma, int sm_margin,
                                   void* dx, float* dgamma, float* dbeta,
                                   void* stream);

/*
 * Delayed-scaling recipe step (closes the loop around RN_QUANT_FP8_DELAYED;
 * the page describes delayed scaling but not its bookkeeping, so this is the
 * common recipe with margin 0):
 *   amax_history: device fp32 [history_len], most recent first, updated in
 *                 place: shifted down one place, *amax written at index 0;
 *   amax:         device fp32 scalar, the new amax (e.g. a forward's output);
 *   scale:        device fp32 scalar, in: the current scale, out: the next,
 *                 fp32(448 / max(history)) by IEEE division, or unchanged
 *                 when that maximum is 0, negative, infinite or NaN;
 *   scale_inv:    device fp32 scalar, out: fp32(1 / scale).
 * 1 <= history_len <= 1024 (else RN_ERR_INVALID / RN_ERR_UNSUPPORTED);
 * one small kernel on `stream`.
 */
rn_status rn_delayed_scaling_update(float* amax_history, int64_t history_len,
                                    const float* amax, float* scale,
                                    float* scale_inv, void* stream);

/*
 * Scaled activations (page "Activation + GroupedLinear Fusion for MOE and
 * other MOE optimizations", section "Better Kernels for Scaled Activations":
 * scaled SReLU, SwiGLU and clamped SwiGLU as fused kernels whose backward
 * also returns the gradient of the scales).  The page gives no formula;
 * standard readings:
 *   y[i, j] = s_i * act(x)[i, j], one fp32 scale per row (NULL: all 1);
 *   RN_ACT_SRELU           x [N, H]:  act = max(x, 0)^2
 *   RN_ACT_SWIGLU          x [N, 2H] = [a | b]: act = a * sigmoid(a) * b
 *   RN_ACT_CLAMPED_SWIGLU  x [N, 2H] = [a | b]: ac = min(a, limit),
 *                          bc = clamp(b, -limit, limit),
 *                          act = ac * sigmoid(alpha * ac) * (bc + 1)
 *                          (limit >= 0; e.g. limit 7, alpha 1.702)
 * sigmoid(z) = 1 / (1 + exp(-z)); y is formed in fp32.  limit and alpha are
 * ignored by the other forms.  Outputs of non-finite inputs are unspecified.
 */
typedef enum {
  RN_ACT_SRELU = 0,
  RN_ACT_SWIGLU = 1,
  RN_ACT_CLAMPED_SWIGLU = 2
} rn_act;

/*
 * Forward: H is the OUTPUT width; x is [N, H] (SReLU) or [N, 2H] in `dtype`
 * (16-byte aligned; H * element size a multiple of 16), scales fp32 [N] or
 * NULL.  `mode` and *out as for rn_layernorm_fwd, with MXFP8 giving the
 * rowwise 1x32 blocks only (data [N, H], row_scales [N, H/32]; col_data and
 * col_scales must be NULL, else RN_ERR_UNSUPPORTED; H % 32 == 0) and NVFP4
 * not offered (RN_ERR_UNSUPPORTED).  FP8_CURRENT reads x twice (amax pass,
 * then quantize).  Asynchronous on `stream`; no workspace.
 */
rn_status rn_scaled_act_fwd(rn_act act, const void* x, rn_dtype dtype,
                            const float* scales, int64_t N, int64_t H,
                            float limit, float alpha, rn_quant_mode mode,
                            const rn_output* out, void* stream);

/*
 * Backward: dy [N, H] and x (the forward's input) in `dtype`; writes
 *   dx [N, H] or [N, 2H] (the shape of x, `dtype`):
 *       dx = s_i * dy * d act / d x   (the a half, then the b half);
 *       the clamps pass the gradient where the input lies within the
 *       bounds, bounds included;
 *   dscales fp32 [N] (may be NULL to skip): sum_j dy[i, j] * act(x)[i, j].
 * dx is rounded once to `dtype`; dscales is an fp32 sum in an unspecified
 * but fixed order.  Pointers 16-byte aligned (dscales 4).
 */
rn_status rn_scaled_act_bwd(rn_act act, const void* dy, const void* x, rn_dtype dtype,
                            const float* scales, int64_t N, int64_t H,
                            float limit, float alpha, void* dx, float* dscales,
                            void* stream);

/*
 * Quantization stage alone on caller-given fp32 values y [N, H] (the
 * page's UNFUSED path: norm, then a separate quantize).  Same output
 * descriptor and arithmetic as the fused forward for `mode`
 * (FP8_DELAYED, FP8_CURRENT, MXFP8 or NVFP4); lets the quantizer be checked bit
 * for bit on arbitrary fp32 inputs.
 */
rn_status rn_quantize_only(const float* y, int64_t N, int64_t H,
                           rn_quant_mode mode, const rn_output* out,
                           void* stream);

/* Static message for a status code. */
const char* rn_status_str(rn_status s);

/*
 * Reads and clears the device-side error word of the current device
 * (synchronizes the device).  Kernels never trap: a pipeline wait that
 * exceeds its time limit records a nonzero code here and the kernel runs
 * to completion.  *code = 0 means no error was recorded.
 */
rn_status rn_device_error(unsigned int* code);

/* ABI version of this header (increments on incompatible change). */
int rn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RN_H_ */
