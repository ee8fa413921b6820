// Host-side plumbing shared by the translation units of the library: kernel
// parameter blocks, launch plans and the per-unit launch functions.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/rn.h"

namespace rn {

// what a kernel does before quantizing: normalize (RMSNorm / LayerNorm) or
// take its fp32 input as y already (the stand-alone quantize entry point)
enum NormKind : int { kRms = 0, kLn = 1, kIdentity = 2 };

// quantization variants of the row-wise forward kernel
enum FwdQuant : int {
  kQNone = 0,       // bf16 or fp32 output
  kQDelayed = 1,    // E4M3 with a given scale, + amax
  kQCurAmax = 2,    // current scaling, pass 1: statistics + amax, no output
  kQCurQuant = 3,   // current scaling, pass 2: quantize with 448/amax
  kQNvfp4 = 4,      // NVFP4, pass 2 (pass 1 is kQCurAmax): E2M1 codes with an
                    // E4M3 scale per 16 elements and S = 448*6/amax
  kQMxRow = 5,      // MXFP8 rowwise blocks only (1x32, E8M0 scales), one pass
};

// NVFP4 pass 2 keeps a table of the 128 element factors S / value(scale
// code) in shared memory
constexpr int kNvTableBytes = 128 * 4;

struct FwdParams {
  const void* x;
  const float* gamma;   // 16-byte aligned
  const float* beta;
  void* out;            // [N, H] (bf16/fp32 or E4M3 codes); NVFP4: [N, H/2]
  uint8_t* scales;      // NVFP4: E4M3 block-scale codes [N, H/16]; kQMxRow: E8M0 [N, H/32]
  float* mu;            // LayerNorm: written (pass 1) or read (kQCurQuant)
  float* rsigma;
  const float* scale;   // kQDelayed
  float* amax;          // kQDelayed, kQCurAmax: reduced into; kQCurQuant: read
  float* scale_inv;     // kQCurQuant, kQNvfp4 (kQDelayed: written by the init kernel)
  float* scale_out;     // kQCurQuant, kQNvfp4
  int N, H;
  float eps;
  int zcg;              // zero-centered gamma
  int out_f32;          // kQNone: 1 = fp32 output, 0 = bf16
  const void* residual; // residual add: the residual [N, H] (x's dtype), or NULL
  void* residual_out;   // residual add: h = x + residual [N, H], or NULL
  int workers;          // worker warps (a multiple of the row group size)
  int Q;                // ring slots; workers / group size <= (Q - 1) rows a slot
  int rps_log2;         // a slot holds 2^rps_log2 adjacent rows (one copy)
  int reverse;          // walk the rows from the last one
};

struct MxParams {
  const void* x;
  const float* gamma;
  const float* beta;
  uint8_t* data;        // rowwise codes [N, H] or NULL
  uint8_t* row_scales;  // [N, H/32]
  uint8_t* col_data;    // [H, N] or NULL
  uint8_t* col_scales;  // [H, N/32]
  float* mu;
  float* rsigma;
  int N, H;
  float eps;
  int zcg;
  int apply_warps;
  int stats_warps;
  int Q;
  int n_tiles;          // N / 32
  int n_tbar;           // ring kernel: tile "ready" barriers (> Q / 32 + 1)
};

struct BwdParams {
  const void* dz;
  const void* x;
  const float* mu;
  const float* rsigma;
  const float* gamma;
  void* dx;
  float* part;          // workspace partials [C][nacc][H]
  int N, H;
  int zcg;
  int chunk_rows;       // rows per dgamma/dbeta partial
  int apply_warps;
  int stats_warps;
  int Q;
  int n_chunks;
};

struct ColReduceParams {
  const float* part;    // [C][nacc][H]
  float* dgamma;
  float* dbeta;
  int H;
  int n_chunks;
  int nacc;
};

// scaled activations (forward with a quantize epilogue, backward)
enum ActKind : int { kActSrelu = 0, kActSwiglu = 1, kActClampedSwiglu = 2 };

struct ActParams {
  const void* x;          // [N, H] (SReLU) or [N, 2H] (gate half, linear half)
  const void* dy;         // backward: [N, H]
  void* out;              // forward: y (bf16 / fp32) or E4M3 codes [N, H];
                          // backward: dx, the shape of x
  uint8_t* row_scales;    // forward MXFP8 (rowwise): E8M0 [N, H/32], else NULL
  const float* scales;    // [N] row scales, or NULL (all 1)
  const float* scale;     // FP8 delayed
  float* amax;            // FP8 modes
  float* scale_inv;       // FP8 current (pass 2)
  float* scale_out;       // FP8 current (pass 2)
  float* dscales;         // backward: [N] or NULL
  int N, H;               // H: output width
  float limit, alpha;     // clamped SwiGLU
  int out_f32;            // forward NONE: fp32 output
};

// launch shape shared by the persistent kernels
struct Launch {
  int work;             // independent work items (tiles / chunks): grid upper bound
  int sms;              // SMs the grid may use (SMs - sm_margin)
  int per_sm;           // CTAs per SM the shared-memory plan was sized for
  int threads;          // consumer threads + one producer warp
  size_t smem;
};

// per-device limits, queried once
struct DeviceInfo {
  int sms;
  int smem_optin;       // per CTA
  int smem_per_sm;      // per SM
};
rn_status device_info(DeviceInfo* out);

// Grid of a persistent kernel: min(work, sms * CTAs per SM), where CTAs per
// SM is the planned count capped by what the kernel's resources allow.
template <class Kernel>
rn_status persistent_grid(Kernel k, const Launch& l, int* grid) {
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, l.threads, l.smem) != cudaSuccess)
    return RN_ERR_CUDA;
  const int per = occ < 1 ? 1 : (occ < l.per_sm ? occ : l.per_sm);
  const long long g = (long long)l.sms * per;
  int n = (int)(g < l.work ? g : l.work);
  *grid = n < 1 ? 1 : n;
  return RN_OK;
}

// launch functions (one per translation unit family)
// row shape of the forward: G warps per row, NC 16-byte chunks per lane;
// one: one row a slot, compiled as such (the planner sets it when it
// groups no rows and the shape has that instantiation)
struct FwdShape {
  int g, nc;
  bool one;
};
// pdl: launch as a programmatic dependent of the previous kernel
rn_status launch_fwd(int nk, bool bf16, const FwdShape& sh, int qmode, const FwdParams& p,
                     const Launch& l, bool pdl, cudaStream_t s);
// the same with a residual add (p.residual, p.residual_out set; no pass 2 of
// current scaling, which reads the stored sum through launch_fwd)
rn_status launch_fwd_res(int nk, bool bf16, const FwdShape& sh, int qmode, const FwdParams& p,
                         const Launch& l, bool pdl, cudaStream_t s);
// one-thread kernel: amax = 0 and, when scale != NULL, scale_inv = 1/scale
rn_status launch_fwd_init(float* amax, const float* scale, float* scale_inv, cudaStream_t s);
rn_status launch_mx(int nk, bool bf16, int ng, const MxParams& p, const Launch& l,
                    cudaStream_t s);
// MXFP8 both directions from boxes of 32 rows x 4 column blocks of 128
// bytes, read twice (statistics, then quantization): 16 worker warps; H a
// multiple of 128 / element size, N of 32; Q = box slots
constexpr int kMxBoxThreads = 32 * 16;
constexpr size_t kMxBoxBytes = 16384;
rn_status launch_mx_box(int nk, bool bf16, const MxParams& p, const Launch& l, cudaStream_t s);
// backward with stats warps: bf16 rows (fp32 rows take the fused kernel);
// the wide shape (one CTA per SM) is compiled for at most 512 threads (128
// registers a thread) and for at most kBwdWideThreads (96 registers), the
// most its planner asks for (16 apply warps, 1 stats warp and the producer
// at H = 16384)
constexpr int kBwdWideThreads512 = 512;
constexpr int kBwdWideThreads = 576;
rn_status launch_bwd(bool ln, bool bf16, int ng, const BwdParams& p, const Launch& l,
                     cudaStream_t s);
// backward without stats or producer warps, fp32 rows of up to 16 warps x
// 32 threads x 16 elements (big: one CTA per SM, up to 16 warps; otherwise
// up to 8 warps, several CTAs per SM)
rn_status launch_bwd_fused(bool ln, bool big, const BwdParams& p, const Launch& l,
                           cudaStream_t s);
rn_status launch_colreduce(const ColReduceParams& p, cudaStream_t s);

// scaled activations; qmode kQNone with p.row_scales set = MXFP8 rowwise;
// sms: SMs the grid may use; pdl: programmatic dependent of the previous kernel
rn_status launch_act_fwd(int act, bool bf16, int qmode, const ActParams& p, int sms, bool pdl,
                         cudaStream_t s);
rn_status launch_act_bwd(int act, bool bf16, const ActParams& p, int sms, cudaStream_t s);

// delayed-scaling history step (one CTA; 1 <= L <= kMaxHistory)
constexpr int kMaxHistory = 1024;
rn_status launch_amax_history(float* hist, int L, const float* amax, float* scale,
                              float* scale_inv, cudaStream_t s);

// device error words, one per translation unit
rn_status read_clear_error_fwd(unsigned* code);
rn_status read_clear_error_fwd_res(unsigned* code);
rn_status read_clear_error_mx(unsigned* code);
rn_status read_clear_error_bwd(unsigned* code);

}  // namespace rn
