// LayerNorm / RMSNorm forward fused with MXFP8 output quantization: 1x32
// rowwise and 32x1 columnwise blocks, each with an E8M0 shared scale (page
// "Implementation:NVIDIA TransformerEngine PyTorch Ext Normalization",
// section "Description": the fully fused MXFP8 path).
//
// Design (one persistent CTA per SM, warp-specialized like the row-wise
// forward): the producer lane streams rows of x into a shared-memory ring
// with cp.async.bulk; the CTA works on tiles of 32 rows (the height of a
// column block):
//   phase 1  one warp per row: mean / rsigma from shared memory;
//   phase 2  each consumer thread owns 4 consecutive columns (gamma / beta in
//            registers):
//            pass A  for every row of the tile: y, the 1x32 row-block maximum
//                    (8 lanes x 4 columns, 3 shuffle steps), its E8M0 code,
//                    the rowwise E4M3 codes; and the running maximum of each
//                    of the thread's 4 columns;
//            pass B  the 4 column-block codes, then y again for the 32 rows,
//                    quantized with the column scales; each column's 32 codes
//                    are packed in registers and written as 32 contiguous
//                    bytes of the transposed [H, N] columnwise array.
// y is recomputed in pass B from the bf16/fp32 row still in shared memory
// (cheaper than keeping 32x4 fp32 values per thread), with the same
// instructions as in pass A so both directions quantize identical y32.
#include <cuda_runtime.h>

#include "rn_device.cuh"
#include "rn_internal.h"

namespace rn {
namespace {

__device__ unsigned g_err_mx;

constexpr int kMaxThreads = 512 + 32;
constexpr int kTile = 32;

template <typename TIn>
__device__ __forceinline__ void load4(const unsigned char* rowp, int v, float* f);

template <>
__device__ __forceinline__ void load4<uint16_t>(const unsigned char* rowp, int v, float* f) {
  bf16x4_to_f32(*reinterpret_cast<const uint2*>(rowp + (size_t)v * 8), f);
}

template <>
__device__ __forceinline__ void load4<float>(const unsigned char* rowp, int v, float* f) {
  const float4 a = *reinterpret_cast<const float4*>(rowp + (size_t)v * 16);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
}

template <int NK>
__device__ __forceinline__ void apply4(float* y, float mean, float rs, const float* g,
                                       const float* b) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (NK == kLn)
      y[i] = fmaf((y[i] - mean) * rs, g[i], b[i]);
    else if constexpr (NK == kRms)
      y[i] = (y[i] * rs) * g[i];
  }
}

template <typename TIn, int NG, int NK>
__global__ void __launch_bounds__(kMaxThreads, 1) rn_mx_kernel(const MxParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int TH = blockDim.x - 32;
  const int W = TH >> 5;
  const int H = p.H;
  const int N = p.N;
  const int nchunks = H >> 2;
  const uint32_t row_bytes = (uint32_t)H * sizeof(TIn);
  const int Q = p.Q;

  unsigned char* ring = smem;
  float2* stats = reinterpret_cast<float2*>(smem + (size_t)Q * row_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(stats + 2 * kTile);
  uint64_t* empty = full + Q;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Q; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), W);
    }
    fence_barrier_init();
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;

  if (warp == W) {
    if (lane == 0) {
      const unsigned char* xb = static_cast<const unsigned char*>(p.x);
      uint32_t q = 0;
      for (int t = blockIdx.x; t < p.n_tiles; t += G) {
        for (int k = 0; k < kTile; ++k, ++q) {
          const int r = t * kTile + k;
          const uint32_t s = q % Q, use = q / Q;
          if (use > 0) mbar_wait(smem_u32(&empty[s]), (use - 1) & 1, &g_err_mx, kErrEmptyWait);
          mbar_arrive_expect_tx(smem_u32(&full[s]), row_bytes);
          bulk_g2s(smem_u32(ring + (size_t)s * row_bytes), xb + (size_t)r * row_bytes, row_bytes,
                   smem_u32(&full[s]));
        }
      }
      for (uint32_t k = q > (uint32_t)Q ? q - Q : 0; k < q; ++k)
        mbar_wait(smem_u32(&full[k % Q]), (k / Q) & 1, &g_err_mx, kErrDrainWait);
    }
    return;
  }

  const int t = threadIdx.x;
  float gv[NG][4], bv[NG][4];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int v = g * TH + t;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      gv[g][i] = 0.f;
      bv[g][i] = 0.f;
      if (NK != kIdentity && v < nchunks) {
        const float gam = p.gamma[v * 4 + i];
        gv[g][i] = p.zcg ? 1.0f + gam : gam;
        if (NK == kLn && p.beta) bv[g][i] = p.beta[v * 4 + i];
      }
    }
  }
  const float hf = (float)H;
  const int hs = H >> 5;   // row scales per row
  const int ns = N >> 5;   // column scales per column

  uint32_t q = 0;
  int it = 0;
  for (int tile = blockIdx.x; tile < p.n_tiles; tile += G, ++it) {
    const int r0 = tile * kTile;
    float2* st = stats + (it & 1) * kTile;

    // every consumer warp waits for all 32 rows of the tile once
    for (int k = 0; k < kTile; ++k) {
      const uint32_t qq = q + k;
      mbar_wait(smem_u32(&full[qq % Q]), (qq / Q) & 1, &g_err_mx, kErrFullWait);
    }

    if constexpr (NK != kIdentity) {
      for (int k = warp; k < kTile; k += W) {
        const unsigned char* rowp = ring + (size_t)((q + k) % Q) * row_bytes;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        float mean = 0.f;
        if constexpr (NK == kLn) {
          for (int c = lane; c < nchunks; c += 32) {
            float xf[4];
            load4<TIn>(rowp, c, xf);
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] += xf[i];
          }
          mean = __fdiv_rn(warp_sum((acc[0] + acc[2]) + (acc[1] + acc[3])), hf);
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i] = 0.f;
        }
        for (int c = lane; c < nchunks; c += 32) {
          float xf[4];
          load4<TIn>(rowp, c, xf);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float d = (NK == kLn) ? xf[i] - mean : xf[i];
            acc[i] = fmaf(d, d, acc[i]);
          }
        }
        const float var = __fdiv_rn(warp_sum((acc[0] + acc[2]) + (acc[1] + acc[3])), hf);
        const float rs = __frsqrt_rn(var + p.eps);
        if (lane == 0) {
          st[k] = make_float2(mean, rs);
          if (NK == kLn) p.mu[r0 + k] = mean;
          p.rsigma[r0 + k] = rs;
        }
      }
      consumer_sync(TH);
    }

#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const int v = g * TH + t;
      const bool valid = v < nchunks;
      float cmax[4] = {0.f, 0.f, 0.f, 0.f};
      // ------------------------------------------------------------ pass A
      for (int k = 0; k < kTile; ++k) {
        const unsigned char* rowp = ring + (size_t)((q + k) % Q) * row_bytes;
        float mean = 0.f, rs = 1.f;
        if constexpr (NK != kIdentity) {
          const float2 m = st[k];
          mean = m.x;
          rs = m.y;
        }
        float y[4] = {0.f, 0.f, 0.f, 0.f};
        if (valid) {
          load4<TIn>(rowp, v, y);
          apply4<NK>(y, mean, rs, gv[g], bv[g]);
        }
        if (p.data != nullptr) {
          float m = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) m = amax_acc(m, y[i]);
          uint32_t mb = abs_bits(m);
          mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
          mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
          mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 4));
          const uint32_t code = e8m0_code(__uint_as_float(mb));
          const float inv = e8m0_inv_scale(code);
          if (valid) {
            const size_t row = (size_t)(r0 + k);
            *reinterpret_cast<uint32_t*>(p.data + row * H + (size_t)v * 4) =
                pack_e4m3x4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv);
            if ((t & 7) == 0) p.row_scales[row * hs + (v >> 3)] = (uint8_t)code;
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) cmax[i] = amax_acc(cmax[i], y[i]);
      }
      // ------------------------------------------------------------ pass B
      if (p.col_data != nullptr) {
        float cinv[4];
        uint32_t ccode[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ccode[i] = e8m0_code(cmax[i]);
          cinv[i] = e8m0_inv_scale(ccode[i]);
        }
        uint32_t cq[4][8];
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {
          float y4[4][4];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int k = 4 * k4 + kk;
            const unsigned char* rowp = ring + (size_t)((q + k) % Q) * row_bytes;
            float mean = 0.f, rs = 1.f;
            if constexpr (NK != kIdentity) {
              const float2 m = st[k];
              mean = m.x;
              rs = m.y;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) y4[kk][i] = 0.f;
            if (valid) {
              load4<TIn>(rowp, v, y4[kk]);
              apply4<NK>(y4[kk], mean, rs, gv[g], bv[g]);
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
            cq[i][k4] = pack_e4m3x4(y4[0][i] * cinv[i], y4[1][i] * cinv[i], y4[2][i] * cinv[i],
                                    y4[3][i] * cinv[i]);
        }
        if (valid) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const size_t col = (size_t)v * 4 + i;
            uint4* dst = reinterpret_cast<uint4*>(p.col_data + col * N + (size_t)r0);
            dst[0] = make_uint4(cq[i][0], cq[i][1], cq[i][2], cq[i][3]);
            dst[1] = make_uint4(cq[i][4], cq[i][5], cq[i][6], cq[i][7]);
            p.col_scales[col * ns + tile] = (uint8_t)ccode[i];
          }
        }
      }
    }
    // release the tile's slots
    __syncwarp();
    if (lane == 0)
      for (int k = 0; k < kTile; ++k) mbar_arrive(smem_u32(&empty[(q + k) % Q]));
    q += kTile;
  }
}

template <typename TIn, int NG, int NK>
rn_status launch_t(const MxParams& p, const Launch& l, cudaStream_t s) {
  auto k = rn_mx_kernel<TIn, NG, NK>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l.smem) !=
      cudaSuccess)
    return RN_ERR_CUDA;
  k<<<l.grid, l.threads, l.smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

template <typename TIn, int NK>
rn_status launch_ng(int ng, const MxParams& p, const Launch& l, cudaStream_t s) {
  switch (ng) {
    case 1: return launch_t<TIn, 1, NK>(p, l, s);
    case 2: return launch_t<TIn, 2, NK>(p, l, s);
    default: return RN_ERR_UNSUPPORTED;
  }
}

}  // namespace

rn_status launch_mx(int nk, bool bf16, int ng, const MxParams& p, const Launch& l,
                    cudaStream_t s) {
  if (nk == kIdentity) return bf16 ? RN_ERR_UNSUPPORTED : launch_ng<float, kIdentity>(ng, p, l, s);
  if (bf16)
    return nk == kLn ? launch_ng<uint16_t, kLn>(ng, p, l, s) : launch_ng<uint16_t, kRms>(ng, p, l, s);
  return nk == kLn ? launch_ng<float, kLn>(ng, p, l, s) : launch_ng<float, kRms>(ng, p, l, s);
}

rn_status read_clear_error_mx(unsigned* code) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_mx, sizeof(v)) != cudaSuccess) return RN_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_err_mx, &zero, sizeof(zero)) != cudaSuccess) return RN_ERR_CUDA;
  *code = v;
  return RN_OK;
}

}  // namespace rn
