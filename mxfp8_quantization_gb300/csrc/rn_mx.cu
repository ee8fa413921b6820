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
// Arithmetic is on element pairs (f32x2); bf16 inputs enter through the
// mixed-precision forms.
#include <cuda_runtime.h>

#include "rn_device.cuh"
#include "rn_internal.h"

namespace rn {
namespace {

__device__ unsigned g_err_mx;

constexpr int kMaxThreads = 512 + 32;
constexpr int kTile = 32;

// y of the 4 columns (two pairs) of chunk v in one row
template <typename TIn, int NK>
__device__ __forceinline__ void y4(const unsigned char* rowp, int v, float mean, float rs,
                                   const float2* g, const float2* b, float2* y) {
  using V = Vec<TIn, 4>;
  const typename V::Raw raw = V::load(rowp, v);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if constexpr (NK == kLn)
      y[i] = fma2(mul2(V::sub(raw, i, mean), splat2(rs)), g[i], b[i]);
    else if constexpr (NK == kRms)
      y[i] = mul2(mul2(V::f32(raw, i), splat2(rs)), g[i]);
    else
      y[i] = V::f32(raw, i);
  }
}

template <typename TIn, int NG, int NK>
__global__ void __launch_bounds__(kMaxThreads, 1) rn_mx_kernel(const MxParams p) {
  using V = Vec<TIn, 4>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int TH = blockDim.x - 32;
  const int W = TH >> 5;
  const int H = p.H;
  const int N = p.N;
  const int nchunks = H >> 2;
  const uint32_t row_bytes = (uint32_t)H * sizeof(TIn);
  const uint32_t Q = (uint32_t)p.Q;

  unsigned char* ring = smem;
  float2* stats = reinterpret_cast<float2*>(smem + (size_t)Q * row_bytes);  // [2][32]
  uint64_t* full = reinterpret_cast<uint64_t*>(stats + 2 * kTile);
  uint64_t* empty = full + Q;

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < Q; ++i) {
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
      RingPos pos{0u, 0u};
      uint32_t issued = 0;
      for (int t = blockIdx.x; t < p.n_tiles; t += G) {
        for (int k = 0; k < kTile; ++k, ++issued) {
          const int r = t * kTile + k;
          const uint32_t s = pos.slot;
          if (issued >= Q) mbar_wait(smem_u32(&empty[s]), pos.phase ^ 1u, &g_err_mx, kErrEmptyWait);
          mbar_arrive_expect_tx(smem_u32(&full[s]), row_bytes);
          bulk_g2s(smem_u32(ring + (size_t)s * row_bytes), xb + (size_t)r * row_bytes, row_bytes,
                   smem_u32(&full[s]));
          pos.advance(1, Q);
        }
      }
      const uint32_t first = issued > Q ? issued - Q : 0;
      for (uint32_t k = first; k < issued; ++k)
        mbar_wait(smem_u32(&full[k % Q]), (k / Q) & 1u, &g_err_mx, kErrDrainWait);
    }
    return;
  }

  const int t = threadIdx.x;
  float2 g2[NG][2], b2[NG][2];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int v = g * TH + t;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      g2[g][i] = make_float2(0.f, 0.f);
      b2[g][i] = make_float2(0.f, 0.f);
      if (NK != kIdentity && v < nchunks) {
        const int c = v * 4 + 2 * i;
        const float ga = p.gamma[c], gb = p.gamma[c + 1];
        g2[g][i] = p.zcg ? make_float2(1.0f + ga, 1.0f + gb) : make_float2(ga, gb);
        if (NK == kLn && p.beta) b2[g][i] = make_float2(p.beta[c], p.beta[c + 1]);
      }
    }
  }
  const float hf = (float)H;
  const int hs = H >> 5;   // row scales per row
  const int ns = N >> 5;   // column scales per column

  RingPos pos{0u, 0u};
  int it = 0;
  for (int tile = blockIdx.x; tile < p.n_tiles; tile += G, ++it) {
    const int r0 = tile * kTile;
    float2* st = stats + (it & 1) * kTile;
    // the ring slot of each row of the tile: slot0 + k, wrapping once
    const uint32_t slot0 = pos.slot;
    auto slot_of = [&](int k) -> uint32_t {
      const uint32_t s = slot0 + (uint32_t)k;
      return s >= Q ? s - Q : s;
    };

    // every consumer warp waits for all 32 rows of the tile once
    {
      RingPos rp = pos;
      for (int k = 0; k < kTile; ++k) {
        mbar_wait(smem_u32(&full[rp.slot]), rp.phase, &g_err_mx, kErrFullWait);
        rp.advance(1, Q);
      }
    }

    if constexpr (NK != kIdentity) {
      for (int k = warp; k < kTile; k += W) {
        const unsigned char* rowp = ring + (size_t)slot_of(k) * row_bytes;
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
        float mean = 0.f;
        if constexpr (NK == kLn) {
          for (int c = lane; c < nchunks; c += 32) {
            const typename V::Raw raw = V::load(rowp, c);
            V::acc(a0, raw, 0);
            V::acc(a1, raw, 1);
          }
          mean = __fdiv_rn(warp_sum((a0.x + a0.y) + (a1.x + a1.y)), hf);
          a0 = a1 = make_float2(0.f, 0.f);
        }
        for (int c = lane; c < nchunks; c += 32) {
          const typename V::Raw raw = V::load(rowp, c);
          if constexpr (NK == kLn) {
            const float2 d0 = V::sub(raw, 0, mean), d1 = V::sub(raw, 1, mean);
            a0 = fma2(d0, d0, a0);
            a1 = fma2(d1, d1, a1);
          } else {
            V::sq_acc(a0, raw, 0);
            V::sq_acc(a1, raw, 1);
          }
        }
        const float var = __fdiv_rn(warp_sum((a0.x + a0.y) + (a1.x + a1.y)), hf);
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
      float cm[4] = {0.f, 0.f, 0.f, 0.f};
      // ------------------------------------------------------------ pass A
      for (int k = 0; k < kTile; k += 2) {
        float2 y[2][2];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          float mean = 0.f, rs = 1.f;
          if constexpr (NK != kIdentity) {
            const float2 m = st[k + kk];
            mean = m.x;
            rs = m.y;
          }
          y[kk][0] = y[kk][1] = make_float2(0.f, 0.f);
          if (valid)
            y4<TIn, NK>(ring + (size_t)slot_of(k + kk) * row_bytes, v, mean, rs, g2[g], b2[g], y[kk]);
          if (p.data != nullptr) {
            uint32_t mb = abs_bits(amax_acc2(amax_acc2(0.f, y[kk][0]), y[kk][1]));
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 4));
            const uint32_t code = e8m0_code(__uint_as_float(mb));
            const float2 inv = splat2(e8m0_inv_scale(code));
            if (valid) {
              const size_t row = (size_t)(r0 + k + kk);
              const float2 q0 = mul2(y[kk][0], inv), q1 = mul2(y[kk][1], inv);
              *reinterpret_cast<uint32_t*>(p.data + row * H + (size_t)v * 4) =
                  pack_e4m3x2(q0.x, q0.y) | (pack_e4m3x2(q1.x, q1.y) << 16);
              if ((t & 7) == 0) p.row_scales[row * hs + (v >> 3)] = (uint8_t)code;
            }
          }
        }
        cm[0] = amax_acc2(cm[0], make_float2(y[0][0].x, y[1][0].x));
        cm[1] = amax_acc2(cm[1], make_float2(y[0][0].y, y[1][0].y));
        cm[2] = amax_acc2(cm[2], make_float2(y[0][1].x, y[1][1].x));
        cm[3] = amax_acc2(cm[3], make_float2(y[0][1].y, y[1][1].y));
      }
      // ------------------------------------------------------------ pass B
      if (p.col_data != nullptr) {
        uint32_t ccode[4];
        float cinv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ccode[i] = e8m0_code(cm[i]);
          cinv[i] = e8m0_inv_scale(ccode[i]);
        }
        const float2 ci01 = make_float2(cinv[0], cinv[1]), ci23 = make_float2(cinv[2], cinv[3]);
        uint32_t cq[4][8];
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {
          float2 q[4][2];  // [row][pair] scaled by the column scales
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int k = 4 * k4 + kk;
            float mean = 0.f, rs = 1.f;
            if constexpr (NK != kIdentity) {
              const float2 m = st[k];
              mean = m.x;
              rs = m.y;
            }
            float2 y[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            if (valid)
              y4<TIn, NK>(ring + (size_t)slot_of(k) * row_bytes, v, mean, rs, g2[g], b2[g], y);
            q[kk][0] = mul2(y[0], ci01);
            q[kk][1] = mul2(y[1], ci23);
          }
          cq[0][k4] = pack_e4m3x2(q[0][0].x, q[1][0].x) | (pack_e4m3x2(q[2][0].x, q[3][0].x) << 16);
          cq[1][k4] = pack_e4m3x2(q[0][0].y, q[1][0].y) | (pack_e4m3x2(q[2][0].y, q[3][0].y) << 16);
          cq[2][k4] = pack_e4m3x2(q[0][1].x, q[1][1].x) | (pack_e4m3x2(q[2][1].x, q[3][1].x) << 16);
          cq[3][k4] = pack_e4m3x2(q[0][1].y, q[1][1].y) | (pack_e4m3x2(q[2][1].y, q[3][1].y) << 16);
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
    if (lane == 0) {
      RingPos rp = pos;
      for (int k = 0; k < kTile; ++k) {
        mbar_arrive(smem_u32(&empty[rp.slot]));
        rp.advance(1, Q);
      }
    }
    pos.advance(kTile, Q);
  }
}

template <typename TIn, int NG, int NK>
rn_status launch_t(const MxParams& p, const Launch& l, cudaStream_t s) {
  auto k = rn_mx_kernel<TIn, NG, NK>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l.smem) !=
      cudaSuccess)
    return RN_ERR_CUDA;
  int grid = 1;
  if (persistent_grid(k, l, &grid) != RN_OK) return RN_ERR_CUDA;
  k<<<grid, l.threads, l.smem, s>>>(p);
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
