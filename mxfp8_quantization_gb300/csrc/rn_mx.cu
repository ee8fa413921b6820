// LayerNorm / RMSNorm forward fused with MXFP8 output quantization: 1x32
// rowwise and 32x1 columnwise blocks, each with an E8M0 shared scale (page
// "Implementation:NVIDIA TransformerEngine PyTorch Ext Normalization",
// section "Description": the fully fused MXFP8 path).
//
// Design (one persistent CTA per SM, warp-specialized, no CTA-wide barrier
// on the row path):
//   producer     one lane streams rows of x into a shared-memory ring with
//                cp.async.bulk ("full" mbarrier per slot);
//   stats warps  take rows in turn: mean / rsigma from shared memory
//                (LayerNorm: two passes), published on the slot's "ready"
//                mbarrier and written to mu / rsigma;
//   apply warps  work on tiles of 32 rows (the height of a column block);
//                every thread owns 8 consecutive columns (gamma / beta in
//                registers):
//       pass A   for every row of the tile: y, the 1x32 row-block maximum (4
//                lanes x 8 columns, 2 shuffle steps), its E8M0 code, the
//                rowwise E4M3 codes; and the running maximum of each of the
//                thread's 8 columns;
//       pass B   the 8 column-block codes, then y again for the 32 rows,
//                quantized with the column scales, in two sweeps of 16 rows;
//                each column's 16 codes of a sweep are packed in registers and
//                written as 16 contiguous bytes of the transposed [H, N]
//                columnwise array;
//   then the tile's 32 slots are released ("empty").
// y is recomputed in pass B from the row still in shared memory (cheaper
// than keeping 32x8 fp32 values per thread), with the same instructions as
// in pass A so both directions quantize identical y32.  Arithmetic is on
// element pairs (f32x2); bf16 inputs enter through the mixed-precision forms.
#include <cuda_runtime.h>

#include "rn_device.cuh"
#include "rn_internal.h"

namespace rn {
namespace {

__device__ unsigned g_err_mx;

// apply + stats warps + the producer: at most 16 warps (128 registers each)
constexpr int kMaxThreads = 16 * 32;
constexpr int kTile = 32;

// y of the 8 columns (four pairs) of chunk v in one row
template <typename TIn, int NK>
__device__ __forceinline__ void y8(const unsigned char* rowp, int v, float mean, float rs,
                                   const float2* g, const float2* b, float2* y) {
  using V = Vec<TIn, 8>;
  const typename V::Raw raw = V::load(rowp, v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (NK == kLn)
      y[i] = fma2(mul2(V::sub(raw, i, mean), splat2(rs)), g[i], b[i]);
    else if constexpr (NK == kRms)
      y[i] = mul2(mul2(V::f32(raw, i), splat2(rs)), g[i]);
    else
      y[i] = V::f32(raw, i);
  }
}

template <typename TIn, int NK>
__global__ void __launch_bounds__(kMaxThreads, 1) rn_mx_kernel(const MxParams p) {
  using V = Vec<TIn, 8>;
  constexpr bool STATS = (NK != kIdentity);
  extern __shared__ __align__(128) unsigned char smem[];
  const int A = p.apply_warps;
  const int S = STATS ? p.stats_warps : 0;
  const int H = p.H;
  const int N = p.N;
  const int nchunks = H >> 3;
  const uint32_t row_bytes = (uint32_t)H * sizeof(TIn);
  const uint32_t Q = (uint32_t)p.Q;

  unsigned char* ring = smem;
  float2* rstat = reinterpret_cast<float2*>(smem + (size_t)Q * row_bytes);  // [Q]
  uint64_t* full = reinterpret_cast<uint64_t*>(rstat + Q);
  uint64_t* ready = full + Q;
  uint64_t* empty = ready + Q;

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < Q; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&ready[i]), 1);
      mbar_init(smem_u32(&empty[i]), A);
    }
    fence_barrier_init();
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;

  if (warp == A + S) {
    // ------------------------------------------------------------ producer
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

  if (warp >= A) {
    // --------------------------------------------------------- stats warps
    if constexpr (STATS) {
      const int j = warp - A;
      const float inv_h = 1.0f / (float)H;
      RingPos pos{0u, 0u};
      int q = 0;
      for (int t = blockIdx.x; t < p.n_tiles; t += G) {
        for (int k = 0; k < kTile; ++k, ++q) {
          if (q % S == j) {
            const uint32_t s = pos.slot;
            mbar_wait(smem_u32(&full[s]), pos.phase, &g_err_mx, kErrStatsWait);
            const unsigned char* rowp = ring + (size_t)s * row_bytes;
            float2 a[4];
            float mean = 0.f;
            if constexpr (NK == kLn) {
#pragma unroll
              for (int i = 0; i < 4; ++i) a[i] = make_float2(0.f, 0.f);
              for (int c = lane; c < nchunks; c += 32) {
                const typename V::Raw raw = V::load(rowp, c);
#pragma unroll
                for (int i = 0; i < 4; ++i) V::acc(a[i], raw, i);
              }
              mean = warp_sum((a[0].x + a[0].y) + (a[1].x + a[1].y) + (a[2].x + a[2].y) +
                              (a[3].x + a[3].y)) * inv_h;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = make_float2(0.f, 0.f);
            for (int c = lane; c < nchunks; c += 32) {
              const typename V::Raw raw = V::load(rowp, c);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                if constexpr (NK == kLn) {
                  const float2 d = V::sub(raw, i, mean);
                  a[i] = fma2(d, d, a[i]);
                } else {
                  V::sq_acc(a[i], raw, i);
                }
              }
            }
            const float m2 = warp_sum((a[0].x + a[0].y) + (a[1].x + a[1].y) + (a[2].x + a[2].y) +
                                      (a[3].x + a[3].y));
            const float rs = __frsqrt_rn(m2 * inv_h + p.eps);
            if (lane == 0) {
              const int r = t * kTile + k;
              rstat[s] = make_float2(mean, rs);
              if (NK == kLn) p.mu[r] = mean;
              p.rsigma[r] = rs;
              mbar_arrive(smem_u32(&ready[s]));
            }
          }
          pos.advance(1, Q);
        }
      }
    }
    return;
  }

  // ---------------------------------------------------------- apply warps
  const int t = threadIdx.x;
  const int v = t;  // this thread's chunk of 8 columns
  const bool valid = v < nchunks;
  float2 g2[4], b2[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    g2[i] = make_float2(0.f, 0.f);
    b2[i] = make_float2(0.f, 0.f);
    if (NK != kIdentity && valid) {
      const int c = v * 8 + 2 * i;
      const float ga = p.gamma[c], gb = p.gamma[c + 1];
      g2[i] = p.zcg ? make_float2(1.0f + ga, 1.0f + gb) : make_float2(ga, gb);
      if (NK == kLn && p.beta) b2[i] = make_float2(p.beta[c], p.beta[c + 1]);
    }
  }
  const int hs = H >> 5;   // row scales per row
  const int ns = N >> 5;   // column scales per column

  RingPos pos{0u, 0u};
  for (int tile = blockIdx.x; tile < p.n_tiles; tile += G) {
    const int r0 = tile * kTile;
    const uint32_t slot0 = pos.slot;
    // ------------------------------------------------------------ pass A
    float cm[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) cm[i] = 0.f;
    {
      RingPos rp = pos;
      for (int k = 0; k < kTile; k += 2) {
        float2 y[2][4];
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          const uint32_t s = rp.slot;
          mbar_wait(smem_u32(&full[s]), rp.phase, &g_err_mx, kErrFullWait);
          float mean = 0.f, rs = 1.f;
          if constexpr (STATS) {
            mbar_wait(smem_u32(&ready[s]), rp.phase, &g_err_mx, kErrReadyWait);
            const float2 m = rstat[s];
            mean = m.x;
            rs = m.y;
          }
          rp.advance(1, Q);
#pragma unroll
          for (int i = 0; i < 4; ++i) y[kk][i] = make_float2(0.f, 0.f);
          if (valid) y8<TIn, NK>(ring + (size_t)s * row_bytes, v, mean, rs, g2, b2, y[kk]);
          if (p.data != nullptr) {
            float m = amax_acc2(amax_acc2(0.f, y[kk][0]), y[kk][1]);
            m = amax_acc2(amax_acc2(m, y[kk][2]), y[kk][3]);
            uint32_t mb = abs_bits(m);
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
            const uint32_t code = e8m0_code(__uint_as_float(mb));
            const float2 inv = splat2(e8m0_inv_scale(code));
            if (valid) {
              const size_t row = (size_t)(r0 + k + kk);
              uint32_t c[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 q = mul2(y[kk][i], inv);
                c[i] = pack_e4m3x2(q.x, q.y);
              }
              *reinterpret_cast<uint2*>(p.data + row * H + (size_t)v * 8) =
                  make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
              if ((t & 3) == 0) p.row_scales[row * hs + (v >> 2)] = (uint8_t)code;
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          cm[2 * i] = amax_acc2(cm[2 * i], make_float2(y[0][i].x, y[1][i].x));
          cm[2 * i + 1] = amax_acc2(cm[2 * i + 1], make_float2(y[0][i].y, y[1][i].y));
        }
      }
    }
    // ------------------------------------------------------------ pass B
    if (p.col_data != nullptr) {
      uint32_t ccode[8];
      float cinv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ccode[i] = e8m0_code(cm[i]);
        cinv[i] = e8m0_inv_scale(ccode[i]);
      }
      // two sweeps of 16 rows; each row's y is formed once for all 8 columns
#pragma unroll
      for (int sweep = 0; sweep < 2; ++sweep) {
        uint32_t cq[8][4];  // [column][word]: codes of rows 16*sweep + 4*word .. +3
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          float2 q[4][4];  // [row][pair] scaled by the column scales
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int k = 16 * sweep + 4 * k4 + kk;
            uint32_t s = slot0 + (uint32_t)k;
            s = s >= Q ? s - Q : s;
            float mean = 0.f, rs = 1.f;
            if constexpr (STATS) {
              const float2 m = rstat[s];
              mean = m.x;
              rs = m.y;
            }
            float2 y[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                           make_float2(0.f, 0.f)};
            if (valid) y8<TIn, NK>(ring + (size_t)s * row_bytes, v, mean, rs, g2, b2, y);
#pragma unroll
            for (int i = 0; i < 4; ++i) q[kk][i] = mul2(y[i], make_float2(cinv[2 * i], cinv[2 * i + 1]));
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            cq[2 * i][k4] = pack_e4m3x2(q[0][i].x, q[1][i].x) | (pack_e4m3x2(q[2][i].x, q[3][i].x) << 16);
            cq[2 * i + 1][k4] = pack_e4m3x2(q[0][i].y, q[1][i].y) | (pack_e4m3x2(q[2][i].y, q[3][i].y) << 16);
          }
        }
        if (valid) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const size_t col = (size_t)v * 8 + i;
            *reinterpret_cast<uint4*>(p.col_data + col * N + (size_t)r0 + 16 * sweep) =
                make_uint4(cq[i][0], cq[i][1], cq[i][2], cq[i][3]);
          }
        }
      }
      if (valid) {
#pragma unroll
        for (int i = 0; i < 8; ++i) p.col_scales[((size_t)v * 8 + i) * ns + tile] = (uint8_t)ccode[i];
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

template <typename TIn, int NK>
rn_status launch_t(const MxParams& p, const Launch& l, cudaStream_t s) {
  auto k = rn_mx_kernel<TIn, NK>;
  if (l.threads > kMaxThreads) return RN_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l.smem) !=
      cudaSuccess)
    return RN_ERR_CUDA;
  int grid = 1;
  if (persistent_grid(k, l, &grid) != RN_OK) return RN_ERR_CUDA;
  k<<<grid, l.threads, l.smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

}  // namespace

rn_status launch_mx(int nk, bool bf16, int ng, const MxParams& p, const Launch& l,
                    cudaStream_t s) {
  (void)ng;
  if (nk == kIdentity) return bf16 ? RN_ERR_UNSUPPORTED : launch_t<float, kIdentity>(p, l, s);
  if (bf16) return nk == kLn ? launch_t<uint16_t, kLn>(p, l, s) : launch_t<uint16_t, kRms>(p, l, s);
  return nk == kLn ? launch_t<float, kLn>(p, l, s) : launch_t<float, kRms>(p, l, s);
}

rn_status read_clear_error_mx(unsigned* code) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_mx, sizeof(v)) != cudaSuccess) return RN_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_err_mx, &zero, sizeof(zero)) != cudaSuccess) return RN_ERR_CUDA;
  *code = v;
  return RN_OK;
}

}  // namespace rn
