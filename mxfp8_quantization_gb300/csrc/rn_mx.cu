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
//   apply warps  work on tiles of 32 rows (the height of a column block),
//                each warp on 64-column sub-tiles: every thread holds y for
//                an 8-row x 8-column block in registers, computed once
//                (gamma / beta for its columns from the L1-cached global
//                copies).  From those registers it forms
//       rowwise  the 1x32 row-block maxima (4 lanes, 2 shuffle steps), their
//                E8M0 codes and the rowwise E4M3 codes;
//       colwise  the 32x1 column-block maxima (4 row groups, 2 shuffle
//                steps), their codes, and the columnwise codes, 8 per column
//                per thread, stored as 8 contiguous bytes of the transposed
//                [H, N] array;
//   then the tile's 32 slots are released ("empty").
// Both directions quantize the same y32 (one computation per element).
// Arithmetic is on element pairs (f32x2); bf16 inputs enter through the
// mixed-precision forms.
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
            // not paced by the apply warps: wait for the previous use of the
            // slot to be released first, so that the parity wait below
            // cannot match a phase one lap old (stats warps < slots)
            if (q >= (int)Q) mbar_wait(smem_u32(&empty[s]), pos.phase ^ 1u, &g_err_mx, kErrStatsWait);
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
  // Each apply warp takes 64-column sub-tiles of the 32-row tile (w, w + A,
  // ...).  Lane = hb*16 + rg*4 + cc: the thread holds y of rows 8rg..8rg+7
  // and columns 64*sub + 32*hb + 8*cc .. +7 in registers.  A row block (32
  // columns) spans the 4 lanes cc = 0..3 (shuffles xor 1, 2); a column block
  // (32 rows) spans the 4 lanes rg = 0..3 (shuffles xor 4, 8).
  const int hb = lane >> 4, rg = (lane >> 2) & 3, cc = lane & 3;
  const int nsub = (nchunks + 7) >> 3;
  const int hs = H >> 5;   // row scales per row
  const int ns = N >> 5;   // column scales per column

  RingPos pos{0u, 0u};
  for (int tile = blockIdx.x; tile < p.n_tiles; tile += G) {
    const int r0 = tile * kTile;
    // the whole warp waits for the tile's 32 rows (warp-uniform waits; "ready"
    // implies the row has landed)
    {
      RingPos rp = pos;
      for (int k = 0; k < kTile; ++k) {
        if constexpr (STATS)
          mbar_wait(smem_u32(&ready[rp.slot]), rp.phase, &g_err_mx, kErrReadyWait);
        else
          mbar_wait(smem_u32(&full[rp.slot]), rp.phase, &g_err_mx, kErrFullWait);
        rp.advance(1, Q);
      }
    }
    uint32_t slot[8];
    float2 st8[8];
    {
      RingPos rp = pos.ahead(8 * rg, Q);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        slot[j] = rp.slot;
        st8[j] = STATS ? rstat[rp.slot] : make_float2(0.f, 1.f);
        rp.advance(1, Q);
      }
    }
    for (int sub = warp; sub < nsub; sub += A) {
      const int v = sub * 8 + hb * 4 + cc;  // chunk of 8 columns
      const bool valid = v < nchunks;
      float2 g2[4], b2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        g2[i] = make_float2(0.f, 0.f);
        b2[i] = make_float2(0.f, 0.f);
        if (NK != kIdentity && valid) {
          const int c = v * 8 + 2 * i;
          const float ga = __ldg(p.gamma + c), gb = __ldg(p.gamma + c + 1);
          g2[i] = p.zcg ? make_float2(1.0f + ga, 1.0f + gb) : make_float2(ga, gb);
          if (NK == kLn && p.beta) b2[i] = make_float2(__ldg(p.beta + c), __ldg(p.beta + c + 1));
        }
      }
      float2 y[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int i = 0; i < 4; ++i) y[j][i] = make_float2(0.f, 0.f);
        if (valid) y8<TIn, NK>(ring + (size_t)slot[j] * row_bytes, v, st8[j].x, st8[j].y, g2, b2, y[j]);
      }
      // ------------------------------------------------- rowwise 1x32 blocks
      if (p.data != nullptr) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float m = amax_acc2(amax_acc2(0.f, y[j][0]), y[j][1]);
          m = amax_acc2(amax_acc2(m, y[j][2]), y[j][3]);
          uint32_t mb = abs_bits(m);
          mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
          mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
          const uint32_t code = e8m0_code(__uint_as_float(mb));
          const float2 inv = splat2(e8m0_inv_scale(code));
          if (valid) {
            const size_t row = (size_t)(r0 + 8 * rg + j);
            uint32_t c[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 q = mul2(y[j][i], inv);
              c[i] = pack_e4m3x2(q.x, q.y);
            }
            *reinterpret_cast<uint2*>(p.data + row * H + (size_t)v * 8) =
                make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
            if (cc == 0) p.row_scales[row * hs + (v >> 2)] = (uint8_t)code;
          }
        }
      }
      // ---------------------------------------------- columnwise 32x1 blocks
      if (p.col_data != nullptr) {
        float cm[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float a = 0.f, b = 0.f;
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            a = amax_acc2(a, make_float2(y[j][i].x, y[j + 1][i].x));
            b = amax_acc2(b, make_float2(y[j][i].y, y[j + 1][i].y));
          }
          cm[2 * i] = a;
          cm[2 * i + 1] = b;
        }
        float cinv[8];
        uint32_t ccode[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t mb = abs_bits(cm[c]);
          mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 4));
          mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 8));
          ccode[c] = e8m0_code(__uint_as_float(mb));
          cinv[c] = e8m0_inv_scale(ccode[c]);
        }
        if (valid) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 ci = make_float2(cinv[2 * i], cinv[2 * i + 1]);
            float2 q[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) q[j] = mul2(y[j][i], ci);
            const uint32_t lo0 = pack_e4m3x2(q[0].x, q[1].x) | (pack_e4m3x2(q[2].x, q[3].x) << 16);
            const uint32_t hi0 = pack_e4m3x2(q[4].x, q[5].x) | (pack_e4m3x2(q[6].x, q[7].x) << 16);
            const uint32_t lo1 = pack_e4m3x2(q[0].y, q[1].y) | (pack_e4m3x2(q[2].y, q[3].y) << 16);
            const uint32_t hi1 = pack_e4m3x2(q[4].y, q[5].y) | (pack_e4m3x2(q[6].y, q[7].y) << 16);
            const size_t col = (size_t)v * 8 + 2 * i;
            *reinterpret_cast<uint2*>(p.col_data + col * N + (size_t)(r0 + 8 * rg)) = make_uint2(lo0, hi0);
            *reinterpret_cast<uint2*>(p.col_data + (col + 1) * N + (size_t)(r0 + 8 * rg)) =
                make_uint2(lo1, hi1);
          }
          if (rg == 0) {
#pragma unroll
            for (int c = 0; c < 8; ++c) p.col_scales[((size_t)v * 8 + c) * ns + tile] = (uint8_t)ccode[c];
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
