// Row-wise LayerNorm / RMSNorm forward with fused output quantization
// (page "Implementation:NVIDIA TransformerEngine PyTorch Ext Normalization",
// section "Description": the fully fused delayed-scaling path and both
// passes of the norm+amax-then-quantize current-scaling path).
//
// Design (one persistent CTA per SM, warp-specialized):
//   * warp W (the last one) is the producer: one lane streams whole rows of x
//     into a ring of Q shared-memory slots with the bulk-copy engine
//     (cp.async.bulk, completion on a per-slot "full" mbarrier) and refills a
//     slot as soon as every consumer warp has released it ("empty" mbarrier);
//   * consumer warps 0..W-1 take tiles of T rows:
//       phase 1  the row statistics from shared memory: WPR warps share a
//                row (one when rows are short), each taking an interleaved
//                slice of its 16-byte chunks; LayerNorm slices are reduced
//                exactly in two passes (slice mean, then centred sum of
//                squares) and merged in slice order with Chan's pairwise
//                update; RMSNorm slices give sums of squares, added in
//                order; then mu / rsigma are written;
//       phase 2  every consumer thread owns fixed 16-byte column chunks
//                (gamma / beta live in its registers for the whole kernel) and
//                forms y = (x-mu)*rsigma*g + beta (RMSNorm: x*rsigma*g) for
//                each row of the tile, then stores bf16/fp32 or E4M3 codes;
//   * the per-tensor amax is reduced per thread, per CTA, then with one
//     atomicMax on the fp32 bit pattern (ordered like the values for
//     non-negative numbers, NaN above +inf).
// Current scaling runs the kernel twice: pass 1 (statistics + amax, no
// output) and pass 2 (quantize with 448/amax, reading mu/rsigma back), the
// second walking the tiles backwards so that it starts on the rows that
// pass 1 left in L2.
#include <cuda_runtime.h>

#include "rn_device.cuh"
#include "rn_internal.h"

namespace rn {
namespace {

__device__ unsigned g_err_fwd;

constexpr int kMaxThreads = 512 + 32;

template <typename TIn>
struct Chunk;

template <>
struct Chunk<uint16_t> {  // bf16 storage
  static constexpr int VEC = 8;
  __device__ __forceinline__ static void load(const unsigned char* p, int c, float* f) {
    const uint4 v = *reinterpret_cast<const uint4*>(p + (size_t)c * 16);
    bf16x8_to_f32(v, f);
  }
};

template <>
struct Chunk<float> {
  static constexpr int VEC = 4;
  __device__ __forceinline__ static void load(const unsigned char* p, int c, float* f) {
    const float4 v = *reinterpret_cast<const float4*>(p + (size_t)c * 16);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
};

template <int VEC>
__device__ __forceinline__ float tree_sum(const float* a) {
  float s[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) s[i] = a[i];
#pragma unroll
  for (int w = VEC / 2; w > 0; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) s[i] += s[i + w];
  return s[0];
}

// store VEC outputs of one chunk
template <int VEC, int QM>
__device__ __forceinline__ void store_chunk(const FwdParams& p, size_t elem, const float* y,
                                            float scale) {
  if constexpr (QM == kQNone) {
    if (p.out_f32) {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(p.out) + elem);
#pragma unroll
      for (int i = 0; i < VEC / 4; ++i)
        o[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
    } else {
      uint16_t* o = static_cast<uint16_t*>(p.out) + elem;
      if constexpr (VEC == 8) {
        *reinterpret_cast<uint4*>(o) =
            make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                       pack_bf16x2(y[6], y[7]));
      } else {
        *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
      }
    }
  } else {
    uint8_t* o = static_cast<uint8_t*>(p.out) + elem;
    float s[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) s[i] = y[i] * scale;
    if constexpr (VEC == 8) {
      *reinterpret_cast<uint2*>(o) =
          make_uint2(pack_e4m3x4(s[0], s[1], s[2], s[3]), pack_e4m3x4(s[4], s[5], s[6], s[7]));
    } else {
      *reinterpret_cast<uint32_t*>(o) = pack_e4m3x4(s[0], s[1], s[2], s[3]);
    }
  }
}

template <typename TIn, int NG, int NK, int QM>
__global__ void __launch_bounds__(kMaxThreads, 1) rn_fwd_kernel(const FwdParams p) {
  using C = Chunk<TIn>;
  constexpr int VEC = C::VEC;
  constexpr bool LN = (NK == kLn);
  extern __shared__ __align__(128) unsigned char smem[];

  const int TH = blockDim.x - 32;  // consumer threads
  const int W = TH >> 5;           // consumer warps
  const int H = p.H;
  const int nchunks = H / VEC;
  const uint32_t row_bytes = (uint32_t)H * sizeof(TIn);
  const int Q = p.Q;
  const int WPR = p.wpr;

  unsigned char* ring = smem;
  float2* stats = reinterpret_cast<float2*>(smem + (size_t)Q * row_bytes);
  float4* part = reinterpret_cast<float4*>(stats + 2 * p.T);   // [T * WPR]
  uint32_t* red = reinterpret_cast<uint32_t*>(part + p.T * p.wpr);
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 32);
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
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const unsigned char* xb = static_cast<const unsigned char*>(p.x);
      uint32_t q = 0;
      for (int t = blockIdx.x; t < p.n_tiles; t += G) {
        const int tt = p.reverse ? p.n_tiles - 1 - t : t;
        const int r0 = tt * p.T;
        const int r1 = min(r0 + p.T, p.N);
        for (int r = r0; r < r1; ++r, ++q) {
          const uint32_t s = q % Q, use = q / Q;
          if (use > 0) mbar_wait(smem_u32(&empty[s]), (use - 1) & 1, &g_err_fwd, kErrEmptyWait);
          mbar_arrive_expect_tx(smem_u32(&full[s]), row_bytes);
          bulk_g2s(smem_u32(ring + (size_t)s * row_bytes), xb + (size_t)r * row_bytes, row_bytes,
                   smem_u32(&full[s]));
        }
      }
      // every copy this CTA issued must have landed before it exits
      for (uint32_t k = q > (uint32_t)Q ? q - Q : 0; k < q; ++k)
        mbar_wait(smem_u32(&full[k % Q]), (k / Q) & 1, &g_err_fwd, kErrDrainWait);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int t = threadIdx.x;
  float gv[NG][VEC], bv[NG][VEC];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int v = g * TH + t;
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      gv[g][i] = 0.f;
      bv[g][i] = 0.f;
    }
    if (v < nchunks) {
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        if constexpr (NK != kIdentity) {
          const float gam = p.gamma[v * VEC + i];
          gv[g][i] = p.zcg ? 1.0f + gam : gam;
        }
        if constexpr (LN) bv[g][i] = p.beta ? p.beta[v * VEC + i] : 0.0f;
      }
    }
  }

  float scale = 1.0f;
  if constexpr (QM == kQDelayed) scale = *p.scale;
  if constexpr (QM == kQCurQuant) {
    const float am = *p.amax;
    scale = (am == 0.0f) ? 1.0f : __fdiv_rn(448.0f, am);
    if (blockIdx.x == 0 && t == 0) {
      *p.scale_out = scale;
      *p.scale_inv = __fdiv_rn(1.0f, scale);
    }
  }
  if constexpr (QM == kQDelayed) {
    if (blockIdx.x == 0 && t == 0) *p.scale_inv = __fdiv_rn(1.0f, scale);
  }
  float amax_t = 0.0f;
  const float inv_h_num = (float)H;

  uint32_t q = 0;
  int it = 0;
  for (int tk = blockIdx.x; tk < p.n_tiles; tk += G, ++it) {
    const int tt = p.reverse ? p.n_tiles - 1 - tk : tk;
    const int r0 = tt * p.T;
    const int nrows = min(p.T, p.N - r0);
    float2* st = stats + (it & 1) * p.T;

    if constexpr (QM != kQCurQuant && NK != kIdentity) {
      // ---------------------------------------------- phase 1: statistics
      // WPR warps share a row; warp (k, j) takes chunks j*32 + lane + i*32*WPR
      // of row k and leaves (mean, M2, n) of its slice (LayerNorm; exact
      // two-pass within the slice) or its sum of squares (RMSNorm)
      for (int item = warp; item < nrows * WPR; item += W) {
        const int k = item / WPR, j = item - k * WPR;
        const uint32_t qq = q + k;
        const uint32_t s = qq % Q;
        mbar_wait(smem_u32(&full[s]), (qq / Q) & 1, &g_err_fwd, kErrFullWait);
        const unsigned char* rowp = ring + (size_t)s * row_bytes;
        float acc[VEC];
        float smean = 0.0f, cnt = 0.0f;
        if constexpr (LN) {
#pragma unroll
          for (int i = 0; i < VEC; ++i) acc[i] = 0.0f;
          for (int c = j * 32 + lane; c < nchunks; c += 32 * WPR) {
            float xf[VEC];
            C::load(rowp, c, xf);
#pragma unroll
            for (int i = 0; i < VEC; ++i) acc[i] += xf[i];
            cnt += (float)VEC;
          }
          cnt = warp_sum(cnt);
          smean = cnt > 0.0f ? __fdiv_rn(warp_sum(tree_sum<VEC>(acc)), cnt) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[i] = 0.0f;
        for (int c = j * 32 + lane; c < nchunks; c += 32 * WPR) {
          float xf[VEC];
          C::load(rowp, c, xf);
#pragma unroll
          for (int i = 0; i < VEC; ++i) {
            const float d = LN ? xf[i] - smean : xf[i];
            acc[i] = fmaf(d, d, acc[i]);
          }
        }
        const float m2 = warp_sum(tree_sum<VEC>(acc));
        if (lane == 0) part[k * WPR + j] = make_float4(smean, m2, cnt, 0.0f);
      }
      consumer_sync(TH);
      // merge the slices of each row in slice order (Chan et al.)
      if (t < nrows) {
        const int k = t;
        float mean = 0.0f, m2, n;
        const float4 p0 = part[k * WPR];
        if constexpr (LN) {
          mean = p0.x;
          m2 = p0.y;
          n = p0.z;
          for (int j = 1; j < WPR; ++j) {
            const float4 pj = part[k * WPR + j];
            if (pj.z > 0.0f) {
              const float n2 = n + pj.z;
              const float delta = pj.x - mean;
              mean = fmaf(delta, __fdiv_rn(pj.z, n2), mean);
              m2 = m2 + pj.y + delta * delta * __fdiv_rn(n * pj.z, n2);
              n = n2;
            }
          }
        } else {
          m2 = p0.y;
          for (int j = 1; j < WPR; ++j) m2 += part[k * WPR + j].y;
        }
        const float rs = __frsqrt_rn(__fdiv_rn(m2, inv_h_num) + p.eps);
        st[k] = make_float2(mean, rs);
        if constexpr (LN) p.mu[r0 + k] = mean;
        p.rsigma[r0 + k] = rs;
      }
      consumer_sync(TH);
    }

    // ------------------------------------------- phase 2: apply + output
    for (int k = 0; k < nrows; ++k) {
      const uint32_t qq = q + k;
      const uint32_t s = qq % Q;
      mbar_wait(smem_u32(&full[s]), (qq / Q) & 1, &g_err_fwd, kErrFullWait);
      float mean = 0.0f, rs = 1.0f;
      if constexpr (NK == kIdentity) {
      } else if constexpr (QM == kQCurQuant) {
        rs = p.rsigma[r0 + k];
        mean = LN ? p.mu[r0 + k] : 0.0f;
      } else {
        const float2 m = st[k];
        mean = m.x;
        rs = m.y;
      }
      const unsigned char* rowp = ring + (size_t)s * row_bytes;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const int v = g * TH + t;
        if (v < nchunks) {
          float y[VEC];
          C::load(rowp, v, y);
#pragma unroll
          for (int i = 0; i < VEC; ++i) {
            if constexpr (LN)
              y[i] = fmaf((y[i] - mean) * rs, gv[g][i], bv[g][i]);
            else if constexpr (NK == kRms)
              y[i] = (y[i] * rs) * gv[g][i];
          }
          if constexpr (QM == kQDelayed || QM == kQCurAmax) {
#pragma unroll
            for (int i = 0; i < VEC; ++i) amax_t = amax_acc(amax_t, y[i]);
          }
          if constexpr (QM != kQCurAmax)
            store_chunk<VEC, QM>(p, (size_t)(r0 + k) * H + (size_t)v * VEC, y, scale);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
    q += nrows;
  }

  if constexpr (QM == kQDelayed || QM == kQCurAmax) {
    const uint32_t b = warp_umax(abs_bits(amax_t));
    if (lane == 0) red[warp] = b;
    consumer_sync(TH);
    if (t == 0) {
      uint32_t m = 0;
      for (int w = 0; w < W; ++w) m = max(m, red[w]);
      atomicMax(reinterpret_cast<unsigned int*>(p.amax), m);
    }
  }
}

template <typename TIn, int NG, int NK, int QM>
rn_status launch_t(const FwdParams& p, const Launch& l, cudaStream_t s) {
  auto k = rn_fwd_kernel<TIn, NG, NK, QM>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l.smem) !=
      cudaSuccess)
    return RN_ERR_CUDA;
  k<<<l.grid, l.threads, l.smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

template <typename TIn, int NK, int QM>
rn_status launch_ng(int ng, const FwdParams& p, const Launch& l, cudaStream_t s) {
  switch (ng) {
    case 1: return launch_t<TIn, 1, NK, QM>(p, l, s);
    case 2: return launch_t<TIn, 2, NK, QM>(p, l, s);
    case 4: return launch_t<TIn, 4, NK, QM>(p, l, s);
    default: return RN_ERR_UNSUPPORTED;
  }
}

template <typename TIn, int NK>
rn_status launch_q(int ng, int qmode, const FwdParams& p, const Launch& l, cudaStream_t s) {
  switch (qmode) {
    case kQNone:
      if constexpr (NK == kIdentity) return RN_ERR_UNSUPPORTED;
      else return launch_ng<TIn, NK, kQNone>(ng, p, l, s);
    case kQDelayed: return launch_ng<TIn, NK, kQDelayed>(ng, p, l, s);
    case kQCurAmax: return launch_ng<TIn, NK, kQCurAmax>(ng, p, l, s);
    case kQCurQuant: return launch_ng<TIn, NK, kQCurQuant>(ng, p, l, s);
    default: return RN_ERR_INVALID;
  }
}

}  // namespace

rn_status launch_fwd(int nk, bool bf16, int ng, int qmode, const FwdParams& p, const Launch& l,
                     cudaStream_t s) {
  if (nk == kIdentity)
    return bf16 ? RN_ERR_UNSUPPORTED : launch_q<float, kIdentity>(ng, qmode, p, l, s);
  if (bf16)
    return nk == kLn ? launch_q<uint16_t, kLn>(ng, qmode, p, l, s)
                     : launch_q<uint16_t, kRms>(ng, qmode, p, l, s);
  return nk == kLn ? launch_q<float, kLn>(ng, qmode, p, l, s)
                   : launch_q<float, kRms>(ng, qmode, p, l, s);
}

rn_status read_clear_error_fwd(unsigned* code) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_fwd, sizeof(v)) != cudaSuccess) return RN_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_err_fwd, &zero, sizeof(zero)) != cudaSuccess) return RN_ERR_CUDA;
  *code = v;
  return RN_OK;
}

}  // namespace rn
