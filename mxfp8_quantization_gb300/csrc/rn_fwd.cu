// Row-wise LayerNorm / RMSNorm forward with fused output quantization
// (page "Implementation:NVIDIA TransformerEngine PyTorch Ext Normalization",
// section "Description": the fully fused delayed-scaling path and both
// passes of the norm+amax-then-quantize current-scaling path).
//
// Design (persistent CTAs, one or two per SM; warp-specialized, with no
// CTA-wide barrier on the row path):
//   * producer warp: one lane streams whole rows of x into a ring of Q
//     shared-memory slots with the bulk-copy engine (cp.async.bulk,
//     completion on the slot's "full" mbarrier) and refills a slot as soon as
//     the apply warps have released it ("empty"); when a pass needs the saved
//     mu / rsigma of a row, the same lane fetches them into the slot with
//     4-byte cp.async tracked by the same barrier;
//   * stats warps: warp j of S takes rows j, j+S, ... of the CTA's sequence
//     and computes its statistics from shared memory (LayerNorm: two passes,
//     mean then centred sum of squares; RMSNorm: sum of squares), writes
//     mu / rsigma and publishes (mean, rsigma) on the slot's "ready"
//     mbarrier;
//   * apply warps: every thread owns fixed 16-byte column chunks (gamma /
//     beta in registers for the whole kernel); for each row in order it waits
//     for "ready", forms y = (x-mu)*rsigma*g + beta (RMSNorm: x*rsigma*g),
//     stores bf16/fp32 or E4M3 codes, and releases the slot;
//   so statistics of later rows are computed while earlier rows are applied.
//   * arithmetic is done on pairs of elements with the packed fp32 (f32x2)
//     instructions, and bf16 inputs enter through the mixed-precision
//     add/sub/fma forms, which round exactly like convert-then-operate;
//   * the per-tensor amax is reduced per thread, per CTA, then with one
//     atomicMax on the fp32 bit pattern (ordered like the values for
//     non-negative numbers, NaN above +inf).
// Current scaling runs the kernel twice: pass 1 (statistics + amax, no
// output) and pass 2 (quantize with 448/amax, no stats warps), the second
// walking the tiles backwards so that it starts on the rows pass 1 left in
// L2.
#include <cuda_runtime.h>

#include "rn_device.cuh"
#include "rn_internal.h"

namespace rn {
namespace {

__device__ unsigned g_err_fwd;

// compact shape: at most 8 apply + 4 stats warps + the producer, two CTAs
// per SM; wide shape: up to 16 apply + 8 stats warps + the producer, one CTA
constexpr int kMaxThreads = 416;
constexpr int kMaxThreadsWide = 800;

// store the PAIRS y pairs of one chunk in the output format
template <int PAIRS, int QM>
__device__ __forceinline__ void store_chunk(const FwdParams& p, size_t elem, const float2* y,
                                            float scale) {
  if constexpr (QM == kQNone) {
    if (p.out_f32) {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(p.out) + elem);
#pragma unroll
      for (int i = 0; i < PAIRS / 2; ++i)
        o[i] = make_float4(y[2 * i].x, y[2 * i].y, y[2 * i + 1].x, y[2 * i + 1].y);
    } else {
      uint16_t* o = static_cast<uint16_t*>(p.out) + elem;
      if constexpr (PAIRS == 4) {
        *reinterpret_cast<uint4*>(o) =
            make_uint4(pack_bf16x2(y[0].x, y[0].y), pack_bf16x2(y[1].x, y[1].y),
                       pack_bf16x2(y[2].x, y[2].y), pack_bf16x2(y[3].x, y[3].y));
      } else {
        *reinterpret_cast<uint2*>(o) =
            make_uint2(pack_bf16x2(y[0].x, y[0].y), pack_bf16x2(y[1].x, y[1].y));
      }
    }
  } else {
    uint8_t* o = static_cast<uint8_t*>(p.out) + elem;
    uint32_t c[PAIRS];
#pragma unroll
    for (int i = 0; i < PAIRS; ++i) {
      const float2 s = mul2(y[i], splat2(scale));
      c[i] = pack_e4m3x2(s.x, s.y);
    }
    if constexpr (PAIRS == 4)
      *reinterpret_cast<uint2*>(o) = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
    else
      *reinterpret_cast<uint32_t*>(o) = c[0] | (c[1] << 16);
  }
}

// Enumerates the rows of this CTA in the order every role visits them:
// tiles blockIdx.x, blockIdx.x + gridDim.x, ... (walked from the last tile
// when reverse), T rows each.
struct RowWalk {
  int tk, r, r1;
  __device__ __forceinline__ bool next(const FwdParams& p) {
    if (++r < r1) return true;
    tk = (tk < 0) ? (int)blockIdx.x : tk + (int)gridDim.x;
    if (tk >= p.n_tiles) return false;
    const int tt = p.reverse ? p.n_tiles - 1 - tk : tk;
    r = tt * p.T;
    r1 = min(r + p.T, p.N);
    return true;
  }
};

template <typename TIn, int NG, int NK, int QM, bool WIDE>
__global__ void __launch_bounds__(WIDE ? kMaxThreadsWide : kMaxThreads, WIDE ? 1 : 2)
    rn_fwd_kernel(const FwdParams p) {
  constexpr int VEC = 16 / (int)sizeof(TIn);
  using V = Vec<TIn, VEC>;
  constexpr int PAIRS = V::PAIRS;
  constexpr bool LN = (NK == kLn);
  // pass 2 of current scaling gets mu / rsigma with each row
  constexpr bool META = (QM == kQCurQuant && NK != kIdentity);
  // rows whose statistics stats warps compute
  constexpr bool STATS = (QM != kQCurQuant && NK != kIdentity);
  extern __shared__ __align__(128) unsigned char smem[];

  const int A = p.apply_warps;           // warps 0 .. A-1
  const int S = STATS ? p.stats_warps : 0;  // warps A .. A+S-1; producer: A+S
  const int TH = A * 32;                 // apply threads
  const int H = p.H;
  const int nchunks = H / VEC;
  const uint32_t row_bytes = (uint32_t)H * sizeof(TIn);
  const uint32_t Q = (uint32_t)p.Q;

  unsigned char* ring = smem;
  float2* rstat = reinterpret_cast<float2*>(smem + (size_t)Q * row_bytes);  // [Q] (mean, rsigma)
  uint32_t* red = reinterpret_cast<uint32_t*>(rstat + Q);                   // [32]
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 32);                   // row landed
  uint64_t* ready = full + Q;                                               // statistics written
  uint64_t* empty = ready + Q;                                              // slot released

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < Q; ++i) {
      mbar_init(smem_u32(&full[i]), META ? 2 : 1);
      mbar_init(smem_u32(&ready[i]), 1);
      mbar_init(smem_u32(&empty[i]), A);
    }
    fence_barrier_init();
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (warp == A + S) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const unsigned char* xb = static_cast<const unsigned char*>(p.x);
      RingPos pos{0u, 0u};
      uint32_t issued = 0;
      RowWalk wk{-1, 0, 0};
      while (wk.next(p)) {
        const int r = wk.r;
        const uint32_t s = pos.slot;
        if (issued >= Q) mbar_wait(smem_u32(&empty[s]), pos.phase ^ 1u, &g_err_fwd, kErrEmptyWait);
        const uint32_t bar = smem_u32(&full[s]);
        if constexpr (META) {
          if (LN) cp_async4(smem_u32(&rstat[s].x), p.mu + r);
          cp_async4(smem_u32(&rstat[s].y), p.rsigma + r);
          cp_async_arrive(bar);
        }
        mbar_arrive_expect_tx(bar, row_bytes);
        bulk_g2s(smem_u32(ring + (size_t)s * row_bytes), xb + (size_t)r * row_bytes, row_bytes, bar);
        pos.advance(1, Q);
        ++issued;
      }
      // every copy this CTA issued must have landed before it exits
      const uint32_t first = issued > Q ? issued - Q : 0;
      for (uint32_t k = first; k < issued; ++k)
        mbar_wait(smem_u32(&full[k % Q]), (k / Q) & 1u, &g_err_fwd, kErrDrainWait);
    }
    return;
  }

  if (warp >= A) {
    // --------------------------------------------------------- stats warps
    // stats warp j takes rows j, j + S, j + 2S, ... of the CTA's sequence;
    // LayerNorm: two passes over the row in shared memory (mean, then the
    // centred sum of squares); RMSNorm: one pass (sum of squares)
    if constexpr (STATS) {
      const int j = warp - A;
      const float inv_h = 1.0f / (float)H;
      RingPos pos{0u, 0u};
      RowWalk wk{-1, 0, 0};
      int q = 0;
      while (wk.next(p)) {
        if (q++ % S == j) {
          const uint32_t s = pos.slot;
          // a stats warp is not paced by the apply warps: before waiting for
          // this use of the slot it waits for the previous use to be
          // released, so that the parity wait below cannot match a phase
          // one lap old (alias-free because stats warps are fewer than slots)
          if (q > (int)Q) mbar_wait(smem_u32(&empty[s]), pos.phase ^ 1u, &g_err_fwd, kErrStatsWait);
          mbar_wait(smem_u32(&full[s]), pos.phase, &g_err_fwd, kErrStatsWait);
          const unsigned char* rowp = ring + (size_t)s * row_bytes;
          float2 a[PAIRS];
          float mean = 0.0f;
          if constexpr (LN) {
#pragma unroll
            for (int i = 0; i < PAIRS; ++i) a[i] = make_float2(0.f, 0.f);
            for (int c = lane; c < nchunks; c += 32) {
              const typename V::Raw raw = V::load(rowp, c);
#pragma unroll
              for (int i = 0; i < PAIRS; ++i) V::acc(a[i], raw, i);
            }
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < PAIRS; ++i) sum += a[i].x + a[i].y;
            mean = warp_sum(sum) * inv_h;
          }
#pragma unroll
          for (int i = 0; i < PAIRS; ++i) a[i] = make_float2(0.f, 0.f);
          for (int c = lane; c < nchunks; c += 32) {
            const typename V::Raw raw = V::load(rowp, c);
#pragma unroll
            for (int i = 0; i < PAIRS; ++i) {
              if constexpr (LN) {
                const float2 d = V::sub(raw, i, mean);
                a[i] = fma2(d, d, a[i]);
              } else {
                V::sq_acc(a[i], raw, i);
              }
            }
          }
          float m2 = 0.f;
#pragma unroll
          for (int i = 0; i < PAIRS; ++i) m2 += a[i].x + a[i].y;
          const float rs = __frsqrt_rn(warp_sum(m2) * inv_h + p.eps);
          if (lane == 0) {
            rstat[s] = make_float2(mean, rs);
            if constexpr (LN) p.mu[wk.r] = mean;
            p.rsigma[wk.r] = rs;
            mbar_arrive(smem_u32(&ready[s]));
          }
        }
        pos.advance(1, Q);
      }
    }
    return;
  }

  // ---------------------------------------------------------- apply warps
  const int t = threadIdx.x;
  float2 g2[NG][PAIRS], b2[NG][PAIRS];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int v = g * TH + t;
#pragma unroll
    for (int i = 0; i < PAIRS; ++i) {
      g2[g][i] = make_float2(0.f, 0.f);
      b2[g][i] = make_float2(0.f, 0.f);
      if (NK != kIdentity && v < nchunks) {
        const int c = v * VEC + 2 * i;
        const float ga = p.gamma[c], gb = p.gamma[c + 1];
        g2[g][i] = p.zcg ? make_float2(1.0f + ga, 1.0f + gb) : make_float2(ga, gb);
        if (LN && p.beta != nullptr) b2[g][i] = make_float2(p.beta[c], p.beta[c + 1]);
      }
    }
  }

  float scale = 1.0f;
  if constexpr (QM == kQDelayed) {
    scale = *p.scale;
    if (blockIdx.x == 0 && t == 0) *p.scale_inv = __fdiv_rn(1.0f, scale);
  }
  if constexpr (QM == kQCurQuant) {
    const float am = *p.amax;
    scale = (am == 0.0f) ? 1.0f : __fdiv_rn(448.0f, am);
    if (blockIdx.x == 0 && t == 0) {
      *p.scale_out = scale;
      *p.scale_inv = __fdiv_rn(1.0f, scale);
    }
  }
  float ymax = 0.0f, ymin = 0.0f;  // amax = max(ymax, -ymin)

  RingPos pos{0u, 0u};
  RowWalk wk{-1, 0, 0};
  while (wk.next(p)) {
    const uint32_t s = pos.slot;
    // "ready" is published by a stats warp after it saw the row land, so it
    // implies "full"
    if constexpr (STATS)
      mbar_wait(smem_u32(&ready[s]), pos.phase, &g_err_fwd, kErrReadyWait);
    else
      mbar_wait(smem_u32(&full[s]), pos.phase, &g_err_fwd, kErrFullWait);
    float mean = 0.0f, rs = 1.0f;
    if constexpr (STATS || META) {
      const float2 m = rstat[s];
      mean = LN ? m.x : 0.0f;
      rs = m.y;
    }
    const unsigned char* rowp = ring + (size_t)s * row_bytes;
    const size_t rowe = (size_t)wk.r * H;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const int v = g * TH + t;
      if (v < nchunks) {
        const typename V::Raw raw = V::load(rowp, v);
        float2 y[PAIRS];
#pragma unroll
        for (int i = 0; i < PAIRS; ++i) {
          if constexpr (LN) {
            y[i] = fma2(mul2(V::sub(raw, i, mean), splat2(rs)), g2[g][i], b2[g][i]);
          } else if constexpr (NK == kRms) {
            y[i] = mul2(mul2(V::f32(raw, i), splat2(rs)), g2[g][i]);
          } else {
            y[i] = V::f32(raw, i);
          }
          if constexpr (QM == kQDelayed || QM == kQCurAmax) {
            ymax = max3(ymax, y[i]);
            ymin = min3(ymin, y[i]);
          }
        }
        if constexpr (QM != kQCurAmax) store_chunk<PAIRS, QM>(p, rowe + (size_t)v * VEC, y, scale);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    pos.advance(1, Q);
  }

  if constexpr (QM == kQDelayed || QM == kQCurAmax) {
    float amax_t;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(amax_t) : "f"(ymax), "f"(-ymin));
    const uint32_t b = warp_umax(abs_bits(amax_t));
    if (lane == 0) red[warp] = b;
    consumer_sync(TH);
    if (t == 0) {
      uint32_t m = 0;
      for (int w = 0; w < A; ++w) m = max(m, red[w]);
      atomicMax(reinterpret_cast<unsigned int*>(p.amax), m);
    }
  }
}

template <typename TIn, int NG, int NK, int QM, bool WIDE>
rn_status launch_t(const FwdParams& p, const Launch& l, cudaStream_t s) {
  auto k = rn_fwd_kernel<TIn, NG, NK, QM, WIDE>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l.smem) !=
      cudaSuccess)
    return RN_ERR_CUDA;
  int grid = 1;
  if (persistent_grid(k, l, &grid) != RN_OK) return RN_ERR_CUDA;
  k<<<grid, l.threads, l.smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

// compact shape for NG 1 and 2; wide shape for NG 2, 4 and 8
template <typename TIn, int NK, int QM>
rn_status launch_ng(int ng, const FwdParams& p, const Launch& l, cudaStream_t s) {
  const bool wide = l.threads > kMaxThreads || l.per_sm == 1;
  if (!wide) {
    switch (ng) {
      case 1: return launch_t<TIn, 1, NK, QM, false>(p, l, s);
      case 2: return launch_t<TIn, 2, NK, QM, false>(p, l, s);
      default: return RN_ERR_UNSUPPORTED;
    }
  }
  if (l.threads > kMaxThreadsWide) return RN_ERR_UNSUPPORTED;
  switch (ng) {
    case 2: return launch_t<TIn, 2, NK, QM, true>(p, l, s);
    case 4: return launch_t<TIn, 4, NK, QM, true>(p, l, s);
    case 8: return launch_t<TIn, 8, NK, QM, true>(p, l, s);
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
