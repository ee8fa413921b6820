// Scaled activations, forward with a quantize epilogue and backward (page
// "Activation + GroupedLinear Fusion for MOE and other MOE optimizations",
// section "Better Kernels for Scaled Activations": scaled SReLU, SwiGLU and
// clamped SwiGLU as single fused kernels; the backward returns the input
// gradient and the gradient of the scales).
//
//   y[i, j]   = s_i * act(x)[i, j]
//   SReLU     act = max(x, 0)^2                          (H inputs a row)
//   SwiGLU    act = silu(a) * b, silu(a) = a * sigmoid(a) (2H inputs a row:
//             a = the first H, b = the last H)
//   clamped   act = ac * sigmoid(alpha ac) * (bc + 1), ac = min(a, L),
//             bc = clamp(b, -L, L)
//   backward  dx = s_i * dy * act'(x) (both halves for the GLU forms),
//             dscales_i = sum_j dy[i, j] * act(x)[i, j]
//
// Both directions are streaming, elementwise work with one row reduction
// (the backward's dscales) or one tensor reduction (amax): a warp takes a
// row (rows w, w + W, ... for global warp w of W), each lane 16-byte chunks
// c = lane + 32 k of the output columns, issues every load of a slice of
// up to 4 chunks a lane (dy too in the backward; the gate and the linear
// half for the GLU forms) before any arithmetic, so that a warp keeps 4-6 KB
// in flight (24 warps an SM in the forward, 16 in the backward), and stores
// the results with 8-32-byte stores.  Rows longer than a slice are walked in
// slices.  No shared-memory staging: nothing is reused.
// Output modes as for the normalization: bf16 / fp32, FP8 with a given scale
// (+ amax), FP8 with current scaling in two launches (amax pass, then
// quantize with 448/amax, a programmatic dependent), and MXFP8 rowwise (1x32
// blocks over the 4 or 8 lanes that hold them; no columnwise copy).
#include <cuda_runtime.h>

#include "rn_device.cuh"
#include "rn_internal.h"

namespace rn {
namespace {

constexpr int kActThreads = 256;
constexpr int kActNC = 4;     // chunks a lane holds per slice (forward)
constexpr int kActBwdNC = 4;  // the same for the backward (three streams in)

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// the VEC fp32 values of one 16-byte chunk
template <typename TIn>
__device__ __forceinline__ void chunk_f32(const uint4& v, float* f);
template <>
__device__ __forceinline__ void chunk_f32<uint16_t>(const uint4& v, float* f) {
  bf16x8_to_f32(v, f);
}
template <>
__device__ __forceinline__ void chunk_f32<float>(const uint4& v, float* f) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}

// 1 / (1 + exp(-z)): the hardware exponential __expf (relative error at most
// 2 + 1.17 |z| ulp by the CUDA documentation's bound, so within 2^-18 for
// |z| <= 25; the more accurate expf made the SwiGLU forward to MXFP8
// 126.9 us against 106.1 us at 65536 x 2048, and to FP8 current 199.7 against
// 183.4 us), then the fast reciprocal-based division (2 ulp; a correctly
// rounded reciprocal cost a third of the forward's time)
__device__ __forceinline__ float sigmoid_f(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

// act(a[, b]) for one element
template <int ACT>
__device__ __forceinline__ float act_value(float a, float b, float lim, float alpha) {
  if constexpr (ACT == kActSrelu) {
    const float t = fmaxf(a, 0.0f);
    return t * t;
  } else if constexpr (ACT == kActSwiglu) {
    return (a * sigmoid_f(a)) * b;
  } else {
    const float ac = fminf(a, lim), bc = fminf(fmaxf(b, -lim), lim);
    return (ac * sigmoid_f(alpha * ac)) * (bc + 1.0f);
  }
}

// act(a, b) and its derivatives d/da, d/db for one element
template <int ACT>
__device__ __forceinline__ void act_grad(float a, float b, float lim, float alpha, float& v,
                                         float& da, float& db) {
  if constexpr (ACT == kActSrelu) {
    const float t = fmaxf(a, 0.0f);
    v = t * t;
    da = 2.0f * t;
    db = 0.0f;
  } else if constexpr (ACT == kActSwiglu) {
    const float sg = sigmoid_f(a);
    const float si = a * sg;
    v = si * b;
    da = (b * sg) * (1.0f + a * (1.0f - sg));
    db = si;
  } else {
    const float ac = fminf(a, lim), bc = fminf(fmaxf(b, -lim), lim);
    const float sg = sigmoid_f(alpha * ac);
    const float si = ac * sg;
    v = si * (bc + 1.0f);
    da = (a <= lim) ? ((bc + 1.0f) * sg) * (1.0f + (alpha * ac) * (1.0f - sg)) : 0.0f;
    db = (b >= -lim && b <= lim) ? si : 0.0f;
  }
}

// E4M3 codes of s * y for one chunk (VEC values), element 0 in the low byte
template <int VEC>
__device__ __forceinline__ void store_e4m3(uint8_t* o, const float* y, float s) {
  float2 z[VEC / 2];
#pragma unroll
  for (int i = 0; i < VEC / 2; ++i) z[i] = mul2(make_float2(y[2 * i], y[2 * i + 1]), splat2(s));
  if constexpr (VEC == 8)
    *reinterpret_cast<uint2*>(o) = make_uint2(pack_e4m3x4(z[0].x, z[0].y, z[1].x, z[1].y),
                                              pack_e4m3x4(z[2].x, z[2].y, z[3].x, z[3].y));
  else
    *reinterpret_cast<uint32_t*>(o) = pack_e4m3x4(z[0].x, z[0].y, z[1].x, z[1].y);
}

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    asm("max.NaN.f32 %0, %0, %1;" : "+f"(v) : "f"(w));
  }
  return v;
}

template <int ACT, typename TIn, int QM>
__global__ void __launch_bounds__(kActThreads, 3) rn_act_fwd_kernel(const ActParams p) {
  constexpr int VEC = 16 / (int)sizeof(TIn);
  constexpr bool GLU = (ACT != kActSrelu);
  constexpr bool AMAX = (QM == kQDelayed || QM == kQCurAmax);
  __shared__ float red[kActThreads / 32];
  const int lane = threadIdx.x & 31;
  const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int nw = (int)((gridDim.x * blockDim.x) >> 5);
  const int H = p.H;
  const int nco = H / VEC;  // output chunks a row
  const size_t in_w = GLU ? 2 * (size_t)H : (size_t)H;
  const bool mx = p.row_scales != nullptr;  // MXFP8 rowwise (QM == kQNone with codes)

  if (QM == kQCurAmax && threadIdx.x == 0) pdl_launch_dependents();
  float scale = 1.0f;
  if constexpr (QM == kQDelayed) scale = *p.scale;
  if constexpr (QM == kQCurQuant) {
    pdl_wait();  // amax comes from pass 1
    const float am = *p.amax;
    scale = (am == 0.0f) ? 1.0f : __fdiv_rn(448.0f, am);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      *p.scale_out = scale;
      *p.scale_inv = __fdiv_rn(1.0f, scale);
    }
  }
  float amax = 0.0f;

  for (int row = gw; row < p.N; row += nw) {
    const float s = p.scales ? __ldg(p.scales + row) : 1.0f;
    const unsigned char* xrow =
        static_cast<const unsigned char*>(p.x) + (size_t)row * in_w * sizeof(TIn);
    for (int c0 = 0; c0 < nco; c0 += 32 * kActNC) {
      uint4 va[kActNC], vb[kActNC];
#pragma unroll
      for (int k = 0; k < kActNC; ++k) {
        const int c = c0 + lane + 32 * k;
        if (c < nco) {
          va[k] = ldg_stream(xrow + (size_t)c * 16);
          if constexpr (GLU) vb[k] = ldg_stream(xrow + (size_t)H * sizeof(TIn) + (size_t)c * 16);
        }
      }
#pragma unroll
      for (int k = 0; k < kActNC; ++k) {
        const int c = c0 + lane + 32 * k;
        const bool valid = c < nco;
        float y[VEC];
        float bm = 0.0f;  // MXFP8: max |y| of the chunk
        if (valid) {
          float a[VEC], b[VEC];
          chunk_f32<TIn>(va[k], a);
          if constexpr (GLU) chunk_f32<TIn>(vb[k], b);
#pragma unroll
          for (int e = 0; e < VEC; ++e) y[e] = act_value<ACT>(a[e], GLU ? b[e] : 0.0f, p.limit, p.alpha) * s;
          // magnitudes two at a time (3-input max; NaN wins)
#pragma unroll
          for (int e = 0; e < VEC; e += 2) {
            if constexpr (AMAX) amax = amax_acc2(amax, make_float2(y[e], y[e + 1]));
            if (QM == kQNone && mx) bm = amax_acc2(bm, make_float2(y[e], y[e + 1]));
          }
        }
        if (QM == kQNone && mx) {
          // a 1x32 block is 32 / VEC adjacent lanes (all valid or none:
          // H % 32 == 0 and slices end on multiples of 32 chunks)
#pragma unroll
          for (int o = 1; o < 32 / VEC; o <<= 1) {
            const float w = __shfl_xor_sync(0xFFFFFFFFu, bm, o);
            asm("max.NaN.f32 %0, %0, %1;" : "+f"(bm) : "f"(w));
          }
          if (valid) {
            const uint32_t code = e8m0_code(bm);
            const float inv = e8m0_inv_scale(code);
            store_e4m3<VEC>(static_cast<uint8_t*>(p.out) + (size_t)row * H + (size_t)c * VEC, y, inv);
            if ((lane & (32 / VEC - 1)) == 0)
              p.row_scales[(size_t)row * (H / 32) + (size_t)c * VEC / 32] = (uint8_t)code;
          }
          continue;
        }
        if (!valid || QM == kQCurAmax) continue;
        if constexpr (QM == kQNone) {
          if (p.out_f32) {
            float4* o = reinterpret_cast<float4*>(static_cast<unsigned char*>(p.out) +
                                                  ((size_t)row * H + (size_t)c * VEC) * 4);
#pragma unroll
            for (int q = 0; q < VEC / 4; ++q)
              o[q] = make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
          } else {
            unsigned char* o =
                static_cast<unsigned char*>(p.out) + ((size_t)row * H + (size_t)c * VEC) * 2;
            if constexpr (VEC == 8)
              *reinterpret_cast<uint4*>(o) =
                  make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                             pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
            else
              *reinterpret_cast<uint2*>(o) =
                  make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
          }
        } else {  // E4M3 codes with the tensor scale
          store_e4m3<VEC>(static_cast<uint8_t*>(p.out) + (size_t)row * H + (size_t)c * VEC, y, scale);
        }
      }
    }
  }

  if constexpr (AMAX) {
    const float m = warp_max_nan(amax);
    if (lane == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t b = 0;
      for (int w = 0; w < kActThreads / 32; ++w) b = max(b, abs_bits(red[w]));
      pdl_wait();  // amax was zeroed by the kernel this one depends on
      atomicMax(reinterpret_cast<unsigned int*>(p.amax), b);
    }
  }
}

template <int ACT, typename TIn>
__global__ void __launch_bounds__(kActThreads, 2) rn_act_bwd_kernel(const ActParams p) {
  constexpr int VEC = 16 / (int)sizeof(TIn);
  constexpr bool GLU = (ACT != kActSrelu);
  const int lane = threadIdx.x & 31;
  const int gw = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int nw = (int)((gridDim.x * blockDim.x) >> 5);
  const int H = p.H;
  const int nco = H / VEC;
  const size_t in_w = GLU ? 2 * (size_t)H : (size_t)H;

  for (int row = gw; row < p.N; row += nw) {
    const float s = p.scales ? __ldg(p.scales + row) : 1.0f;
    const unsigned char* xrow =
        static_cast<const unsigned char*>(p.x) + (size_t)row * in_w * sizeof(TIn);
    const unsigned char* dyrow =
        static_cast<const unsigned char*>(p.dy) + (size_t)row * H * sizeof(TIn);
    unsigned char* dxrow = static_cast<unsigned char*>(p.out) + (size_t)row * in_w * sizeof(TIn);
    float dsum = 0.0f;
    for (int c0 = 0; c0 < nco; c0 += 32 * kActBwdNC) {
      uint4 va[kActBwdNC], vb[kActBwdNC], vd[kActBwdNC];
#pragma unroll
      for (int k = 0; k < kActBwdNC; ++k) {
        const int c = c0 + lane + 32 * k;
        if (c < nco) {
          vd[k] = ldg_stream(dyrow + (size_t)c * 16);
          va[k] = ldg_stream(xrow + (size_t)c * 16);
          if constexpr (GLU) vb[k] = ldg_stream(xrow + (size_t)H * sizeof(TIn) + (size_t)c * 16);
        }
      }
#pragma unroll
      for (int k = 0; k < kActBwdNC; ++k) {
        const int c = c0 + lane + 32 * k;
        if (c >= nco) continue;
        float a[VEC], b[VEC], d[VEC], ga[VEC], gb[VEC];
        chunk_f32<TIn>(va[k], a);
        chunk_f32<TIn>(vd[k], d);
        if constexpr (GLU) chunk_f32<TIn>(vb[k], b);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          float v, da, db;
          act_grad<ACT>(a[e], GLU ? b[e] : 0.0f, p.limit, p.alpha, v, da, db);
          const float sd = s * d[e];
          ga[e] = sd * da;
          gb[e] = sd * db;
          dsum = fmaf(d[e], v, dsum);
        }
        if constexpr (VEC == 8) {
          *reinterpret_cast<uint4*>(dxrow + (size_t)c * 16) =
              make_uint4(pack_bf16x2(ga[0], ga[1]), pack_bf16x2(ga[2], ga[3]),
                         pack_bf16x2(ga[4], ga[5]), pack_bf16x2(ga[6], ga[7]));
          if constexpr (GLU)
            *reinterpret_cast<uint4*>(dxrow + (size_t)H * 2 + (size_t)c * 16) =
                make_uint4(pack_bf16x2(gb[0], gb[1]), pack_bf16x2(gb[2], gb[3]),
                           pack_bf16x2(gb[4], gb[5]), pack_bf16x2(gb[6], gb[7]));
        } else {
          *reinterpret_cast<float4*>(dxrow + (size_t)c * 16) = make_float4(ga[0], ga[1], ga[2], ga[3]);
          if constexpr (GLU)
            *reinterpret_cast<float4*>(dxrow + (size_t)H * 4 + (size_t)c * 16) =
                make_float4(gb[0], gb[1], gb[2], gb[3]);
        }
      }
    }
    if (p.dscales != nullptr) {
      const float t = warp_sum(dsum);
      if (lane == 0) p.dscales[row] = t;
    }
  }
}

template <typename Kernel>
rn_status launch_persistent(Kernel k, const ActParams& p, int sms, bool pdl, cudaStream_t s) {
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kActThreads, 0) != cudaSuccess)
    return RN_ERR_CUDA;
  if (occ < 1) occ = 1;
  const long long warps_needed = p.N;  // one warp a row
  long long grid = (long long)sms * occ;
  const long long by_rows = (warps_needed + kActThreads / 32 - 1) / (kActThreads / 32);
  if (grid > by_rows) grid = by_rows;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kActThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, k, p) != cudaSuccess) return RN_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

template <int ACT, typename TIn>
rn_status fwd_q(int qmode, const ActParams& p, int sms, bool pdl, cudaStream_t s) {
  switch (qmode) {
    case kQNone: return launch_persistent(rn_act_fwd_kernel<ACT, TIn, kQNone>, p, sms, pdl, s);
    case kQDelayed: return launch_persistent(rn_act_fwd_kernel<ACT, TIn, kQDelayed>, p, sms, pdl, s);
    case kQCurAmax: return launch_persistent(rn_act_fwd_kernel<ACT, TIn, kQCurAmax>, p, sms, pdl, s);
    case kQCurQuant: return launch_persistent(rn_act_fwd_kernel<ACT, TIn, kQCurQuant>, p, sms, pdl, s);
    default: return RN_ERR_INVALID;
  }
}

template <int ACT>
rn_status fwd_t(bool bf16, int qmode, const ActParams& p, int sms, bool pdl, cudaStream_t s) {
  return bf16 ? fwd_q<ACT, uint16_t>(qmode, p, sms, pdl, s) : fwd_q<ACT, float>(qmode, p, sms, pdl, s);
}

template <int ACT>
rn_status bwd_t(bool bf16, const ActParams& p, int sms, cudaStream_t s) {
  return bf16 ? launch_persistent(rn_act_bwd_kernel<ACT, uint16_t>, p, sms, false, s)
              : launch_persistent(rn_act_bwd_kernel<ACT, float>, p, sms, false, s);
}

}  // namespace

rn_status launch_act_fwd(int act, bool bf16, int qmode, const ActParams& p, int sms, bool pdl,
                         cudaStream_t s) {
  switch (act) {
    case kActSrelu: return fwd_t<kActSrelu>(bf16, qmode, p, sms, pdl, s);
    case kActSwiglu: return fwd_t<kActSwiglu>(bf16, qmode, p, sms, pdl, s);
    case kActClampedSwiglu: return fwd_t<kActClampedSwiglu>(bf16, qmode, p, sms, pdl, s);
    default: return RN_ERR_INVALID;
  }
}

rn_status launch_act_bwd(int act, bool bf16, const ActParams& p, int sms, cudaStream_t s) {
  switch (act) {
    case kActSrelu: return bwd_t<kActSrelu>(bf16, p, sms, s);
    case kActSwiglu: return bwd_t<kActSwiglu>(bf16, p, sms, s);
    case kActClampedSwiglu: return bwd_t<kActClampedSwiglu>(bf16, p, sms, s);
    default: return RN_ERR_INVALID;
  }
}

}  // namespace rn
