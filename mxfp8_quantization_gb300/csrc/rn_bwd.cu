// LayerNorm / RMSNorm backward: dx, and dgamma / dbeta reduced over all rows
// (page "Implementation:NVIDIA TransformerEngine PyTorch Ext Normalization",
// sections "Description" and "Signature": layernorm_bwd / rmsnorm_bwd).
//
// With xhat = (x - mu) * rsigma (RMSNorm: x * rsigma), g = gamma (or
// 1 + gamma when zero-centered) and dy = dz * g:
//   LayerNorm  dx = rsigma * (dy - mean(dy) - xhat * mean(dy * xhat))
//   RMSNorm    dx = rsigma * (dy - xhat * mean(dy * xhat))
//   dgamma = sum_rows dz * xhat,  dbeta = sum_rows dz.
//
// Kernel 1 (persistent, warp-specialized like the forward): the producer
// lane streams the x row and the dz row of each row into one shared-memory
// slot with two bulk copies; the consumers take tiles of T rows:
//   phase 1  the two row means mean(dy), mean(dy * xhat): WPR warps share a
//            row (one when rows are short), each summing an interleaved slice
//            of its chunks; the slices are added in slice order (g is read
//            from a shared-memory copy);
//   phase 2  each thread owns fixed 16-byte column chunks: dx for every row
//            of the tile, plus running per-column sums of dz * xhat and dz
//            in registers.
// Rows are grouped in fixed chunks of tiles_per_chunk * T rows; at the end
// of a chunk its column sums are written to the workspace as one fp32
// partial row.  The chunk size depends on N and H only, and each partial is
// summed in row order, so the partials do not depend on the grid.
// Kernel 2 adds the partials of each column in chunk order (a fixed tree:
// 32 strided sequential sums, then the 32 results in order).
#include <cuda_runtime.h>

#include "rn_device.cuh"
#include "rn_internal.h"

namespace rn {
namespace {

__device__ unsigned g_err_bwd;

constexpr int kMaxThreads = 512 + 32;

template <typename TIn>
struct BChunk;

template <>
struct BChunk<uint16_t> {
  static constexpr int VEC = 8;
  __device__ __forceinline__ static void load(const unsigned char* p, int c, float* f) {
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(p + (size_t)c * 16), f);
  }
  __device__ __forceinline__ static void store(void* base, size_t elem, const float* y) {
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + elem) =
        make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                   pack_bf16x2(y[6], y[7]));
  }
};

template <>
struct BChunk<float> {
  static constexpr int VEC = 4;
  __device__ __forceinline__ static void load(const unsigned char* p, int c, float* f) {
    const float4 v = *reinterpret_cast<const float4*>(p + (size_t)c * 16);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  __device__ __forceinline__ static void store(void* base, size_t elem, const float* y) {
    *reinterpret_cast<float4*>(static_cast<float*>(base) + elem) = make_float4(y[0], y[1], y[2], y[3]);
  }
};

template <typename TIn, int NG, bool LN>
__global__ void __launch_bounds__(kMaxThreads, 1) rn_bwd_kernel(const BwdParams p) {
  using C = BChunk<TIn>;
  constexpr int VEC = C::VEC;
  extern __shared__ __align__(128) unsigned char smem[];

  const int TH = blockDim.x - 32;
  const int W = TH >> 5;
  const int H = p.H;
  const int nchunks = H / VEC;
  const uint32_t row_bytes = (uint32_t)H * sizeof(TIn);
  const uint32_t slot_bytes = 2 * row_bytes;  // x row, then dz row
  const int Q = p.Q;
  const int WPR = p.wpr;

  unsigned char* ring = smem;
  float* gs = reinterpret_cast<float*>(smem + (size_t)Q * slot_bytes);  // g, [H]
  float4* stats = reinterpret_cast<float4*>(gs + H);                     // [2][T]
  float2* part = reinterpret_cast<float2*>(stats + 2 * p.T);             // [T * WPR]
  uint64_t* full = reinterpret_cast<uint64_t*>(part + p.T * p.wpr);
  uint64_t* empty = full + Q;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Q; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), W);
    }
    fence_barrier_init();
  }
  for (int j = threadIdx.x; j < H; j += blockDim.x) {
    const float gam = p.gamma[j];
    gs[j] = p.zcg ? 1.0f + gam : gam;
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int tpc = p.tiles_per_chunk;

  if (warp == W) {
    if (lane == 0) {
      const unsigned char* xb = static_cast<const unsigned char*>(p.x);
      const unsigned char* db = static_cast<const unsigned char*>(p.dz);
      uint32_t q = 0;
      for (int c = blockIdx.x; c < p.n_chunks; c += G) {
        const int t1 = min((c + 1) * tpc, p.n_tiles);
        for (int tt = c * tpc; tt < t1; ++tt) {
          const int r0 = tt * p.T;
          const int r1 = min(r0 + p.T, p.N);
          for (int r = r0; r < r1; ++r, ++q) {
            const uint32_t s = q % Q, use = q / Q;
            if (use > 0) mbar_wait(smem_u32(&empty[s]), (use - 1) & 1, &g_err_bwd, kErrEmptyWait);
            const uint32_t bar = smem_u32(&full[s]);
            mbar_arrive_expect_tx(bar, slot_bytes);
            const uint32_t dst = smem_u32(ring + (size_t)s * slot_bytes);
            bulk_g2s(dst, xb + (size_t)r * row_bytes, row_bytes, bar);
            bulk_g2s(dst + row_bytes, db + (size_t)r * row_bytes, row_bytes, bar);
          }
        }
      }
      for (uint32_t k = q > (uint32_t)Q ? q - Q : 0; k < q; ++k)
        mbar_wait(smem_u32(&full[k % Q]), (k / Q) & 1, &g_err_bwd, kErrDrainWait);
    }
    return;
  }

  const int t = threadIdx.x;
  float gv[NG][VEC];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int v = g * TH + t;
#pragma unroll
    for (int i = 0; i < VEC; ++i) gv[g][i] = (v < nchunks) ? gs[v * VEC + i] : 0.f;
  }
  const float hf = (float)H;
  const int nacc = LN ? 2 : 1;

  uint32_t q = 0;
  int it = 0;
  for (int c = blockIdx.x; c < p.n_chunks; c += G) {
    float adg[NG][VEC], adb[NG][VEC];
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        adg[g][i] = 0.f;
        adb[g][i] = 0.f;
      }
    const int t1 = min((c + 1) * tpc, p.n_tiles);
    for (int tt = c * tpc; tt < t1; ++tt, ++it) {
      const int r0 = tt * p.T;
      const int nrows = min(p.T, p.N - r0);
      float4* st = stats + (it & 1) * p.T;

      // ------------------------------------------- phase 1: row reductions
      // WPR warps share a row: warp (k, j) sums chunks j*32 + lane + i*32*WPR
      for (int item = warp; item < nrows * WPR; item += W) {
        const int k = item / WPR, j = item - k * WPR;
        const uint32_t qq = q + k;
        const uint32_t s = qq % Q;
        mbar_wait(smem_u32(&full[s]), (qq / Q) & 1, &g_err_bwd, kErrFullWait);
        const unsigned char* xr = ring + (size_t)s * slot_bytes;
        const unsigned char* dr = xr + row_bytes;
        const float mu = LN ? p.mu[r0 + k] : 0.f;
        const float rs = p.rsigma[r0 + k];
        float s1[VEC], s2[VEC];
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          s1[i] = 0.f;
          s2[i] = 0.f;
        }
        for (int cc = j * 32 + lane; cc < nchunks; cc += 32 * WPR) {
          float xf[VEC], df[VEC];
          C::load(xr, cc, xf);
          C::load(dr, cc, df);
          const float4* gp = reinterpret_cast<const float4*>(gs + cc * VEC);
#pragma unroll
          for (int jj = 0; jj < VEC / 4; ++jj) {
            const float4 g4 = gp[jj];
            const float gg[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int e = 4 * jj + i;
              const float xh = (LN ? xf[e] - mu : xf[e]) * rs;
              const float dy = df[e] * gg[i];
              s1[e] += dy;
              s2[e] = fmaf(dy, xh, s2[e]);
            }
          }
        }
        float a1 = 0.f, a2 = 0.f;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          a1 += s1[i];
          a2 += s2[i];
        }
        a1 = warp_sum(a1);
        a2 = warp_sum(a2);
        if (lane == 0) part[k * WPR + j] = make_float2(a1, a2);
      }
      consumer_sync(TH);
      if (t < nrows) {
        const int k = t;
        float a1 = 0.f, a2 = 0.f;
        for (int j = 0; j < WPR; ++j) {
          const float2 pj = part[k * WPR + j];
          a1 += pj.x;
          a2 += pj.y;
        }
        st[k] = make_float4(LN ? p.mu[r0 + k] : 0.f, p.rsigma[r0 + k],
                            LN ? __fdiv_rn(a1, hf) : 0.f, __fdiv_rn(a2, hf));
      }
      consumer_sync(TH);

      // ------------------------------------------------- phase 2: dx, sums
      for (int k = 0; k < nrows; ++k) {
        const uint32_t qq = q + k;
        const uint32_t s = qq % Q;
        mbar_wait(smem_u32(&full[s]), (qq / Q) & 1, &g_err_bwd, kErrFullWait);
        const float4 m = st[k];
        const unsigned char* xr = ring + (size_t)s * slot_bytes;
        const unsigned char* dr = xr + row_bytes;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const int v = g * TH + t;
          if (v < nchunks) {
            float xf[VEC], df[VEC], dx[VEC];
            C::load(xr, v, xf);
            C::load(dr, v, df);
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
              const float xh = (LN ? xf[i] - m.x : xf[i]) * m.y;
              const float dy = df[i] * gv[g][i];
              dx[i] = (dy - fmaf(xh, m.w, m.z)) * m.y;
              adg[g][i] = fmaf(df[i], xh, adg[g][i]);
              if (LN) adb[g][i] += df[i];
            }
            C::store(p.dx, (size_t)(r0 + k) * H + (size_t)v * VEC, dx);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
      }
      q += nrows;
    }
    // chunk finished: write its partial column sums
    float* prow = p.part + (size_t)c * nacc * H;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const int v = g * TH + t;
      if (v < nchunks) {
#pragma unroll
        for (int j = 0; j < VEC / 4; ++j) {
          reinterpret_cast<float4*>(prow + (size_t)v * VEC)[j] =
              make_float4(adg[g][4 * j], adg[g][4 * j + 1], adg[g][4 * j + 2], adg[g][4 * j + 3]);
          if (LN)
            reinterpret_cast<float4*>(prow + H + (size_t)v * VEC)[j] =
                make_float4(adb[g][4 * j], adb[g][4 * j + 1], adb[g][4 * j + 2], adb[g][4 * j + 3]);
        }
      }
    }
  }
}

// dgamma[j] (a = 0) / dbeta[j] (a = 1) = sum over chunks of part[c][a][j].
// Block: 32 warps x 32 lanes; lane owns 4 adjacent columns of a 128-column
// slice; warp w sums chunks w, w+32, ... in order; then thread j of the
// first 128 adds the 32 warp sums in warp order.  Fixed order throughout.
__global__ void __launch_bounds__(1024) rn_colreduce_kernel(const ColReduceParams p) {
  __shared__ float4 red[32][33];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a = blockIdx.y;
  const int col = blockIdx.x * 128 + lane * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (col < p.H) {
    const float* base = p.part + (size_t)a * p.H + col;
    const size_t stride = (size_t)p.nacc * p.H;
    for (int c = warp; c < p.n_chunks; c += 32) {
      const float4 v = *reinterpret_cast<const float4*>(base + (size_t)c * stride);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
  }
  red[warp][lane] = acc;
  __syncthreads();
  if (threadIdx.x < 128) {
    const int l = threadIdx.x >> 2, e = threadIdx.x & 3;
    const int j = blockIdx.x * 128 + threadIdx.x;
    float s = 0.f;
    for (int w = 0; w < 32; ++w) {
      const float4 v = red[w][l];
      s += (e == 0) ? v.x : (e == 1) ? v.y : (e == 2) ? v.z : v.w;
    }
    if (j < p.H) (a == 0 ? p.dgamma : p.dbeta)[j] = s;
  }
}

template <typename TIn, int NG, bool LN>
rn_status launch_t(const BwdParams& p, const Launch& l, cudaStream_t s) {
  auto k = rn_bwd_kernel<TIn, NG, LN>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l.smem) !=
      cudaSuccess)
    return RN_ERR_CUDA;
  k<<<l.grid, l.threads, l.smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

template <typename TIn, bool LN>
rn_status launch_ng(int ng, const BwdParams& p, const Launch& l, cudaStream_t s) {
  switch (ng) {
    case 1: return launch_t<TIn, 1, LN>(p, l, s);
    case 2: return launch_t<TIn, 2, LN>(p, l, s);
    case 4: return launch_t<TIn, 4, LN>(p, l, s);
    default: return RN_ERR_UNSUPPORTED;
  }
}

}  // namespace

rn_status launch_bwd(bool ln, bool bf16, int ng, const BwdParams& p, const Launch& l,
                     cudaStream_t s) {
  if (bf16) return ln ? launch_ng<uint16_t, true>(ng, p, l, s) : launch_ng<uint16_t, false>(ng, p, l, s);
  return ln ? launch_ng<float, true>(ng, p, l, s) : launch_ng<float, false>(ng, p, l, s);
}

rn_status launch_colreduce(const ColReduceParams& p, cudaStream_t s) {
  dim3 grid((p.H + 127) / 128, p.nacc);
  rn_colreduce_kernel<<<grid, 1024, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

rn_status read_clear_error_bwd(unsigned* code) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_bwd, sizeof(v)) != cudaSuccess) return RN_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_err_bwd, &zero, sizeof(zero)) != cudaSuccess) return RN_ERR_CUDA;
  *code = v;
  return RN_OK;
}

}  // namespace rn
