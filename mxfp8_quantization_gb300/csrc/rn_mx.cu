// LayerNorm / RMSNorm forward fused with MXFP8 output quantization: 1x32
// rowwise and 32x1 columnwise blocks, each with an E8M0 shared scale (page
// "Implementation:NVIDIA TransformerEngine PyTorch Ext Normalization",
// section "Description": the fully fused MXFP8 path).
//
// Two kernels: rn_mx_slab_kernel (further below) for bf16 rows of whole
// 64-column slabs, and the ring kernel described here for the other rows
// (fp32, other widths, the stand-alone quantizer).
//
// Ring-kernel design (one persistent CTA per SM, warp-specialized, no
// CTA-wide barrier on the row path):
//   producer     one lane streams rows of x into a shared-memory ring with
//                cp.async.bulk ("full" mbarrier per slot);
//   stats warps  take rows in turn: mean / rsigma from shared memory
//                (LayerNorm: two passes), written to mu / rsigma and to the
//                slot, and counted on the tile's "ready" mbarrier (32
//                arrivals: one per row of the 32-row tile);
//   apply warps  work on tiles of 32 rows (the height of a column block),
//                each warp on 64-column sub-tiles: every thread holds y for
//                an 8-row x 8-column block in registers, computed once
//                (gamma / beta from a shared-memory copy staged at start).
//                One sweep over |y| gives the thread's 8 row maxima and 8
//                column maxima; from those
//       rowwise  the 1x32 block maxima (the 4 lanes of a block reduce-scatter
//                them, so that each lane encodes 2 of the 8 blocks it touches
//                and the inverse scales are gathered back), the E8M0 codes
//                and the rowwise E4M3 codes;
//       colwise  the same for the 32x1 blocks (4 row groups), and the
//                columnwise codes, 8 per column per thread, stored as 8
//                contiguous bytes of the transposed [H, N] array;
//                output addresses advance from per-tile cursors;
//   then the tile's 32 slots are released ("empty").
// Both directions quantize the same y32 (one computation per element).
// Arithmetic is on element pairs (f32x2); bf16 inputs enter through the
// mixed-precision forms.  When H is a multiple of 64 every sub-tile is whole
// and no lane needs a bounds test.
#include <cuda.h>  // CUtensorMap (the encoder is fetched through the runtime)
#include <cuda_runtime.h>

#include "rn_device.cuh"
#include "rn_internal.h"

namespace rn {
namespace {

__device__ unsigned g_err_mx;

// apply + stats warps + the producer: at most 16 warps (128 registers each)
constexpr int kMaxThreads = 16 * 32;
constexpr int kTile = 32;

// one chunk of 8 columns from shared memory (32-bit shared address)
template <typename TIn>
__device__ __forceinline__ typename Vec<TIn, 8>::Raw load8(uint32_t addr);

template <>
__device__ __forceinline__ Vec<uint16_t, 8>::Raw load8<uint16_t>(uint32_t addr) {
  Vec<uint16_t, 8>::Raw r;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3])
               : "r"(addr));
  return r;
}

template <>
__device__ __forceinline__ Vec<float, 8>::Raw load8<float>(uint32_t addr) {
  Vec<float, 8>::Raw r;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.p[0].x), "=f"(r.p[0].y), "=f"(r.p[1].x), "=f"(r.p[1].y)
               : "r"(addr));
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.p[2].x), "=f"(r.p[2].y), "=f"(r.p[3].x), "=f"(r.p[3].y)
               : "r"(addr + 16));
  return r;
}

// maxima with NaN winning
__device__ __forceinline__ float max3n(float a, float b, float c) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ float max2n(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// The 8 maxima a lane holds for items 0..7 (rows or columns of its 8 x 8
// block) are reduced over the 4 lanes of a block group, which differ in the
// lane bits s1 (high) and s0 (low).  The lane with group index gi = 2 b1 + b0
// ends with the group maxima of items gi and gi + 4 (a two-step
// reduce-scatter: 6 shuffles instead of 16 for a full all-reduce).
__device__ __forceinline__ void block_max_scatter(const float (&v)[8], int b1, int b0, int s1,
                                                  int s0, float& o0, float& o1) {
  float r[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int k = (m & 1) + 4 * (m >> 1);  // 0, 1, 4, 5
    const float keep = b1 ? v[k + 2] : v[k];
    const float send = b1 ? v[k] : v[k + 2];
    r[m] = max2n(keep, __shfl_xor_sync(0xFFFFFFFFu, send, s1));
  }
  const float k0 = b0 ? r[1] : r[0], x0 = b0 ? r[0] : r[1];
  const float k1 = b0 ? r[3] : r[2], x1 = b0 ? r[2] : r[3];
  o0 = max2n(k0, __shfl_xor_sync(0xFFFFFFFFu, x0, s0));
  o1 = max2n(k1, __shfl_xor_sync(0xFFFFFFFFu, x1, s0));
}

// The inverse of block_max_scatter's layout: from each lane's values for
// items gi and gi + 4, every lane of the group gets all 8 (two steps, 6
// shuffles).
__device__ __forceinline__ void gather8(float i0, float i1, int b1, int b0, int s1, int s0,
                                        float (&out)[8]) {
  const float p0 = __shfl_xor_sync(0xFFFFFFFFu, i0, s0);
  const float p1 = __shfl_xor_sync(0xFFFFFFFFu, i1, s0);
  float a[4];  // items 2 b1 + {0, 1, 4, 5}
  a[0] = b0 ? p0 : i0;
  a[1] = b0 ? i0 : p0;
  a[2] = b0 ? p1 : i1;
  a[3] = b0 ? i1 : p1;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int k = (m & 1) + 4 * (m >> 1);
    const float q = __shfl_xor_sync(0xFFFFFFFFu, a[m], s1);
    out[k] = b1 ? q : a[m];
    out[k + 2] = b1 ? a[m] : q;
  }
}

// FULL: H % 64 == 0 (whole sub-tiles); SNC: 8-column chunks of a row a stats
// lane holds (nchunks <= 32 SNC), SFULL: exactly SNC
template <typename TIn, int NK, bool FULL, int SNC, bool SFULL>
__global__ void __launch_bounds__(kMaxThreads, 1) rn_mx_kernel(const MxParams p) {
  using V = Vec<TIn, 8>;
  constexpr bool STATS = (NK != kIdentity);
  constexpr bool LN = (NK == kLn);
  extern __shared__ __align__(128) unsigned char smem[];
  const int A = p.apply_warps;
  const int S = STATS ? p.stats_warps : 0;
  const int H = p.H;
  const int N = p.N;
  const int nchunks = H >> 3;  // chunks of 8 columns
  const uint32_t row_bytes = (uint32_t)H * sizeof(TIn);
  constexpr uint32_t kChunkBytes = 8 * sizeof(TIn);
  const uint32_t Q = (uint32_t)p.Q;
  const int NT = p.n_tbar;
  const size_t gb_bytes = STATS ? (size_t)H * sizeof(float) * (LN ? 2 : 1) : 0;

  float4* gsm = reinterpret_cast<float4*>(smem);  // [2][nchunks]: chunk c's g, part j
  float4* bsm = gsm + 2 * (size_t)nchunks;        // same for beta (LayerNorm)
  unsigned char* ring = smem + gb_bytes;
  float2* rstat = reinterpret_cast<float2*>(ring + (size_t)Q * row_bytes);  // [Q]
  uint64_t* full = reinterpret_cast<uint64_t*>(rstat + Q);
  uint64_t* empty = full + Q;
  uint64_t* tready = empty + Q;  // [NT]: statistics of a tile's 32 rows written

  for (uint32_t i = threadIdx.x; i < Q; i += blockDim.x) {
    mbar_init(smem_u32(&full[i]), 1);
    mbar_init(smem_u32(&empty[i]), A);
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i < NT; i += blockDim.x) {
    mbar_init(smem_u32(&tready[i]), kTile);
    fence_barrier_init();
  }
  if constexpr (STATS) {
    const int n4 = H / 4;
    for (int u = threadIdx.x; u < n4; u += blockDim.x) {
      const int c = u >> 1, j = u & 1;
      const float4 gv = reinterpret_cast<const float4*>(p.gamma)[u];
      gsm[j * nchunks + c] =
          p.zcg ? make_float4(1.0f + gv.x, 1.0f + gv.y, 1.0f + gv.z, 1.0f + gv.w) : gv;
      if (LN)
        bsm[j * nchunks + c] = p.beta ? reinterpret_cast<const float4*>(p.beta)[u]
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
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
      // stats warp j takes rows j, j + S, j + 2S, ... of the CTA's sequence
      // (row q: tile blockIdx.x + (q / 32) * grid, row q % 32 of it)
      const int my_tiles = p.n_tiles > (int)blockIdx.x ? (p.n_tiles - 1 - (int)blockIdx.x) / G + 1 : 0;
      const int nq = my_tiles * kTile;
      RingPos pos{0u, 0u};
      pos.advance((uint32_t)j, Q);
      for (int q = j; q < nq; q += S, pos.advance((uint32_t)S, Q)) {
        const int t = (int)blockIdx.x + (q / kTile) * G;
        const int k = q % kTile;
        const uint32_t s = pos.slot;
        // not paced by the apply warps: wait for the previous use of the
        // slot to be released first, so that the parity wait below
        // cannot match a phase one lap old (stats warps < slots)
        if (q >= (int)Q) mbar_wait(smem_u32(&empty[s]), pos.phase ^ 1u, &g_err_mx, kErrStatsWait);
        mbar_wait(smem_u32(&full[s]), pos.phase, &g_err_mx, kErrStatsWait);
        // the row part of this lane (chunks lane, lane + 32, ...) in registers
        const unsigned char* rowp = ring + (size_t)s * row_bytes;
        typename V::Raw raw[SNC];
#pragma unroll
        for (int k = 0; k < SNC; ++k)
          if (SFULL || lane + 32 * k < nchunks) raw[k] = V::load(rowp, lane + 32 * k);
        float2 a[4];
        float mean = 0.f;
        if constexpr (LN) {
#pragma unroll
          for (int i = 0; i < 4; ++i) a[i] = make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < SNC; ++k)
            if (SFULL || lane + 32 * k < nchunks) {
#pragma unroll
              for (int i = 0; i < 4; ++i) V::acc(a[i], raw[k], i);
            }
          mean = warp_sum((a[0].x + a[0].y) + (a[1].x + a[1].y) + (a[2].x + a[2].y) +
                          (a[3].x + a[3].y)) * inv_h;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < SNC; ++k)
          if (SFULL || lane + 32 * k < nchunks) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if constexpr (LN) {
                const float2 d = V::sub(raw[k], i, mean);
                a[i] = fma2(d, d, a[i]);
              } else {
                V::sq_acc(a[i], raw[k], i);
              }
            }
          }
        const float m2 = warp_sum((a[0].x + a[0].y) + (a[1].x + a[1].y) + (a[2].x + a[2].y) +
                                  (a[3].x + a[3].y));
        const float rs = __frsqrt_rn(m2 * inv_h + p.eps);
        if (lane == 0) {
          const int r = t * kTile + k;
          rstat[s] = make_float2(mean, rs);
          if (LN) p.mu[r] = mean;
          p.rsigma[r] = rs;
          // the tile barrier's phases are alias-free: stats warps run at
          // most a ring (Q rows) ahead of the apply warps and NT tile
          // barriers cover more than Q / 32 + 1 tiles
          mbar_arrive(smem_u32(&tready[(q / kTile) % NT]));
        }
      }
    }
    return;
  }

  // ---------------------------------------------------------- apply warps
  // Each apply warp takes 64-column sub-tiles of the 32-row tile (w, w + A,
  // ...).  Lane = hb*16 + rg*4 + cc: the thread holds y of rows 8rg..8rg+7
  // and of chunk cl = 4hb + cc of the sub-tile (columns 64 sub + 8 cl ..
  // + 7).  A row block (32 columns) spans the 4 lanes cc = 0..3 (shuffles
  // xor 1, 2); a column block (32 rows) spans the 4 lanes rg = 0..3
  // (shuffles xor 4, 8).
  const int hb = lane >> 4, rg = (lane >> 2) & 3, cc = lane & 3;
  const int cl = hb * 4 + cc;
  const int nsub = (nchunks + 7) >> 3;
  const int hs = H >> 5;  // row scales per row
  const int ns = N >> 5;  // column scales per column
  const uint32_t ring_u32 = smem_u32(ring);
  const bool rowwise = p.data != nullptr;
  const bool colwise = p.col_data != nullptr;

  RingPos pos{0u, 0u};
  int tl = 0;
  for (int tile = blockIdx.x; tile < p.n_tiles; tile += G, ++tl) {
    const int r0 = tile * kTile;
    if constexpr (STATS) {
      // the 32 rows' statistics are written (which implies they landed)
      mbar_wait(smem_u32(&tready[tl % NT]), (uint32_t)(tl / NT) & 1u, &g_err_mx, kErrReadyWait);
    } else {
      RingPos rp = pos;
      for (int k = 0; k < kTile; ++k) {
        mbar_wait(smem_u32(&full[rp.slot]), rp.phase, &g_err_mx, kErrFullWait);
        rp.advance(1, Q);
      }
    }
    uint32_t rowa[8];  // shared address of this thread's chunk in each of its 8 rows
    float2 st8[8];
    {
      RingPos rp = pos.ahead(8 * rg, Q);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        rowa[j] = ring_u32 + rp.slot * row_bytes + cl * kChunkBytes;
        st8[j] = STATS ? rstat[rp.slot] : make_float2(0.f, 1.f);
        rp.advance(1, Q);
      }
    }
    // output cursors of the tile (offset by sub-tile below)
    uint8_t* const dptr = rowwise ? p.data + ((size_t)(r0 + 8 * rg) * H + cl * 8) : nullptr;
    uint8_t* const sptr = rowwise ? p.row_scales + ((size_t)(r0 + 8 * rg) * hs + hb) : nullptr;
    uint8_t* const cptr = colwise ? p.col_data + ((size_t)cl * 8 * N + r0 + 8 * rg) : nullptr;
    uint8_t* const csptr = colwise ? p.col_scales + ((size_t)cl * 8 * ns + tile) : nullptr;

    for (int sub = warp; sub < nsub; sub += A) {
      const int c = sub * 8 + cl;  // chunk of 8 columns
      const bool valid = FULL || c < nchunks;
      float2 g2[4], b2[4];
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        float4 gv = make_float4(0.f, 0.f, 0.f, 0.f), bv = gv;
        if (STATS && valid) {
          gv = gsm[jj * nchunks + c];
          if (LN) bv = bsm[jj * nchunks + c];
        }
        g2[2 * jj] = make_float2(gv.x, gv.y);
        g2[2 * jj + 1] = make_float2(gv.z, gv.w);
        b2[2 * jj] = make_float2(bv.x, bv.y);
        b2[2 * jj + 1] = make_float2(bv.z, bv.w);
      }
      const uint32_t soff = (uint32_t)sub * 8 * kChunkBytes;
      float2 y[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int i = 0; i < 4; ++i) y[j][i] = make_float2(0.f, 0.f);
        if (valid) {
          const typename V::Raw raw = load8<TIn>(rowa[j] + soff);
          const float2 rs2 = splat2(st8[j].y);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if constexpr (LN)
              y[j][i] = fma2(mul2(V::sub(raw, i, st8[j].x), rs2), g2[i], b2[i]);
            else if constexpr (NK == kRms)
              y[j][i] = mul2(mul2(V::f32(raw, i), rs2), g2[i]);
            else
              y[j][i] = V::f32(raw, i);
          }
        }
      }
      // one sweep over |y|: row maxima (8 values each) and column maxima
      // (8 values each), two rows at a time
      float rmax[8], cmax[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        rmax[k] = 0.f;
        cmax[k] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a0 = fabsf(y[j][i].x), b0 = fabsf(y[j][i].y);
          const float a1 = fabsf(y[j + 1][i].x), b1 = fabsf(y[j + 1][i].y);
          rmax[j] = max3n(rmax[j], a0, b0);
          rmax[j + 1] = max3n(rmax[j + 1], a1, b1);
          cmax[2 * i] = max3n(cmax[2 * i], a0, a1);
          cmax[2 * i + 1] = max3n(cmax[2 * i + 1], b0, b1);
        }
      }
      // ------------------------------------------------- rowwise 1x32 blocks
      // a row block spans the lanes cc = 0..3 (lane bits 2 and 1); lane cc
      // encodes rows cc and cc + 4 and stores their scales
      if (rowwise) {
        float m0, m1;
        block_max_scatter(rmax, cc >> 1, cc & 1, 2, 1, m0, m1);
        const uint32_t code0 = e8m0_code(m0), code1 = e8m0_code(m1);
        float inv[8];
        gather8(e8m0_inv_scale(code0), e8m0_inv_scale(code1), cc >> 1, cc & 1, 2, 1, inv);
        if (valid) {
          uint8_t* dp = dptr + (size_t)sub * 64;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float2 iv = splat2(inv[j]);
            uint32_t q[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 v = mul2(y[j][i], iv);
              q[i] = pack_e4m3x2(v.x, v.y);
            }
            *reinterpret_cast<uint2*>(dp) = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
            dp += H;
          }
          uint8_t* sp = sptr + 2 * sub + (size_t)cc * hs;
          sp[0] = (uint8_t)code0;
          sp[4 * (size_t)hs] = (uint8_t)code1;
        }
      }
      // ---------------------------------------------- columnwise 32x1 blocks
      // a column block spans the lanes rg = 0..3 (lane bits 8 and 4); lane rg
      // encodes columns rg and rg + 4 and stores their scales
      if (colwise) {
        float m0, m1;
        block_max_scatter(cmax, rg >> 1, rg & 1, 8, 4, m0, m1);
        const uint32_t code0 = e8m0_code(m0), code1 = e8m0_code(m1);
        float cinv[8];
        gather8(e8m0_inv_scale(code0), e8m0_inv_scale(code1), rg >> 1, rg & 1, 8, 4, cinv);
        if (valid) {
          uint8_t* cp = cptr + (size_t)sub * 64 * N;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 ci = make_float2(cinv[2 * i], cinv[2 * i + 1]);
            float2 qv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) qv[j] = mul2(y[j][i], ci);
            const uint32_t lo0 = pack_e4m3x2(qv[0].x, qv[1].x) | (pack_e4m3x2(qv[2].x, qv[3].x) << 16);
            const uint32_t hi0 = pack_e4m3x2(qv[4].x, qv[5].x) | (pack_e4m3x2(qv[6].x, qv[7].x) << 16);
            const uint32_t lo1 = pack_e4m3x2(qv[0].y, qv[1].y) | (pack_e4m3x2(qv[2].y, qv[3].y) << 16);
            const uint32_t hi1 = pack_e4m3x2(qv[4].y, qv[5].y) | (pack_e4m3x2(qv[6].y, qv[7].y) << 16);
            *reinterpret_cast<uint2*>(cp) = make_uint2(lo0, hi0);
            *reinterpret_cast<uint2*>(cp + N) = make_uint2(lo1, hi1);
            cp += 2 * (size_t)N;
          }
          uint8_t* csp = csptr + ((size_t)sub * 64 + rg) * ns;
          csp[0] = (uint8_t)code0;
          csp[4 * (size_t)ns] = (uint8_t)code1;
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

// ---------------------------------------------------------------------------
// Slab kernel (bf16, H a multiple of kMxSlabCols).  The ring kernel above
// must hold a whole 32-row tile (the height of a column block) in shared
// memory until every sub-tile of it is quantized; at H = 2048 its ring holds
// about 52 rows, so the next tile's loads overlap only part of the current
// tile's work.  Here the two uses of x are split:
//   row producer  one lane streams whole rows (HBM -> shared, through L2)
//                 into a row ring of about 80 KB (enough in flight for the
//                 SM's share of HBM bandwidth);
//   stats warps   take a row into registers, free its slot at once, and
//                 write mean / rsigma into the tile's statistics buffer
//                 (NT buffers, so statistics run up to NT tiles ahead; the
//                 tile's "ready" barrier counts its 32 rows);
//   slab producer one lane copies, once a tile's statistics are ready, each
//                 32-row x kMxSlabCols slab of it again, now from L2, into a
//                 ring of slabs with one 2-D tensor copy (TMA) a slab;
//   apply warps   warp w takes slabs w, w + A, ... of every tile: the same
//                 8 x 8 register blocks, maxima and codes as the ring kernel,
//                 for the 64-column sub-tile(s) of a slab; then it frees
//                 the slab and, after its last slab of the tile, arrives on
//                 the tile's "done" barrier, which the stats warps wait on
//                 before reusing the tile's statistics buffer.
// HBM reads x about once; the slab copies mostly hit L2 (the rows were read
// moments before).  Six stats warps keep up with LayerNorm's two passes
// (with four the kernel waited on them: 170 vs 146 us at 65536 x 2048).
// Slot reuse is alias-free: the row ring has a multiple of S
// slots and the slab ring a multiple of A, so every slot is always consumed
// by the same warp, which released its previous use itself.
// one 32-row x kMxSlabCols box of x (tensor map `tm`: columns, then rows)
// into shared memory, completion on `bar`
__device__ __forceinline__ void tma_load_box(uint32_t dst, const CUtensorMap* tm, int col, int row,
                                             uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(col), "r"(row), "r"(bar), "l"(pol)
      : "memory");
}

template <int NK, int SNC>
__global__ void __launch_bounds__(kMaxThreads, 1)
    rn_mx_slab_kernel(const MxParams p, const __grid_constant__ CUtensorMap tmx) {
  using V = Vec<uint16_t, 8>;
  constexpr bool LN = (NK == kLn);
  constexpr uint32_t kPieceBytes = kMxSlabCols * 2;  // one row of a slab
  constexpr uint32_t kSlabBytes = kTile * kPieceBytes;
  extern __shared__ __align__(128) unsigned char smem[];
  const int A = p.apply_warps;
  const int S = p.stats_warps;
  const int H = p.H;
  const int N = p.N;
  const int nchunks = H >> 3;
  const uint32_t row_bytes = (uint32_t)H * 2;
  const int nslab = H / kMxSlabCols;
  const uint32_t Qs = (uint32_t)p.Qs, Qa = (uint32_t)p.Q;
  const int NT = p.n_tbar;
  const size_t gb_bytes = (size_t)H * sizeof(float) * (LN ? 2 : 1);

  float4* gsm = reinterpret_cast<float4*>(smem);  // [2][nchunks]
  float4* bsm = gsm + 2 * (size_t)nchunks;
  unsigned char* sring = smem + gb_bytes;                        // [Qs] rows
  unsigned char* aring = sring + (size_t)Qs * row_bytes;         // [Qa] slabs
  float2* tstat = reinterpret_cast<float2*>(aring + (size_t)Qa * kSlabBytes);  // [NT][32]
  uint64_t* sfull = reinterpret_cast<uint64_t*>(tstat + (size_t)NT * kTile);
  uint64_t* sempty = sfull + Qs;
  uint64_t* afull = sempty + Qs;
  uint64_t* aempty = afull + Qa;
  uint64_t* tready = aempty + Qa;  // [NT] 32 rows' statistics written
  uint64_t* tdone = tready + NT;   // [NT] every apply warp finished the tile

  for (uint32_t i = threadIdx.x; i < Qs; i += blockDim.x) {
    mbar_init(smem_u32(&sfull[i]), 1);
    mbar_init(smem_u32(&sempty[i]), 1);
    fence_barrier_init();
  }
  for (uint32_t i = threadIdx.x; i < Qa; i += blockDim.x) {
    mbar_init(smem_u32(&afull[i]), 1);
    mbar_init(smem_u32(&aempty[i]), 1);
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i < NT; i += blockDim.x) {
    mbar_init(smem_u32(&tready[i]), kTile);
    mbar_init(smem_u32(&tdone[i]), A);
    fence_barrier_init();
  }
  {
    const int n4 = H / 4;
    for (int u = threadIdx.x; u < n4; u += blockDim.x) {
      const int c = u >> 1, j = u & 1;
      const float4 gv = reinterpret_cast<const float4*>(p.gamma)[u];
      gsm[j * nchunks + c] =
          p.zcg ? make_float4(1.0f + gv.x, 1.0f + gv.y, 1.0f + gv.z, 1.0f + gv.w) : gv;
      if (LN)
        bsm[j * nchunks + c] = p.beta ? reinterpret_cast<const float4*>(p.beta)[u]
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int ntl = p.n_tiles > (int)blockIdx.x ? (p.n_tiles - 1 - (int)blockIdx.x) / G + 1 : 0;
  const int nq = ntl * kTile;
  const unsigned char* xb = static_cast<const unsigned char*>(p.x);

  if (warp == A + S) {
    // -------------------------------------------------------- row producer
    if (lane == 0) {
      for (int q = 0; q < nq; ++q) {
        const int r = ((int)blockIdx.x + (q / kTile) * G) * kTile + (q % kTile);
        const uint32_t s = (uint32_t)q % Qs;
        if (q >= (int)Qs)
          mbar_wait(smem_u32(&sempty[s]), ((uint32_t)q / Qs - 1u) & 1u, &g_err_mx, kErrEmptyWait);
        mbar_arrive_expect_tx(smem_u32(&sfull[s]), row_bytes);
        bulk_g2s(smem_u32(sring + (size_t)s * row_bytes), xb + (size_t)r * row_bytes, row_bytes,
                 smem_u32(&sfull[s]));
      }
      for (int q = nq > (int)Qs ? nq - (int)Qs : 0; q < nq; ++q)
        mbar_wait(smem_u32(&sfull[q % Qs]), ((uint32_t)q / Qs) & 1u, &g_err_mx, kErrDrainWait);
    }
    return;
  }

  if (warp == A + S + 1) {
    // ------------------------------------------------------- slab producer
    // one tensor copy a slab (a copy per row piece would cost ~36 ns each
    // in the copy engine, 32 times a slab)
    if (lane == 0) {
      const uint64_t pol = l2_evict_first();  // the second and last read
      for (int tl = 0; tl < ntl; ++tl) {
        const int t = (int)blockIdx.x + tl * G;
        mbar_wait(smem_u32(&tready[tl % NT]), (uint32_t)(tl / NT) & 1u, &g_err_mx, kErrReadyWait);
        for (int j = 0; j < nslab; ++j) {
          const uint32_t i = (uint32_t)(tl * nslab + j);
          const uint32_t s = i % Qa;
          if (i >= Qa)
            mbar_wait(smem_u32(&aempty[s]), (i / Qa - 1u) & 1u, &g_err_mx, kErrEmptyWait);
          mbar_arrive_expect_tx(smem_u32(&afull[s]), kSlabBytes);
          tma_load_box(smem_u32(aring + (size_t)s * kSlabBytes), &tmx, j * kMxSlabCols, t * kTile,
                       smem_u32(&afull[s]), pol);
        }
      }
      const uint32_t ni = (uint32_t)(ntl * nslab);
      for (uint32_t i = ni > Qa ? ni - Qa : 0; i < ni; ++i)
        mbar_wait(smem_u32(&afull[i % Qa]), (i / Qa) & 1u, &g_err_mx, kErrDrainWait);
    }
    return;
  }

  if (warp >= A) {
    // --------------------------------------------------------- stats warps
    const int j = warp - A;
    const float inv_h = 1.0f / (float)H;
    for (int q = j; q < nq; q += S) {
      const int tl = q / kTile, k = q % kTile;
      // the statistics buffer of tile tl was last used by tile tl - NT
      if (tl >= NT)
        mbar_wait(smem_u32(&tdone[tl % NT]), (uint32_t)(tl / NT - 1) & 1u, &g_err_mx, kErrStatsWait);
      const uint32_t s = (uint32_t)q % Qs;
      mbar_wait(smem_u32(&sfull[s]), ((uint32_t)q / Qs) & 1u, &g_err_mx, kErrStatsWait);
      const unsigned char* rowp = sring + (size_t)s * row_bytes;
      typename V::Raw raw[SNC];
#pragma unroll
      for (int c = 0; c < SNC; ++c)
        if (lane + 32 * c < nchunks) raw[c] = V::load(rowp, lane + 32 * c);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sempty[s]));
      float2 a[4];
      float mean = 0.f;
      if constexpr (LN) {
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < SNC; ++c)
          if (lane + 32 * c < nchunks) {
#pragma unroll
            for (int i = 0; i < 4; ++i) V::acc(a[i], raw[c], i);
          }
        mean = warp_sum((a[0].x + a[0].y) + (a[1].x + a[1].y) + (a[2].x + a[2].y) +
                        (a[3].x + a[3].y)) * inv_h;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < SNC; ++c)
        if (lane + 32 * c < nchunks) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if constexpr (LN) {
              const float2 d = V::sub(raw[c], i, mean);
              a[i] = fma2(d, d, a[i]);
            } else {
              V::sq_acc(a[i], raw[c], i);
            }
          }
        }
      const float m2 = warp_sum((a[0].x + a[0].y) + (a[1].x + a[1].y) + (a[2].x + a[2].y) +
                                (a[3].x + a[3].y));
      const float rs = __frsqrt_rn(m2 * inv_h + p.eps);
      if (lane == 0) {
        const int r = ((int)blockIdx.x + tl * G) * kTile + k;
        tstat[(tl % NT) * kTile + k] = make_float2(mean, rs);
        if (LN) p.mu[r] = mean;
        p.rsigma[r] = rs;
        mbar_arrive(smem_u32(&tready[tl % NT]));
      }
    }
    return;
  }

  // ---------------------------------------------------------- apply warps
  // lane = hb*16 + rg*4 + cc as in the ring kernel: rows 8rg..8rg+7, chunk
  // cl = 4hb + cc of a 64-column sub-tile
  const int hb = lane >> 4, rg = (lane >> 2) & 3, cc = lane & 3;
  const int cl = hb * 4 + cc;
  const int hs = H >> 5;
  const int ns = N >> 5;
  const bool rowwise = p.data != nullptr;
  const bool colwise = p.col_data != nullptr;
  const uint32_t aring_u32 = smem_u32(aring);

  for (int tl = 0; tl < ntl; ++tl) {
    const int tile = (int)blockIdx.x + tl * G;
    const int r0 = tile * kTile;
    mbar_wait(smem_u32(&tready[tl % NT]), (uint32_t)(tl / NT) & 1u, &g_err_mx, kErrReadyWait);
    float2 st8[8];
#pragma unroll
    for (int jr = 0; jr < 8; ++jr) st8[jr] = tstat[(tl % NT) * kTile + 8 * rg + jr];
    uint8_t* const dptr = rowwise ? p.data + ((size_t)(r0 + 8 * rg) * H + cl * 8) : nullptr;
    uint8_t* const sptr = rowwise ? p.row_scales + ((size_t)(r0 + 8 * rg) * hs + hb) : nullptr;
    uint8_t* const cptr = colwise ? p.col_data + ((size_t)cl * 8 * N + r0 + 8 * rg) : nullptr;
    uint8_t* const csptr = colwise ? p.col_scales + ((size_t)cl * 8 * ns + tile) : nullptr;

    for (int js = warp; js < nslab; js += A) {
      const uint32_t i = (uint32_t)(tl * nslab + js);
      const uint32_t s = i % Qa;
      mbar_wait(smem_u32(&afull[s]), (i / Qa) & 1u, &g_err_mx, kErrFullWait);
      const uint32_t slab = aring_u32 + s * kSlabBytes + 8 * rg * kPieceBytes;
#pragma unroll 1
      for (int u = 0; u < kMxSlabCols / 64; ++u) {
        const int sub = js * (kMxSlabCols / 64) + u;  // 64-column sub-tile of the row
        const int c = sub * 8 + cl;
        float2 g2[4], b2[4];
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const float4 gv = gsm[jj * nchunks + c];
          const float4 bv = LN ? bsm[jj * nchunks + c] : make_float4(0.f, 0.f, 0.f, 0.f);
          g2[2 * jj] = make_float2(gv.x, gv.y);
          g2[2 * jj + 1] = make_float2(gv.z, gv.w);
          b2[2 * jj] = make_float2(bv.x, bv.y);
          b2[2 * jj + 1] = make_float2(bv.z, bv.w);
        }
        const uint32_t coff = (uint32_t)(u * 64 + cl * 8) * 2;
        float2 y[8][4];
#pragma unroll
        for (int jr = 0; jr < 8; ++jr) {
          const typename V::Raw raw = load8<uint16_t>(slab + jr * kPieceBytes + coff);
          const float2 rs2 = splat2(st8[jr].y);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if constexpr (LN)
              y[jr][q] = fma2(mul2(V::sub(raw, q, st8[jr].x), rs2), g2[q], b2[q]);
            else
              y[jr][q] = mul2(mul2(V::f32(raw, q), rs2), g2[q]);
          }
        }
        float rmax[8], cmax[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          rmax[k] = 0.f;
          cmax[k] = 0.f;
        }
#pragma unroll
        for (int jr = 0; jr < 8; jr += 2) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float a0 = fabsf(y[jr][q].x), b0 = fabsf(y[jr][q].y);
            const float a1 = fabsf(y[jr + 1][q].x), b1 = fabsf(y[jr + 1][q].y);
            rmax[jr] = max3n(rmax[jr], a0, b0);
            rmax[jr + 1] = max3n(rmax[jr + 1], a1, b1);
            cmax[2 * q] = max3n(cmax[2 * q], a0, a1);
            cmax[2 * q + 1] = max3n(cmax[2 * q + 1], b0, b1);
          }
        }
        if (rowwise) {
          float m0, m1;
          block_max_scatter(rmax, cc >> 1, cc & 1, 2, 1, m0, m1);
          const uint32_t code0 = e8m0_code(m0), code1 = e8m0_code(m1);
          float inv[8];
          gather8(e8m0_inv_scale(code0), e8m0_inv_scale(code1), cc >> 1, cc & 1, 2, 1, inv);
          uint8_t* dp = dptr + (size_t)sub * 64;
#pragma unroll
          for (int jr = 0; jr < 8; ++jr) {
            const float2 iv = splat2(inv[jr]);
            uint32_t q4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 v = mul2(y[jr][q], iv);
              q4[q] = pack_e4m3x2(v.x, v.y);
            }
            *reinterpret_cast<uint2*>(dp) = make_uint2(q4[0] | (q4[1] << 16), q4[2] | (q4[3] << 16));
            dp += H;
          }
          uint8_t* sp = sptr + 2 * sub + (size_t)cc * hs;
          sp[0] = (uint8_t)code0;
          sp[4 * (size_t)hs] = (uint8_t)code1;
        }
        if (colwise) {
          float m0, m1;
          block_max_scatter(cmax, rg >> 1, rg & 1, 8, 4, m0, m1);
          const uint32_t code0 = e8m0_code(m0), code1 = e8m0_code(m1);
          float cinv[8];
          gather8(e8m0_inv_scale(code0), e8m0_inv_scale(code1), rg >> 1, rg & 1, 8, 4, cinv);
          uint8_t* cp = cptr + (size_t)sub * 64 * N;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 ci = make_float2(cinv[2 * q], cinv[2 * q + 1]);
            float2 qv[8];
#pragma unroll
            for (int jr = 0; jr < 8; ++jr) qv[jr] = mul2(y[jr][q], ci);
            const uint32_t lo0 = pack_e4m3x2(qv[0].x, qv[1].x) | (pack_e4m3x2(qv[2].x, qv[3].x) << 16);
            const uint32_t hi0 = pack_e4m3x2(qv[4].x, qv[5].x) | (pack_e4m3x2(qv[6].x, qv[7].x) << 16);
            const uint32_t lo1 = pack_e4m3x2(qv[0].y, qv[1].y) | (pack_e4m3x2(qv[2].y, qv[3].y) << 16);
            const uint32_t hi1 = pack_e4m3x2(qv[4].y, qv[5].y) | (pack_e4m3x2(qv[6].y, qv[7].y) << 16);
            *reinterpret_cast<uint2*>(cp) = make_uint2(lo0, hi0);
            *reinterpret_cast<uint2*>(cp + N) = make_uint2(lo1, hi1);
            cp += 2 * (size_t)N;
          }
          uint8_t* csp = csptr + ((size_t)sub * 64 + rg) * ns;
          csp[0] = (uint8_t)code0;
          csp[4 * (size_t)ns] = (uint8_t)code1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&aempty[s]));
    }
    if (lane == 0) mbar_arrive(smem_u32(&tdone[tl % NT]));
  }
}

// cuTensorMapEncodeTiled, fetched once through the runtime (no link against
// the driver library)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

template <int NK, int SNC>
rn_status launch_slab_t(const MxParams& p, const Launch& l, cudaStream_t s) {
  auto k = rn_mx_slab_kernel<NK, SNC>;
  if (l.threads > kMaxThreads || p.H % kMxSlabCols != 0 || p.H / 8 > 32 * SNC || p.n_tbar < 2 ||
      p.Qs < p.stats_warps || p.Qs % p.stats_warps != 0 || p.Q % p.apply_warps != 0 ||
      (p.H / kMxSlabCols) % p.apply_warps != 0 || l.threads != 32 * (p.apply_warps + p.stats_warps + 2))
    return RN_ERR_UNSUPPORTED;
  EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr) return RN_ERR_CUDA;
  // x as a 2-D bf16 tensor [N rows][H columns]; boxes of 32 rows x kMxSlabCols
  // columns (128 bytes a row: the inner extent is a multiple of 16 bytes)
  CUtensorMap tm;
  const cuuint64_t dims[2] = {(cuuint64_t)p.H, (cuuint64_t)p.N};
  const cuuint64_t strides[1] = {(cuuint64_t)p.H * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kMxSlabCols, (cuuint32_t)kTile};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return RN_ERR_CUDA;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l.smem) !=
      cudaSuccess)
    return RN_ERR_CUDA;
  int grid = 1;
  if (persistent_grid(k, l, &grid) != RN_OK) return RN_ERR_CUDA;
  k<<<grid, l.threads, l.smem, s>>>(p, tm);
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

template <typename TIn, int NK, bool FULL, int SNC, bool SFULL>
rn_status launch_t(const MxParams& p, const Launch& l, cudaStream_t s) {
  auto k = rn_mx_kernel<TIn, NK, FULL, SNC, SFULL>;
  if (l.threads > kMaxThreads || p.n_tbar < 1 || p.H / 8 > 32 * SNC) return RN_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l.smem) !=
      cudaSuccess)
    return RN_ERR_CUDA;
  int grid = 1;
  if (persistent_grid(k, l, &grid) != RN_OK) return RN_ERR_CUDA;
  k<<<grid, l.threads, l.smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

// bf16 H = 2048 takes the exact shape (whole sub-tiles, 8 chunks a stats
// lane); other H multiples of 64 / of 32 the general ones, with stats lanes
// of up to 16 chunks for bf16 (H <= 4096) and 8 for fp32 (H <= 2048, which
// the ring of >= 33 fp32 rows does not reach anyway)
template <typename TIn, int NK>
rn_status launch_f(const MxParams& p, const Launch& l, cudaStream_t s) {
  constexpr int kSnc = sizeof(TIn) == 2 ? 16 : 8;
  if (sizeof(TIn) == 2 && p.H == 2048) return launch_t<TIn, NK, true, 8, true>(p, l, s);
  if (p.H % 64 == 0) return launch_t<TIn, NK, true, kSnc, false>(p, l, s);
  return launch_t<TIn, NK, false, kSnc, false>(p, l, s);
}

}  // namespace

rn_status launch_mx(int nk, bool bf16, int ng, const MxParams& p, const Launch& l,
                    cudaStream_t s) {
  (void)ng;
  if (nk == kIdentity) return bf16 ? RN_ERR_UNSUPPORTED : launch_f<float, kIdentity>(p, l, s);
  if (bf16) return nk == kLn ? launch_f<uint16_t, kLn>(p, l, s) : launch_f<uint16_t, kRms>(p, l, s);
  return nk == kLn ? launch_f<float, kLn>(p, l, s) : launch_f<float, kRms>(p, l, s);
}

rn_status launch_mx_slab(int nk, const MxParams& p, const Launch& l, cudaStream_t s) {
  if (nk == kLn) return p.H <= 2048 ? launch_slab_t<kLn, 8>(p, l, s) : launch_slab_t<kLn, 16>(p, l, s);
  if (nk == kRms) return p.H <= 2048 ? launch_slab_t<kRms, 8>(p, l, s) : launch_slab_t<kRms, 16>(p, l, s);
  return RN_ERR_UNSUPPORTED;
}

rn_status read_clear_error_mx(unsigned* code) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_mx, sizeof(v)) != cudaSuccess) return RN_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_err_mx, &zero, sizeof(zero)) != cudaSuccess) return RN_ERR_CUDA;
  *code = v;
  return RN_OK;
}

}  // namespace rn
