// LayerNorm / RMSNorm forward fused with MXFP8 output quantization: 1x32
// rowwise and 32x1 columnwise blocks, each with an E8M0 shared scale (page
// "Implementation:NVIDIA TransformerEngine PyTorch Ext Normalization",
// section "Description": the fully fused MXFP8 path).
//
// Two kernels: rn_mx_box_kernel (further below) for rows of whole 128-byte
// column blocks (bf16 H a multiple of 64, every fp32 row, the stand-alone
// quantizer), and the ring kernel described here for the other bf16 rows (H
// of 32 mod 64 columns).
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
// Box kernel (bf16 rows of whole 64-column blocks, fp32 rows, the stand-alone
// quantizer).  The ring kernel above must hold a whole 32-row tile (the
// height of a column block) in shared memory until every sub-tile of it is
// quantized, and its statistics warps and apply warps, fixed in number, leave
// one of the two sides idle.  Here:
//   * x moves in boxes of 32 rows x 4 column blocks of 128 bytes (16 KB, 256
//     bf16 / 128 fp32 columns), one 3-D tensor copy each (dimensions: the
//     128-byte column block, rows, column blocks) with the 128-byte swizzle
//     (chunk c of row r of a column block sits at chunk c ^ (r & 7)), so a
//     warp reading 8 rows' same chunk, or one row's 8 chunks, touches every
//     bank once;
//   * a tile is read twice: its boxes come from HBM for the row statistics
//     (partial sums of each row over half a box, a lane per row, no cross-lane
//     reduction) and again, from L2 moments later, for the quantization (the
//     8 x 8 register blocks, both directions); no buffer holds a whole tile,
//     so any row length fits;
//   * 16 worker warps each do both kinds of work, in rounds: round k merges
//     the partials of tile k - 1 into mu / rsigma (two rows a warp: the mean
//     from the partial sums, then the sum of squared deviations as the
//     partials' own plus n (m_u - mean)^2, both added in a fixed order), takes
//     its share of tile k's statistics half-units and then of tile k - 1's
//     64-column sub-tiles; a named barrier closes the round;
//   * there is no producer warp (a 17th warp would leave 96 registers a
//     thread: the register file of an SM quarter serves its 5 warps): the
//     copies form one sequence in the order the rounds consume them (tile
//     k's statistics boxes, then tile k - 1's quantization boxes), load i
//     going to ring slot i mod Q; thread 0 issues the first Q, and the unit
//     whose release brings a slot's pending-read count to zero issues the
//     slot's next load at once (acquire-release count, then a proxy fence
//     before the copy overwrites what was read); the slot's ticket, set
//     before each refill, makes every consumer's wait alias-free.
// bf16 enters the arithmetic through explicit unpacking (shift / mask) and
// the packed f32x2 instructions.
constexpr int kBoxRows = 32;                                      // a tile
constexpr int kBoxCb = 4;                                         // 128-byte column blocks a box
constexpr uint32_t kBoxBytes = (uint32_t)kBoxRows * 128 * kBoxCb;  // 16 KB
constexpr int kBoxWorkers = 16;
constexpr int kBoxThreads = 32 * kBoxWorkers;

// Lanes of a quantization sub-tile: lane = hb*16 + rg*4 + cc (a quarter warp
// reads two rows' half chunks), or with kLaneRowMajor lane = rg*8 + hb*4 + cc
// (a quarter warp reads one row's 8 chunks, which the swizzle spreads over
// all banks).  Row blocks span the lanes cc (shuffles xor 1, 2), column
// blocks the lanes rg (xor kColS0, kColS1).
constexpr bool kLaneRowMajor = false;
constexpr int kColS0 = kLaneRowMajor ? 8 : 4;
constexpr int kColS1 = kLaneRowMajor ? 16 : 8;

// one box (32 rows x kBoxCb column blocks from column block `cb`, rows from
// `row`) into shared memory, completion on `bar`
__device__ __forceinline__ void tma_load_box3(uint32_t dst, const CUtensorMap* tm, int row, int cb,
                                              uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(row), "r"(cb), "r"(bar), "l"(pol)
      : "memory");
}

// slot (index mod Q) and use (index / Q) of a ring load index, moved forward
struct LoadPos {
  uint32_t idx, slot, use;
  __device__ __forceinline__ void to(uint32_t target, uint32_t q) {
    uint32_t d = target - idx;
    idx = target;
    while (d >= q) {
      d -= q;
      ++use;
    }
    slot += d;
    if (slot >= q) {
      slot -= q;
      ++use;
    }
  }
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// the four element pairs of a 16-byte chunk as fp32 pairs (bf16: 8 elements,
// pairs 0..3; fp32: 4 elements, pairs 0..1)
template <typename TIn>
__device__ __forceinline__ float2 chunk_pair(const uint4& v, int i);
template <>
__device__ __forceinline__ float2 chunk_pair<uint16_t>(const uint4& v, int i) {
  const uint32_t w = i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
template <>
__device__ __forceinline__ float2 chunk_pair<float>(const uint4& v, int i) {
  return i == 0 ? make_float2(__uint_as_float(v.x), __uint_as_float(v.y))
                : make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
}

template <typename TIn, int NK>
__global__ void __launch_bounds__(kBoxThreads, 1)
    rn_mx_box_kernel(const MxParams p, const __grid_constant__ CUtensorMap tmx) {
  constexpr int ESZ = (int)sizeof(TIn);
  constexpr int C0 = 128 / ESZ;          // columns a column block holds
  constexpr int SPB = C0 * kBoxCb / 64;  // 64-column sub-tiles a box holds (4 bf16, 2 fp32)
  constexpr int PPC = 8 / ESZ;           // element pairs a 16-byte chunk holds (4 bf16, 2 fp32)
  constexpr bool STATS = (NK != kIdentity);
  constexpr bool LN = (NK == kLn);
  // arrivals that release one use of a box slot: one from each of its SPB
  // sub-tiles, or EMPTY / 2 from each of its two statistics half-units
  constexpr uint32_t EMPTY = SPB > 2 ? SPB : 2;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // the 128-byte swizzle wants boxes at 1024-byte boundaries
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int H = p.H;
  const int N = p.N;
  const uint32_t Q = (uint32_t)p.Q;
  const int ncb = H / C0;                      // column blocks of a row
  const int nbox = (ncb + kBoxCb - 1) / kBoxCb;
  const int nus = STATS ? 2 * nbox : 0;        // statistics half-units a tile
  const int nua = nbox * SPB;                  // sub-tiles a tile (some may lie past H)
  unsigned char* ring = smem;
  float2* pbuf = reinterpret_cast<float2*>(ring + (size_t)Q * kBoxBytes);  // [2][nus][32]
  float2* tstat = pbuf + 2 * (size_t)nus * kBoxRows;                       // [2][32] (-mean rsigma, rsigma)
  uint64_t* full = reinterpret_cast<uint64_t*>(tstat + 2 * kBoxRows);
  uint64_t* tready = full + Q;                                             // [2]
  uint64_t* sdone = tready + 2;                                            // [2]
  uint32_t* ticket = reinterpret_cast<uint32_t*>(sdone + 2);               // [Q]
  uint32_t* pending = ticket + Q;                                          // [Q] reads left

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int ntl = p.n_tiles > (int)blockIdx.x ? (p.n_tiles - 1 - (int)blockIdx.x) / G + 1 : 0;
  // round k: statistics of tile k, quantization of tile k - 1 (the
  // stand-alone quantizer: quantization of tile k only)
  const int nrounds = STATS ? ntl + 1 : ntl;
  const uint32_t nload = (uint32_t)(STATS ? 2 : 1) * (uint32_t)ntl * (uint32_t)nbox;
  const uint32_t ring_u32 = smem_u32(ring);
  const uint64_t keep = l2_evict_last();   // statistics read: read again soon
  const uint64_t once = l2_evict_first();  // quantization read: the last

  // load i of the sequence into slot i mod Q (its ticket set first)
  auto issue = [&](uint32_t i) {
    const uint32_t s = i % Q, u = i / Q;
    int t, b;
    bool first;
    if (!STATS) {
      t = (int)(i / (uint32_t)nbox);
      b = (int)(i - (uint32_t)t * nbox);
      first = false;
    } else if (i < (uint32_t)nbox) {
      t = 0;
      b = (int)i;
      first = true;
    } else {
      // rounds 1 .. ntl: tile k's statistics boxes (while k < ntl), then tile
      // k - 1's quantization boxes
      const uint32_t j = i - (uint32_t)nbox;
      const int k = 1 + (int)(j / (uint32_t)(2 * nbox));
      const int r = (int)(j - (uint32_t)(k - 1) * 2 * nbox);
      first = (k < ntl) && r < nbox;
      t = first ? k : k - 1;
      b = first ? r : (k < ntl ? r - nbox : r);
    }
    ticket_set(smem_u32(&ticket[s]), u);
    mbar_arrive_expect_tx(smem_u32(&full[s]), kBoxBytes);
    tma_load_box3(ring_u32 + s * kBoxBytes, &tmx, ((int)blockIdx.x + t * G) * kBoxRows, b * kBoxCb,
                  smem_u32(&full[s]), first ? keep : once);
  };
  // a unit done with slot s (use u) gives back its `cnt` reads; the last
  // one refills the slot with load u Q + Q + s
  auto release = [&](uint32_t s, uint32_t u, uint32_t cnt) {
    __syncwarp();
    if (lane == 0) {
      uint32_t old;
      asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
                   : "=r"(old)
                   : "r"(smem_u32(&pending[s])), "r"(0u - cnt)
                   : "memory");
      if (old == cnt) {
        const uint32_t nxt = (u + 1) * Q + s;
        pending[s] = EMPTY;
        if (nxt < nload) {
          fence_proxy_async();  // the reads of the slot before the copy that overwrites it
          issue(nxt);
        }
      }
    }
  };

  for (uint32_t i = threadIdx.x; i < Q; i += blockDim.x) {
    mbar_init(smem_u32(&full[i]), 1);
    ticket[i] = 0xFFFFFFFFu;
    pending[i] = EMPTY;
  }
  if (threadIdx.x < 2) {
    mbar_init(smem_u32(&tready[threadIdx.x]), 1);
    mbar_init(smem_u32(&sdone[threadIdx.x]), kBoxWorkers);
  }
  fence_barrier_init();
  __syncthreads();
  if (threadIdx.x == 0)
    for (uint32_t i = 0; i < Q && i < nload; ++i) issue(i);

  // ------------------------------------------------------------- workers
  const int w = warp;
  const float inv_h = 1.0f / (float)H;
  // quantization lanes: rows 8rg..8rg+7 and chunk cl = 4hb + cc (columns
  // 8cl..8cl+7) of a 64-column sub-tile (the lane layout: kLaneRowMajor)
  const int hb = kLaneRowMajor ? (lane >> 2) & 1 : lane >> 4;
  const int rg = kLaneRowMajor ? lane >> 3 : (lane >> 2) & 3;
  const int cc = lane & 3;
  const int cl = hb * 4 + cc;
  const int hs = H >> 5;
  const int ns = N >> 5;
  const bool rowwise = p.data != nullptr;
  const bool colwise = p.col_data != nullptr;
  LoadPos pos{0u, 0u, 0u};
  uint32_t li = 0;  // ring load index of the first box of the current pass

  for (int k = 0; k < nrounds; ++k) {
    const int ta = STATS ? k - 1 : k;  // the tile quantized in this round
    if constexpr (STATS) {
      // Tile t's statistics units are done once every worker arrived on
      // sdone[t & 1]; worker t mod 16 then merges the tile (a lane per row,
      // its partials added in unit order) and arrives on tready[t & 1], which
      // every worker waits on before quantizing the tile.  Each worker's
      // units of tile t come after its quantization of tile t - 2, and the
      // merge of tile t after every worker's units of tile t, so the partial
      // and (mean, rsigma) buffers are free again when rewritten and no
      // barrier phase can alias (every wait or arrival for tile t follows the
      // completion of tile t - 2's phase of the same barrier).
      if (ta >= 0 && w == (ta & (kBoxWorkers - 1))) {
        mbar_wait(smem_u32(&sdone[ta & 1]), (uint32_t)(ta >> 1) & 1u, &g_err_mx, kErrReadyWait);
        // ---------------------------------------------------------- merge
        const float2* pb = pbuf + (size_t)(ta & 1) * nus * kBoxRows + lane;
        float mean = 0.0f, m2 = 0.0f;
        if constexpr (LN) {
          float sx = 0.0f;
          for (int u = 0; u < nus; ++u) sx += pb[u * kBoxRows].x;
          mean = sx * inv_h;
          for (int u = 0; u < nus; ++u) {
            const int cb0 = (u >> 1) * kBoxCb + 2 * (u & 1);
            const int nv = (cb0 < ncb) + (cb0 + 1 < ncb);
            if (nv > 0) {
              const float2 v = pb[u * kBoxRows];
              const float nf = (float)(nv * C0);  // a power of two
              const float d = v.x * (nv == 2 ? 1.0f / (2 * C0) : 1.0f / C0) - mean;
              m2 += v.y + nf * d * d;
            }
          }
        } else {
          for (int u = 0; u < nus; ++u) m2 += pb[u * kBoxRows].x;
        }
        const float rs = __frsqrt_rn(m2 * inv_h + p.eps);
        const int row = ((int)blockIdx.x + ta * G) * kBoxRows + lane;
        // (-mean rsigma, rsigma): the apply forms x rsigma - mean rsigma with
        // one fma
        tstat[(ta & 1) * kBoxRows + lane] = make_float2(-mean * rs, rs);
        if (LN) p.mu[row] = mean;
        p.rsigma[row] = rs;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tready[ta & 1]));
      }
      if (k < ntl) {
        // ----------------------------------------------- statistics units
        // half-unit u: rows 0..31 (lane = row) x column blocks
        // 2 (u & 1), +1 of box u >> 1; LayerNorm: (sum, sum of squared
        // deviations from the unit's own mean), RMSNorm: (sum of squares, 0)
        float2* pw = pbuf + (size_t)(k & 1) * nus * kBoxRows;
        for (int u = w; u < nus; u += kBoxWorkers) {
          pos.to(li + (uint32_t)(u >> 1), Q);
          const uint32_t s = pos.slot;
          ticket_wait(smem_u32(&ticket[s]), pos.use, &g_err_mx, kErrStatsWait);
          mbar_wait(smem_u32(&full[s]), pos.use & 1u, &g_err_mx, kErrStatsWait);
          const int cb0 = (u >> 1) * kBoxCb + 2 * (u & 1);
          const int nv = min(2, ncb - cb0);  // valid column blocks (0..2), the same on every lane
          const uint32_t base = ring_u32 + s * kBoxBytes + (uint32_t)(u & 1) * 2 * 4096 +
                                (uint32_t)lane * 128;
          // chunk c of column block h of this lane's row
          auto chunk = [&](int h, int c) { return lds128(base + h * 4096 + ((c ^ (lane & 7)) << 4)); };
          float2 a[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) a[i] = make_float2(0.f, 0.f);
          float sx = 0.0f, q2 = 0.0f;
          if constexpr (LN) {
            // per column block (C0 values of the lane's row, converted once
            // into registers): the sum, then the squared deviations from the
            // block's mean; the unit's two blocks are then joined by the
            // pairwise formula M2 = M2_0 + M2_1 + (C0 / 2) (m_0 - m_1)^2
            // (equal counts).  (nv == 0: an empty unit, which the merge skips.)
            float sb[2] = {0.0f, 0.0f}, qb[2] = {0.0f, 0.0f};
#pragma unroll
            for (int h = 0; h < 2; ++h)
              if (h < nv) {
                float2 f[8 * PPC];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                  const uint4 v = chunk(h, c);
#pragma unroll
                  for (int i = 0; i < PPC; ++i) f[c * PPC + i] = chunk_pair<TIn>(v, i);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = f[i];
#pragma unroll
                for (int k = 4; k < 8 * PPC; ++k) a[k & 3] = add2(a[k & 3], f[k]);
                const float s = (a[0].x + a[0].y) + (a[1].x + a[1].y) + (a[2].x + a[2].y) + (a[3].x + a[3].y);
                const float2 bm = splat2(s * (1.0f / C0));
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float2 d = sub2(f[i], bm);
                  a[i] = mul2(d, d);
                }
#pragma unroll
                for (int k = 4; k < 8 * PPC; ++k) {
                  const float2 d = sub2(f[k], bm);
                  a[k & 3] = fma2(d, d, a[k & 3]);
                }
                sb[h] = s;
                qb[h] = (a[0].x + a[0].y) + (a[1].x + a[1].y) + (a[2].x + a[2].y) + (a[3].x + a[3].y);
              }
            sx = sb[0] + sb[1];
            const float dm = (sb[0] - sb[1]) * (1.0f / C0);
            q2 = nv == 2 ? (qb[0] + qb[1]) + (0.5f * C0) * dm * dm : qb[0];
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h)
              if (h < nv) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                  const uint4 v = chunk(h, c);
#pragma unroll
                  for (int i = 0; i < PPC; ++i) {
                    const float2 x = chunk_pair<TIn>(v, i);
                    a[(c * PPC + i) & 3] = fma2(x, x, a[(c * PPC + i) & 3]);
                  }
                }
              }
            sx = (a[0].x + a[0].y) + (a[1].x + a[1].y) + (a[2].x + a[2].y) + (a[3].x + a[3].y);
          }
          release(s, pos.use, EMPTY / 2);
          pw[u * kBoxRows + lane] = make_float2(sx, q2);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sdone[k & 1]));
        li += (uint32_t)nbox;
      }
    }
    if (ta < 0) continue;
    // ------------------------------------------------ quantization units
    const int tile = (int)blockIdx.x + ta * G;
    const int r0 = tile * kBoxRows;
    if constexpr (STATS)
      mbar_wait(smem_u32(&tready[ta & 1]), (uint32_t)(ta >> 1) & 1u, &g_err_mx, kErrReadyWait);
    // this thread's 8 rows' (mean, rsigma)
    const float2* st8 = tstat + (ta & 1) * kBoxRows + 8 * rg;
    // sub-tiles go two at a time (the same box: one wait, one release)
    for (int a2 = w; 2 * a2 < nua; a2 += kBoxWorkers) {
      const int b = (2 * a2) / SPB;
      pos.to(li + (uint32_t)b, Q);
      const uint32_t s = pos.slot;
      ticket_wait(smem_u32(&ticket[s]), pos.use, &g_err_mx, kErrFullWait);
      mbar_wait(smem_u32(&full[s]), pos.use & 1u, &g_err_mx, kErrFullWait);
#pragma unroll 1
      for (int a = 2 * a2; a < 2 * a2 + 2; ++a) {
        const int q = a - b * SPB;
        const int sub = a;  // 64-column sub-tile of the row
        if (64 * sub < H) {
          // (fp32 rows of 32 mod 64 columns end in half a sub-tile; bf16 rows
          // here are whole sub-tiles)
          const bool valid = ESZ == 2 || 64 * sub + 8 * cl < H;
          float2 g2[4], b2[4];
          {
            float4 gv[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
            float4 bv[2] = {gv[0], gv[0]};
            if (STATS && valid) {
              const float4* gp = reinterpret_cast<const float4*>(p.gamma + 64 * sub + 8 * cl);
              gv[0] = __ldg(gp);
              gv[1] = __ldg(gp + 1);
              if (p.zcg) {
#pragma unroll
                for (int jj = 0; jj < 2; ++jj)
                  gv[jj] = make_float4(1.0f + gv[jj].x, 1.0f + gv[jj].y, 1.0f + gv[jj].z, 1.0f + gv[jj].w);
              }
              if (LN && p.beta) {
                const float4* bp = reinterpret_cast<const float4*>(p.beta + 64 * sub + 8 * cl);
                bv[0] = __ldg(bp);
                bv[1] = __ldg(bp + 1);
              }
            }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              g2[2 * jj] = make_float2(gv[jj].x, gv[jj].y);
              g2[2 * jj + 1] = make_float2(gv[jj].z, gv[jj].w);
              b2[2 * jj] = make_float2(bv[jj].x, bv[jj].y);
              b2[2 * jj + 1] = make_float2(bv[jj].z, bv[jj].w);
            }
          }
          // this thread's 8 columns in the box: bf16, chunk cl of column block
          // q; fp32, chunks 2 (cl & 3), +1 of column block 2q + (cl >> 2)
          // row 8 rg + jr of the thread's column block starts at cbb + jr * 128;
          // its chunk k sits at chunk k ^ jr (the 128-byte swizzle)
          const uint32_t cbb = ring_u32 + s * kBoxBytes +
                               (uint32_t)(ESZ == 2 ? q : 2 * q + (cl >> 2)) * 4096 + (uint32_t)rg * 1024;
          const uint32_t ck = ESZ == 2 ? (uint32_t)cl << 4 : (uint32_t)(2 * (cl & 3)) << 4;
          float2 y[8][4];
#pragma unroll
          for (int jr = 0; jr < 8; ++jr) {
            const uint32_t rowa = cbb + jr * 128;
            float2 x2[4];
            if constexpr (ESZ == 2) {
              const uint4 v = lds128(rowa + (ck ^ (jr << 4)));
#pragma unroll
              for (int i = 0; i < 4; ++i) x2[i] = chunk_pair<TIn>(v, i);
            } else {
              const uint4 v0 = lds128(rowa + (ck ^ (jr << 4)));
              const uint4 v1 = lds128(rowa + ((ck + 16) ^ (jr << 4)));
              x2[0] = chunk_pair<TIn>(v0, 0);
              x2[1] = chunk_pair<TIn>(v0, 1);
              x2[2] = chunk_pair<TIn>(v1, 0);
              x2[3] = chunk_pair<TIn>(v1, 1);
            }
            const float2 ms = STATS ? st8[jr] : make_float2(0.f, 1.f);
            const float2 rs2 = splat2(ms.y);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if constexpr (LN)
                y[jr][i] = fma2(fma2(x2[i], rs2, splat2(ms.x)), g2[i], b2[i]);
              else if constexpr (NK == kRms)
                y[jr][i] = mul2(mul2(x2[i], rs2), g2[i]);
              else
                y[jr][i] = x2[i];
              if (ESZ == 4 && !valid) y[jr][i] = make_float2(0.f, 0.f);
            }
          }
          // one sweep over |y|: row maxima (8 values each) and column maxima
          // (8 values each), two rows at a time
          float rmax[8], cmax[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            rmax[i] = 0.f;
            cmax[i] = 0.f;
          }
#pragma unroll
          for (int jr = 0; jr < 8; jr += 2) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float a0 = fabsf(y[jr][i].x), b0 = fabsf(y[jr][i].y);
              const float a1 = fabsf(y[jr + 1][i].x), b1 = fabsf(y[jr + 1][i].y);
              rmax[jr] = max3n(rmax[jr], a0, b0);
              rmax[jr + 1] = max3n(rmax[jr + 1], a1, b1);
              cmax[2 * i] = max3n(cmax[2 * i], a0, a1);
              cmax[2 * i + 1] = max3n(cmax[2 * i + 1], b0, b1);
            }
          }
          // the row blocks' and column blocks' maxima, scales and inverse
          // scales, the two independent shuffle chains side by side
          float rm0, rm1, cm0, cm1;
          block_max_scatter(rmax, cc >> 1, cc & 1, 2, 1, rm0, rm1);
          block_max_scatter(cmax, rg >> 1, rg & 1, kColS1, kColS0, cm0, cm1);
          const uint32_t rcode0 = e8m0_code(rm0), rcode1 = e8m0_code(rm1);
          const uint32_t ccode0 = e8m0_code(cm0), ccode1 = e8m0_code(cm1);
          float inv[8], cinv[8];
          gather8(e8m0_inv_scale(rcode0), e8m0_inv_scale(rcode1), cc >> 1, cc & 1, 2, 1, inv);
          gather8(e8m0_inv_scale(ccode0), e8m0_inv_scale(ccode1), rg >> 1, rg & 1, kColS1, kColS0,
                  cinv);
          if (rowwise && valid) {
            uint8_t* dp = p.data + ((size_t)(r0 + 8 * rg) * H + 64 * sub + 8 * cl);
#pragma unroll
            for (int jr = 0; jr < 8; ++jr) {
              const float2 iv = splat2(inv[jr]);
              float2 v[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) v[i] = mul2(y[jr][i], iv);
              *reinterpret_cast<uint2*>(dp) = make_uint2(pack_e4m3x4(v[0].x, v[0].y, v[1].x, v[1].y),
                                                         pack_e4m3x4(v[2].x, v[2].y, v[3].x, v[3].y));
              dp += H;
            }
            uint8_t* sp = p.row_scales + ((size_t)(r0 + 8 * rg + cc) * hs + 2 * sub + hb);
            sp[0] = (uint8_t)rcode0;
            sp[4 * (size_t)hs] = (uint8_t)rcode1;
          }
          if (colwise && valid) {
            uint8_t* cp = p.col_data + ((size_t)(64 * sub + 8 * cl) * N + r0 + 8 * rg);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 ci = make_float2(cinv[2 * i], cinv[2 * i + 1]);
              float2 qv[8];
#pragma unroll
              for (int jr = 0; jr < 8; ++jr) qv[jr] = mul2(y[jr][i], ci);
              *reinterpret_cast<uint2*>(cp) =
                  make_uint2(pack_e4m3x4(qv[0].x, qv[1].x, qv[2].x, qv[3].x),
                             pack_e4m3x4(qv[4].x, qv[5].x, qv[6].x, qv[7].x));
              *reinterpret_cast<uint2*>(cp + N) =
                  make_uint2(pack_e4m3x4(qv[0].y, qv[1].y, qv[2].y, qv[3].y),
                             pack_e4m3x4(qv[4].y, qv[5].y, qv[6].y, qv[7].y));
              cp += 2 * (size_t)N;
            }
            uint8_t* csp = p.col_scales + ((size_t)(64 * sub + 8 * cl + rg) * ns + tile);
            csp[0] = (uint8_t)ccode0;
            csp[4 * (size_t)ns] = (uint8_t)ccode1;
          }
        }
      }
      release(s, pos.use, 2 * (EMPTY / SPB));
    }
    li += (uint32_t)nbox;
  }
  // every copy issued has been waited on by its readers; after a wait that
  // gave up (an error is recorded) one may still be in flight: wait for each
  // slot's last load before the CTA leaves
  __syncthreads();
  if (threadIdx.x == 0)
    for (uint32_t sl = 0; sl < Q && sl < nload; ++sl) {
      const uint32_t last = sl + Q * ((nload - 1 - sl) / Q);
      mbar_wait(smem_u32(&full[sl]), (last / Q) & 1u, &g_err_mx, kErrDrainWait);
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

template <typename TIn, int NK>
rn_status launch_box_t(const MxParams& p, const Launch& l, cudaStream_t s) {
  auto k = rn_mx_box_kernel<TIn, NK>;
  constexpr int C0 = 128 / (int)sizeof(TIn);
  if (l.threads != kBoxThreads || p.H % C0 != 0 || p.N % kBoxRows != 0 || p.Q < 2)
    return RN_ERR_UNSUPPORTED;
  EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr) return RN_ERR_CUDA;
  // x [N][H] seen as 3-D: the 128-byte column block (C0 elements,
  // contiguous), rows (stride H elements), column blocks (stride C0
  // elements); a box is 32 rows x kBoxCb column blocks, 128-byte swizzled.
  // Column blocks past H / C0 (the last box of a row) read as zeros.
  CUtensorMap tm;
  const cuuint64_t dims[3] = {(cuuint64_t)C0, (cuuint64_t)p.N, (cuuint64_t)(p.H / C0)};
  const cuuint64_t strides[2] = {(cuuint64_t)p.H * sizeof(TIn), (cuuint64_t)128};
  const cuuint32_t box[3] = {(cuuint32_t)C0, (cuuint32_t)kBoxRows, (cuuint32_t)kBoxCb};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      sizeof(TIn) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (enc(&tm, dt, 3, const_cast<void*>(p.x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
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

rn_status launch_mx_box(int nk, bool bf16, const MxParams& p, const Launch& l, cudaStream_t s) {
  if (nk == kIdentity) return bf16 ? RN_ERR_UNSUPPORTED : launch_box_t<float, kIdentity>(p, l, s);
  if (bf16) return nk == kLn ? launch_box_t<uint16_t, kLn>(p, l, s) : launch_box_t<uint16_t, kRms>(p, l, s);
  return nk == kLn ? launch_box_t<float, kLn>(p, l, s) : launch_box_t<float, kRms>(p, l, s);
}

rn_status read_clear_error_mx(unsigned* code) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_mx, sizeof(v)) != cudaSuccess) return RN_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_err_mx, &zero, sizeof(zero)) != cudaSuccess) return RN_ERR_CUDA;
  *code = v;
  return RN_OK;
}

}  // namespace rn
