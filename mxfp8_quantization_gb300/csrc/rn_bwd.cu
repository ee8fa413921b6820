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
// Kernel 1 (persistent, warp-specialized like the forward, no CTA-wide
// barrier on the row path): the producer lane streams the x row and the dz
// row of each row into one shared-memory slot with two bulk copies, and its
// saved mu / rsigma with 4-byte cp.async, all on the slot's "full" barrier;
//   stats warps  take rows in turn and form the two row means mean(dy) and
//                mean(dy * xhat) (g from a shared-memory copy laid out for
//                conflict-free reads, which the stats and apply warps fill
//                while the producer streams the first rows), published on
//                the slot's "ready" barrier;
//   apply warps  own fixed 16-byte column chunks: dx for every row in order,
//                plus running per-column sums of dz * xhat and dz in
//                registers; they release the slot ("empty").
// Rows are grouped in fixed chunks of chunk_rows rows; at the end of a chunk
// its column sums are written to the workspace as one fp32 partial row.  The
// chunk size depends on N (and, for the one-CTA-per-SM shape, on the
// device's SM count), never on the grid or sm_margin, and each partial is
// summed in row order, so the partials do not depend on the grid.
// Kernel 2 adds the partials of each column in a fixed order that depends
// on the chunk count and H only.  Arithmetic is on element pairs (f32x2), with
// bf16 inputs entering through the mixed-precision forms.
#include <cuda_runtime.h>

#include "rn_device.cuh"
#include "rn_internal.h"

namespace rn {
namespace {

__device__ unsigned g_err_bwd;

// compact shape: at most 8 apply + 3 stats warps + the producer, two CTAs
// per SM (24 warps an SM leave 80 registers a thread: a fourth stats warp
// cut that to 72 and made the apply warps spill); wide shape: one CTA per
// SM, compiled twice: for at most 512 threads (128 registers a thread) and
// for at most 576 (96).  (Compiled for 800 threads, i.e. 72 registers, the
// bf16 LayerNorm kernel spilled: 3000 x 5120 took 33.2 us against 28.9 us
// with the 512-thread build.)
constexpr int kMaxThreads = 384;
constexpr int kMaxThreadsWide = kBwdWideThreads;
constexpr int kMaxThreadsWide512 = kBwdWideThreads512;
// compact shape with 4 chunks a thread: 4 apply + 3 stats warps + the
// producer (256 threads, 128 registers: the 4 chunks' gamma and dgamma /
// dbeta sums stay in registers)
constexpr int kMaxThreadsNg4 = 256;
// rows the producer issues before waiting for the first one to land
constexpr uint32_t kStartRows = 2;

// launch shapes of the stats-warp kernel
enum BwdShapeKind : int { kCompact = 0, kWide512 = 1, kWide = 2 };

template <int SK, int NG>
constexpr int bwd_max_threads() {
  return SK == kWide ? kMaxThreadsWide
                     : (SK == kWide512 ? kMaxThreadsWide512 : (NG >= 4 ? kMaxThreadsNg4 : kMaxThreads));
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <typename TIn>
__device__ __forceinline__ void store_dx(void* base, size_t elem, const float2* d);

template <>
__device__ __forceinline__ void store_dx<uint16_t>(void* base, size_t elem, const float2* d) {
  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + elem) =
      make_uint4(pack_bf16x2(d[0].x, d[0].y), pack_bf16x2(d[1].x, d[1].y),
                 pack_bf16x2(d[2].x, d[2].y), pack_bf16x2(d[3].x, d[3].y));
}

template <>
__device__ __forceinline__ void store_dx<float>(void* base, size_t elem, const float2* d) {
  *reinterpret_cast<float4*>(static_cast<float*>(base) + elem) = make_float4(d[0].x, d[0].y, d[1].x, d[1].y);
}

template <typename TIn, int NG, bool LN, int SK>
__global__ void __launch_bounds__(bwd_max_threads<SK, NG>(), SK == kCompact ? 2 : 1)
    rn_bwd_kernel(const BwdParams p) {
  constexpr int VEC = 16 / (int)sizeof(TIn);
  using V = Vec<TIn, VEC>;
  constexpr int PAIRS = V::PAIRS;
  extern __shared__ __align__(128) unsigned char smem[];
  // the column reduction (launched next, as a programmatic dependent) may be
  // placed on SMs as soon as this grid's CTAs retire
  if (threadIdx.x == 0) pdl_launch_dependents();

  const int A = p.apply_warps;          // warps 0 .. A-1
  const int S = p.stats_warps;          // warps A .. A+S-1; producer: A+S
  const int TH = A * 32;
  const int H = p.H;
  const int nchunks = H / VEC;
  const uint32_t row_bytes = (uint32_t)H * sizeof(TIn);
  const uint32_t slot_bytes = 2 * row_bytes;  // x row, then dz row
  const uint32_t Q = (uint32_t)p.Q;

  unsigned char* ring = smem;
  // g as [VEC/4][nchunks] float4: part j of chunk c at gsv[j * nchunks + c],
  // so that 32 lanes reading 32 consecutive chunks touch consecutive 16 bytes
  float4* gsv = reinterpret_cast<float4*>(smem + (size_t)Q * slot_bytes);
  float4* rstat = gsv + (size_t)(VEC / 4) * nchunks;   // [Q] (mu, rsigma, c1, c2)
  float2* meta = reinterpret_cast<float2*>(rstat + Q);  // [Q] (mu, rsigma) as loaded
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + Q);
  uint64_t* ready = full + Q;
  uint64_t* empty = ready + Q;

  for (uint32_t i = threadIdx.x; i < Q; i += blockDim.x) {
    mbar_init(smem_u32(&full[i]), 2);  // bulk copies + the mu/rsigma cp.async
    mbar_init(smem_u32(&ready[i]), 1);
    mbar_init(smem_u32(&empty[i]), A);
    fence_barrier_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  // g is staged by the stats and apply warps while the producer already
  // streams the first rows; a thread issues the loads of up to 4 items
  // before its first store (one trip to memory, not one per item).  Staged
  // behind a CTA barrier ahead of the producer, g held the first row back by
  // ~2 us.
  if (warp < A + S) {
    const int NT = (A + S) * 32, items = H / 4;
    const bool al = (reinterpret_cast<uintptr_t>(p.gamma) & 15) == 0;
    for (int j0 = threadIdx.x; j0 < items; j0 += 4 * NT) {
      float4 g4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = j0 + k * NT;
        if (j < items)
          g4[k] = al ? __ldg(reinterpret_cast<const float4*>(p.gamma) + j)
                     : make_float4(p.gamma[4 * j], p.gamma[4 * j + 1], p.gamma[4 * j + 2],
                                   p.gamma[4 * j + 3]);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int j = j0 + k * NT;
        if (j < items) {
          float4 g = g4[k];
          if (p.zcg) g = make_float4(1.0f + g.x, 1.0f + g.y, 1.0f + g.z, 1.0f + g.w);
          gsv[(j % (VEC / 4)) * nchunks + j / (VEC / 4)] = g;
        }
      }
    }
    named_sync(1, NT);
  }
  const int lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int R = p.chunk_rows;

  if (warp == A + S) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const unsigned char* xb = static_cast<const unsigned char*>(p.x);
      const unsigned char* db = static_cast<const unsigned char*>(p.dz);
      const uint64_t stream_pol = l2_evict_first();
      RingPos pos{0u, 0u};
      uint32_t issued = 0;
      for (int c = blockIdx.x; c < p.n_chunks; c += G) {
        const int r1 = min((c + 1) * R, p.N);
        for (int r = c * R; r < r1; ++r, ++issued) {
          const uint32_t s = pos.slot;
          // the first kStartRows rows go out alone, the rest of the ring once
          // row 0 is in (a start-up burst of whole rings from every SM lands
          // all at once, late)
          if (issued == kStartRows) mbar_wait(smem_u32(&full[0]), 0u, &g_err_bwd, kErrFullWait);
          if (issued >= Q) mbar_wait(smem_u32(&empty[s]), pos.phase ^ 1u, &g_err_bwd, kErrEmptyWait);
          const uint32_t bar = smem_u32(&full[s]);
          if (LN) cp_async4(smem_u32(&meta[s].x), p.mu + r);
          cp_async4(smem_u32(&meta[s].y), p.rsigma + r);
          cp_async_arrive(bar);
          mbar_arrive_expect_tx(bar, slot_bytes);
          const uint32_t dst = smem_u32(ring + (size_t)s * slot_bytes);
          // x and dz are read once here: let them leave L2 first, so that the
          // dgamma/dbeta partials stay there for the column reduction
          bulk_g2s_hint(dst, xb + (size_t)r * row_bytes, row_bytes, bar, stream_pol);
          bulk_g2s_hint(dst + row_bytes, db + (size_t)r * row_bytes, row_bytes, bar, stream_pol);
          pos.advance(1, Q);
        }
      }
      const uint32_t first = issued > Q ? issued - Q : 0;
      for (uint32_t k = first; k < issued; ++k)
        mbar_wait(smem_u32(&full[k % Q]), (k / Q) & 1u, &g_err_bwd, kErrDrainWait);
    }
    return;
  }

  if (warp >= A) {
    // --------------------------------------------------------- stats warps
    // stats warp j takes rows j, j + S, ... of the CTA's sequence: the two
    // row sums of dy = dz * g and dy * (x - mu) (RMSNorm: dy * x), giving
    // c1 = mean(dy) and c2 = mean(dy * xhat) = rsigma * mean(dy * (x - mu))
    const int j = warp - A;
    const float inv_h = 1.0f / (float)H;
    // stats warp j takes rows j, j + S, j + 2S, ... of the CTA's sequence:
    // row `within` of chunk c (c = blockIdx.x, blockIdx.x + grid, ...);
    // only the last chunk of all may be short, and it is the CTA's last
    int c = blockIdx.x, within = j;
    while (within >= R) {
      within -= R;
      c += G;
    }
    RingPos pos{0u, 0u};
    pos.advance((uint32_t)j, Q);
    for (int q = j; c < p.n_chunks; q += S) {
      const int r = c * R + within;
      if (r >= p.N) break;
      const uint32_t s = pos.slot;
      // not paced by the apply warps: wait for the previous use of the
      // slot to be released first, so that the parity wait below cannot
      // match a phase one lap old (alias-free as stats warps < slots)
      if (q >= (int)Q) mbar_wait(smem_u32(&empty[s]), pos.phase ^ 1u, &g_err_bwd, kErrStatsWait);
      mbar_wait(smem_u32(&full[s]), pos.phase, &g_err_bwd, kErrStatsWait);
      const unsigned char* xr = ring + (size_t)s * slot_bytes;
      const unsigned char* dr = xr + row_bytes;
      const float2 m = meta[s];
      const float mu = LN ? m.x : 0.f;
      float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
      for (int cc = lane; cc < nchunks; cc += 32) {
        const typename V::Raw xw = V::load(xr, cc);
        const typename V::Raw dw = V::load(dr, cc);
        float2 gp[PAIRS];
#pragma unroll
        for (int i = 0; i < PAIRS; i += 2) {
          const float4 g4 = gsv[(i / 2) * nchunks + cc];
          gp[i] = make_float2(g4.x, g4.y);
          gp[i + 1] = make_float2(g4.z, g4.w);
        }
#pragma unroll
        for (int i = 0; i < PAIRS; ++i) {
          const float2 d = LN ? V::sub(xw, i, mu) : V::f32(xw, i);
          const float2 dy = mul2(V::f32(dw, i), gp[i]);
          s1 = add2(s1, dy);
          s2 = fma2(dy, d, s2);
        }
      }
      const float a1 = warp_sum(s1.x + s1.y);
      const float a2 = warp_sum(s2.x + s2.y);
      if (lane == 0) {
        rstat[s] = make_float4(mu, m.y, LN ? a1 * inv_h : 0.f, m.y * (a2 * inv_h));
        mbar_arrive(smem_u32(&ready[s]));
      }
      pos.advance((uint32_t)S, Q);
      within += S;
      while (within >= R) {
        within -= R;
        c += G;
      }
    }
    return;
  }

  // ---------------------------------------------------------- apply warps
  const int t = threadIdx.x;
  float2 g2[NG][PAIRS];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int v = g * TH + t;
#pragma unroll
    for (int i = 0; i < PAIRS; i += 2) {
      const float4 g4 = (v < nchunks) ? gsv[(i / 2) * nchunks + v] : make_float4(0.f, 0.f, 0.f, 0.f);
      g2[g][i] = make_float2(g4.x, g4.y);
      g2[g][i + 1] = make_float2(g4.z, g4.w);
    }
  }
  const int nacc = LN ? 2 : 1;
  const uint64_t keep_pol = l2_evict_last();

  RingPos pos{0u, 0u};
  for (int c = blockIdx.x; c < p.n_chunks; c += G) {
    float2 adg[NG][PAIRS], adb[NG][PAIRS];
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int i = 0; i < PAIRS; ++i) {
        adg[g][i] = make_float2(0.f, 0.f);
        adb[g][i] = make_float2(0.f, 0.f);
      }
    const int r1 = min((c + 1) * R, p.N);
    for (int r = c * R; r < r1; ++r) {
      const uint32_t s = pos.slot;
      // "ready" is published after the stats warp saw the row land
      mbar_wait(smem_u32(&ready[s]), pos.phase, &g_err_bwd, kErrReadyWait);
      const float4 m = rstat[s];
      const unsigned char* xr = ring + (size_t)s * slot_bytes;
      const unsigned char* dr = xr + row_bytes;
      const size_t rowe = (size_t)r * H;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const int v = g * TH + t;
        if (v < nchunks) {
          const typename V::Raw xw = V::load(xr, v);
          const typename V::Raw dw = V::load(dr, v);
          float2 dx[PAIRS];
#pragma unroll
          for (int i = 0; i < PAIRS; ++i) {
            const float2 xh = mul2(LN ? V::sub(xw, i, m.x) : V::f32(xw, i), splat2(m.y));
            const float2 dzf = V::f32(dw, i);
            const float2 dy = mul2(dzf, g2[g][i]);
            dx[i] = mul2(sub2(dy, fma2(xh, splat2(m.w), splat2(m.z))), splat2(m.y));
            adg[g][i] = fma2(dzf, xh, adg[g][i]);
            if (LN) adb[g][i] = add2(adb[g][i], dzf);
          }
          store_dx<TIn>(p.dx, rowe + (size_t)v * VEC, dx);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
      pos.advance(1, Q);
    }
    // chunk finished: write its partial column sums (kept in L2 for the
    // column reduction)
    float* prow = p.part + (size_t)c * nacc * H;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const int v = g * TH + t;
      if (v < nchunks) {
#pragma unroll
        for (int jj = 0; jj < PAIRS / 2; ++jj) {
          st_hint_f4(prow + (size_t)v * VEC + 4 * jj,
                     make_float4(adg[g][2 * jj].x, adg[g][2 * jj].y, adg[g][2 * jj + 1].x,
                                 adg[g][2 * jj + 1].y),
                     keep_pol);
          if (LN)
            st_hint_f4(prow + H + (size_t)v * VEC + 4 * jj,
                       make_float4(adb[g][2 * jj].x, adb[g][2 * jj].y, adb[g][2 * jj + 1].x,
                                   adb[g][2 * jj + 1].y),
                       keep_pol);
        }
      }
    }
  }
}

// ------------------------------------------------------------ fused kernel
// fp32 rows of up to 16 warps x 32 threads x 16 elements (H <= 8192): no
// stats warps and no producer warp.  Every thread owns NG fixed
// 16-byte chunks (16 elements of each row; gamma and the dgamma / dbeta sums
// in registers).  Per row it reads its chunks out of the ring slot, forms
// d = x - mu (RMSNorm: x), dz and dy = dz * g in registers and its share of
// the two row sums sum(dy) and sum(dy * d); the warps exchange their sums
// through shared memory around one CTA barrier and add them in a fixed order
// (a butterfly over the warp sums, identical on every thread); then
//   dx = rsigma * dy + P * d + B,  P = -rsigma^2 * c2,  B = -rsigma * c1,
// with c1 = mean(dy) and c2 = mean(dy * xhat) = rsigma * mean(dy * d), which
// is rsigma * (dy - c1 - xhat * c2) regrouped.
// The barrier also frees the row's slot (every thread has read it), so lane 0
// of warp 0 refills it right there with the row Q places ahead (bulk copies
// of x and dz, cp.async of mu / rsigma, on the slot's "full" mbarrier); the
// first rows go out one by one at the start so that row 0 lands early.
constexpr int kFusedCompact = 256;  // <= 8 warps, 2+ CTAs per SM (128 registers)
constexpr int kFusedBig = 512;      // <= 16 warps, 1 CTA per SM (128 registers)

// the rows of this CTA, chunk by chunk (chunks blockIdx.x + k * gridDim.x)
struct ChunkRows {
  int c, r, r1;
  __device__ __forceinline__ bool next(const BwdParams& p) {
    if (++r < r1) return true;
    c = (c < 0) ? (int)blockIdx.x : c + (int)gridDim.x;
    if (c >= p.n_chunks) return false;
    r = c * p.chunk_rows;
    r1 = min(r + p.chunk_rows, p.N);
    return true;
  }
};

template <bool LN>
__device__ __forceinline__ void issue_row(const BwdParams& p, unsigned char* ring, float2* meta,
                                          uint64_t* full, uint32_t s, int r, uint32_t row_bytes,
                                          uint64_t pol) {
  const uint32_t bar = smem_u32(&full[s]);
  if (LN) cp_async4(smem_u32(&meta[s].x), p.mu + r);
  cp_async4(smem_u32(&meta[s].y), p.rsigma + r);
  cp_async_arrive(bar);
  mbar_arrive_expect_tx(bar, 2 * row_bytes);
  const uint32_t dst = smem_u32(ring + (size_t)s * 2 * row_bytes);
  bulk_g2s_hint(dst, static_cast<const unsigned char*>(p.x) + (size_t)r * row_bytes, row_bytes,
                bar, pol);
  bulk_g2s_hint(dst + row_bytes, static_cast<const unsigned char*>(p.dz) + (size_t)r * row_bytes,
                row_bytes, bar, pol);
}

template <typename TIn, int NG, bool LN, bool BIG>
__global__ void __launch_bounds__(BIG ? kFusedBig : kFusedCompact, BIG ? 1 : 2)
    rn_bwd_fused_kernel(const BwdParams p) {
  constexpr int VEC = 16 / (int)sizeof(TIn);
  using V = Vec<TIn, VEC>;
  constexpr int PAIRS = V::PAIRS;
  extern __shared__ __align__(128) unsigned char smem[];
  if (threadIdx.x == 0) pdl_launch_dependents();

  const int A = p.apply_warps;  // warps of the CTA (<= 16)
  const int TH = A * 32;
  const int H = p.H;
  const int nchunks = H / VEC;
  const uint32_t row_bytes = (uint32_t)H * sizeof(TIn);
  const uint32_t slot_bytes = 2 * row_bytes;  // x row, then dz row
  const uint32_t Q = (uint32_t)p.Q;

  unsigned char* ring = smem;
  float2* meta = reinterpret_cast<float2*>(smem + (size_t)Q * slot_bytes);  // [Q] (mu, rsigma)
  float2* red = meta + Q;                                                   // [2][16] warp sums
  uint64_t* full = reinterpret_cast<uint64_t*>(red + 32);

  for (uint32_t i = threadIdx.x; i < Q; i += blockDim.x) {
    mbar_init(smem_u32(&full[i]), 2);  // bulk copies + the mu/rsigma cp.async
    fence_barrier_init();
  }
  __syncthreads();

  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int lane = t & 31;
  const bool issuer = (t == 0);
  const uint64_t stream_pol = l2_evict_first();

  // issue cursor (thread 0): rows handed to the copy engine so far
  ChunkRows iw{-1, 0, 0};
  uint32_t issued = 0;
  bool more = true;
  RingPos ipos{0u, 0u};
  if (issuer) {
    while (issued < (uint32_t)kStartRows && issued < Q && (more = iw.next(p))) {
      issue_row<LN>(p, ring, meta, full, ipos.slot, iw.r, row_bytes, stream_pol);
      ipos.advance(1, Q);
      ++issued;
    }
  }

  float2 g2[NG][PAIRS];
#pragma unroll
  for (int g = 0; g < NG; ++g) {
    const int v = g * TH + t;
#pragma unroll
    for (int i = 0; i < PAIRS; ++i) {
      g2[g][i] = make_float2(0.f, 0.f);
      if (v < nchunks) {
        const int e = v * VEC + 2 * i;
        const float ga = p.gamma[e], gb = p.gamma[e + 1];
        g2[g][i] = p.zcg ? make_float2(1.0f + ga, 1.0f + gb) : make_float2(ga, gb);
      }
    }
  }
  const float inv_h = 1.0f / (float)H;
  const int nacc = LN ? 2 : 1;
  const uint64_t keep_pol = l2_evict_last();

  RingPos pos{0u, 0u};
  uint32_t q = 0;
  for (int c = blockIdx.x; c < p.n_chunks; c += (int)gridDim.x) {
    float2 adg[NG][PAIRS], adb[NG][PAIRS];
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int i = 0; i < PAIRS; ++i) {
        adg[g][i] = make_float2(0.f, 0.f);
        adb[g][i] = make_float2(0.f, 0.f);
      }
    const int r1 = min((c + 1) * p.chunk_rows, p.N);
    for (int r = c * p.chunk_rows; r < r1; ++r, ++q) {
      const uint32_t s = pos.slot;
      // every thread read the slot's previous row before the barrier that
      // let it be refilled, so this parity wait cannot match an older phase
      mbar_wait(smem_u32(&full[s]), pos.phase, &g_err_bwd, kErrFullWait);
      const unsigned char* xr = ring + (size_t)s * slot_bytes;
      const unsigned char* dr = xr + row_bytes;
      const float2 m = meta[s];
      const float mu = LN ? m.x : 0.0f;
      const float rs = m.y;

      // this thread's share of sum(dy) and sum(dy * d)
      float2 d[NG][PAIRS], dzf[NG][PAIRS];
      float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const int v = g * TH + t;
        const bool ok = v < nchunks;
        typename V::Raw xw, dw;
        if (ok) {
          xw = V::load(xr, v);
          dw = V::load(dr, v);
        }
#pragma unroll
        for (int i = 0; i < PAIRS; ++i) {
          d[g][i] = make_float2(0.f, 0.f);
          dzf[g][i] = make_float2(0.f, 0.f);
          if (ok) {
            d[g][i] = LN ? V::sub(xw, i, mu) : V::f32(xw, i);
            dzf[g][i] = V::f32(dw, i);
            const float2 dy = mul2(dzf[g][i], g2[g][i]);
            s1 = add2(s1, dy);
            s2 = fma2(dy, d[g][i], s2);
          }
        }
      }
      const float a1 = LN ? warp_sum(s1.x + s1.y) : 0.0f;
      const float a2 = warp_sum(s2.x + s2.y);
      float2* rb = red + (q & 1u) * 16;
      if (lane == 0) rb[warp] = make_float2(a1, a2);
      // rb[q & 1] is rewritten two rows later, after every thread has passed
      // the next row's barrier (and so has read it)
      __syncthreads();
      pos.advance(1, Q);
      if (issuer) {
        // slot s is free: refill it (and, at the start, the rest of the ring)
        fence_proxy_async();
        const uint32_t target = q + Q;  // rows issued after this: all up to q + Q
        while (more && issued <= target && (more = iw.next(p))) {
          issue_row<LN>(p, ring, meta, full, ipos.slot, iw.r, row_bytes, stream_pol);
          ipos.advance(1, Q);
          ++issued;
        }
      }
      float2 tot = (lane < A) ? rb[lane] : make_float2(0.f, 0.f);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1)
        tot = add2(tot, make_float2(__shfl_xor_sync(0xFFFFFFFFu, tot.x, o),
                                    __shfl_xor_sync(0xFFFFFFFFu, tot.y, o)));
      const float c1 = tot.x * inv_h;         // mean(dy)
      const float c2 = rs * (tot.y * inv_h);  // mean(dy * xhat)
      const float2 P2 = splat2(-(rs * rs) * c2);
      const float2 B2 = splat2(LN ? -rs * c1 : 0.0f);
      const float2 rs2 = splat2(rs);
      const size_t rowe = (size_t)r * H;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const int v = g * TH + t;
        if (v < nchunks) {
          float2 dx[PAIRS];
#pragma unroll
          for (int i = 0; i < PAIRS; ++i) {
            const float2 dy = mul2(dzf[g][i], g2[g][i]);
            dx[i] = fma2(dy, rs2, fma2(d[g][i], P2, B2));
            adg[g][i] = fma2(dzf[g][i], mul2(d[g][i], rs2), adg[g][i]);
            if (LN) adb[g][i] = add2(adb[g][i], dzf[g][i]);
          }
          store_dx<TIn>(p.dx, rowe + (size_t)v * VEC, dx);
        }
      }
    }
    // chunk finished: write its partial column sums (kept in L2 for the
    // column reduction)
    float* prow = p.part + (size_t)c * nacc * H;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const int v = g * TH + t;
      if (v < nchunks) {
#pragma unroll
        for (int jj = 0; jj < PAIRS / 2; ++jj) {
          st_hint_f4(prow + (size_t)v * VEC + 4 * jj,
                     make_float4(adg[g][2 * jj].x, adg[g][2 * jj].y, adg[g][2 * jj + 1].x,
                                 adg[g][2 * jj + 1].y),
                     keep_pol);
          if (LN)
            st_hint_f4(prow + H + (size_t)v * VEC + 4 * jj,
                       make_float4(adb[g][2 * jj].x, adb[g][2 * jj].y, adb[g][2 * jj + 1].x,
                                   adb[g][2 * jj + 1].y),
                       keep_pol);
        }
      }
    }
  }
}

// dgamma[j] (a = 0) / dbeta[j] (a = 1) = sum over chunks of part[c][a][j].
// Block: 32 warps x 32 lanes; lane owns 2 adjacent columns of a 64-column
// slice; warp w sums chunks w, w+32, w+64, ... into eight interleaved
// accumulators (chunk index / 32 mod 8, eight loads in flight), adds them
// pairwise in a fixed tree, then thread j of the first 64 adds the 32 warp
// sums in warp order.  The order depends on the chunk count only.
__global__ void __launch_bounds__(1024) rn_colreduce_kernel(const ColReduceParams p) {
  __shared__ float2 red[32][33];
  pdl_wait();  // the partials come from the backward kernel
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a = blockIdx.y;
  const int col = blockIdx.x * 64 + lane * 2;
  float2 acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = make_float2(0.f, 0.f);
  if (col < p.H) {
    const float* base = p.part + (size_t)a * p.H + col;
    const size_t stride = (size_t)p.nacc * p.H;
    // the partials are read once here; the bwd kernel kept them in L2
    const uint64_t pol = l2_evict_first();
    int c = warp;
    for (; c + 224 < p.n_chunks; c += 256) {
      float2 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = ld_hint_f2(base + (size_t)(c + 32 * i) * stride, pol);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = add2(acc[i], v[i]);
    }
    for (int i = 0; c < p.n_chunks; c += 32, ++i)
      acc[i] = add2(acc[i], ld_hint_f2(base + (size_t)c * stride, pol));
  }
  const float2 s = add2(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])),
                        add2(add2(acc[4], acc[5]), add2(acc[6], acc[7])));
  red[warp][lane] = s;
  __syncthreads();
  if (threadIdx.x < 64) {
    const int l = threadIdx.x >> 1, e = threadIdx.x & 1;
    const int j = blockIdx.x * 64 + threadIdx.x;
    float r = 0.f;
    for (int w = 0; w < 32; ++w) {
      const float2 v = red[w][l];
      r += e ? v.y : v.x;
    }
    if (j < p.H) (a == 0 ? p.dgamma : p.dbeta)[j] = r;
  }
}

// The same sums with 32-column blocks of 16 warps (lane = one column; warp
// w sums chunks w, w+16, ... into the eight accumulators, the tree, then the
// 16 warp sums in warp order), taken when the 64-column blocks would number
// more than kRedOneWave (slices x accumulators; one block an SM of a GB300
// holds): the smaller blocks then spread over every SM in one wave (3000 x
// 5120 LayerNorm 27.0 against 28.8 us, 2000 x 12288 RMSNorm 41.2 against
// 43.0 us), while up to that count the 64-column ones are 1-4 us faster
// (8192 x 4096).  A column's order depends on the warp count and the chunk
// count, so on the problem (and the device's SM count), never on sm_margin.
constexpr int kRedOneWave = 152;

__device__ __forceinline__ float ld_hint_f1(const float* p, uint64_t pol) {
  float v;
  asm volatile("ld.global.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(pol));
  return v;
}

__global__ void __launch_bounds__(16 * 32) rn_colreduce_narrow_kernel(const ColReduceParams p) {
  constexpr int NW = 16;
  __shared__ float red[NW][33];
  pdl_wait();  // the partials come from the backward kernel
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a = blockIdx.y;
  const int col = blockIdx.x * 32 + lane;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  if (col < p.H) {
    const float* base = p.part + (size_t)a * p.H + col;
    const size_t stride = (size_t)p.nacc * p.H;
    const uint64_t pol = l2_evict_first();  // the partials are read once
    int c = warp;
    for (; c + 7 * NW < p.n_chunks; c += 8 * NW) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = ld_hint_f1(base + (size_t)(c + NW * i) * stride, pol);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += v[i];
    }
    // the rest: fewer than 8 chunks a warp
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c + NW * i < p.n_chunks) acc[i] += ld_hint_f1(base + (size_t)(c + NW * i) * stride, pol);
  }
  red[warp][lane] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
  __syncthreads();
  if (threadIdx.x < 32) {
    const int j = blockIdx.x * 32 + threadIdx.x;
    float r = 0.f;
    for (int w = 0; w < NW; ++w) r += red[w][threadIdx.x];
    if (j < p.H) (a == 0 ? p.dgamma : p.dbeta)[j] = r;
  }
}

template <typename TIn, int NG, bool LN, int SK>
rn_status launch_t(const BwdParams& p, const Launch& l, cudaStream_t s) {
  auto k = rn_bwd_kernel<TIn, NG, LN, SK>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l.smem) !=
      cudaSuccess)
    return RN_ERR_CUDA;
  int grid = 1;
  if (persistent_grid(k, l, &grid) != RN_OK) return RN_ERR_CUDA;
  k<<<grid, l.threads, l.smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

template <typename TIn, bool LN, int SK>
rn_status launch_wide(int ng, const BwdParams& p, const Launch& l, cudaStream_t s) {
  switch (ng) {
    case 2: return launch_t<TIn, 2, LN, SK>(p, l, s);
    case 4: return launch_t<TIn, 4, LN, SK>(p, l, s);
    default: return RN_ERR_UNSUPPORTED;
  }
}

// compact shape for NG 1, 2 and 4; wide shape: NG 2 and 4 in the 512-thread
// build, NG 4 in the larger one (the planner takes NG 2 only within 512)
template <typename TIn, bool LN>
rn_status launch_ng(int ng, const BwdParams& p, const Launch& l, cudaStream_t s) {
  const bool wide = l.threads > kMaxThreads || l.per_sm == 1;
  if (!wide) {
    switch (ng) {
      case 1: return launch_t<TIn, 1, LN, kCompact>(p, l, s);
      case 2: return launch_t<TIn, 2, LN, kCompact>(p, l, s);
      case 4:
        if (l.threads > kMaxThreadsNg4) return RN_ERR_UNSUPPORTED;
        return launch_t<TIn, 4, LN, kCompact>(p, l, s);
      default: return RN_ERR_UNSUPPORTED;
    }
  }
  if (l.threads > kMaxThreadsWide) return RN_ERR_UNSUPPORTED;
  if (l.threads <= kMaxThreadsWide512) return launch_wide<TIn, LN, kWide512>(ng, p, l, s);
  if (ng != 4) return RN_ERR_UNSUPPORTED;
  return launch_t<TIn, 4, LN, kWide>(p, l, s);
}

}  // namespace

namespace {

template <typename TIn, int NG, bool LN, bool BIG>
rn_status launch_fused_t(const BwdParams& p, const Launch& l, cudaStream_t s) {
  auto k = rn_bwd_fused_kernel<TIn, NG, LN, BIG>;
  if (l.threads > (BIG ? kFusedBig : kFusedCompact) || p.apply_warps > 16 ||
      l.threads != 32 * p.apply_warps || p.Q < 2)
    return RN_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l.smem) !=
      cudaSuccess)
    return RN_ERR_CUDA;
  int grid = 1;
  if (persistent_grid(k, l, &grid) != RN_OK) return RN_ERR_CUDA;
  k<<<grid, l.threads, l.smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

}  // namespace

// fp32 rows: 4 chunks (16 elements) a thread
rn_status launch_bwd_fused(bool ln, bool big, const BwdParams& p, const Launch& l, cudaStream_t s) {
  if (ln) return big ? launch_fused_t<float, 4, true, true>(p, l, s)
                     : launch_fused_t<float, 4, true, false>(p, l, s);
  return big ? launch_fused_t<float, 4, false, true>(p, l, s)
             : launch_fused_t<float, 4, false, false>(p, l, s);
}

// bf16 rows only: every fp32 row the library accepts (H <= 8192) takes the
// fused kernel
rn_status launch_bwd(bool ln, bool bf16, int ng, const BwdParams& p, const Launch& l,
                     cudaStream_t s) {
  if (!bf16) return RN_ERR_UNSUPPORTED;
  return ln ? launch_ng<uint16_t, true>(ng, p, l, s) : launch_ng<uint16_t, false>(ng, p, l, s);
}

// launched as a programmatic dependent of the backward kernel: its CTAs are
// placed as the backward's CTAs retire and wait (griddepcontrol.wait) for
// the partials
rn_status launch_colreduce(const ColReduceParams& p, cudaStream_t s) {
  const bool narrow = p.nacc * ((p.H + 63) / 64) > kRedOneWave;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = narrow ? dim3((unsigned)((p.H + 31) / 32), (unsigned)p.nacc)
                       : dim3((unsigned)((p.H + 63) / 64), (unsigned)p.nacc);
  cfg.blockDim = dim3(narrow ? 16 * 32 : 32 * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = narrow ? cudaLaunchKernelEx(&cfg, rn_colreduce_narrow_kernel, p)
                               : cudaLaunchKernelEx(&cfg, rn_colreduce_kernel, p);
  if (e != cudaSuccess) return RN_ERR_CUDA;
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
