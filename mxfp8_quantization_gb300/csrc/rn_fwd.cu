// Row-wise LayerNorm / RMSNorm forward with fused output quantization
// (page "Implementation:NVIDIA TransformerEngine PyTorch Ext Normalization",
// section "Description": the fully fused delayed-scaling path and both
// passes of the norm+amax-then-quantize current-scaling path).
//
// Design (one persistent CTA per SM, rows b, b + grid, b + 2 grid, ... for
// CTA b):
//   * producer warp: one lane streams rows of x into a ring of Q
//     shared-memory slots with the bulk-copy engine (cp.async.bulk,
//     completion on the slot's "full" mbarrier) and refills a slot as soon as
//     its rows have been read out ("empty").  A slot holds rps adjacent rows
//     (rps = 2^rps_log2), moved by one copy: a copy engine request has a cost
//     of its own, and rows of 4 KB one copy each left the stream at about
//     two thirds of the HBM rate (65536 x 2048 bf16, FP8 delayed: 93 us with
//     one row a copy, 59 us with two); so CTA b takes the row groups b,
//     b + grid, ... of rps rows each.  When a pass needs the saved
//     mu / rsigma of a row, the same lane fetches them into the slot with
//     4-byte cp.async tracked by the same barrier;
//   * worker warps, in groups of G warps (G = 1 up to H = 4096 bf16 /
//     2048 fp32, larger G for longer rows): a group takes every (W/G)-th row
//     of the CTA's sequence, copies it from its slot into registers (each
//     lane up to 16 chunks of 16 bytes), releases the slot at once, computes
//     the row statistics with warp shuffles (LayerNorm: mean, then the
//     centred sum of squares; RMSNorm: sum of squares; a group of several
//     warps adds its warp sums in warp order through shared memory), then
//     forms y = (x-mu)*rsigma*g + beta (RMSNorm: x*rsigma*g) and stores
//     bf16/fp32 or E4M3 codes.  gamma (+1 when zero-centred) and beta are
//     staged in shared memory once per CTA (read from global memory for the
//     longest rows, where they would not fit beside the ring);
//   so there is no hand-off between warps inside a row, and the per-row cost
//   (waits, reductions, addressing) is spread over up to 128 elements a lane.
//   * arithmetic is done on pairs of elements with the packed fp32 (f32x2)
//     instructions, and bf16 inputs enter through the mixed-precision
//     add/sub forms, which round exactly like convert-then-operate;
//   * the per-tensor amax is reduced per thread, per CTA, then with one
//     atomicMax on the fp32 bit pattern (ordered like the values for
//     non-negative numbers, NaN above +inf).  A one-thread kernel launched
//     just before zeroes amax; the forward is launched as its programmatic
//     dependent and waits for it (griddepcontrol.wait) only before that
//     atomicMax.
// With a residual (RES), the producer brings the residual row along with
// the x row, each lane forms h = x + residual rounded once to the stream
// dtype, stores it (the new residual stream) and normalizes h.  This file is
// compiled twice: as is (the plain instantiations) and with RN_FWD_RES_TU
// set (the residual ones), so that the two halves build in parallel.
// Current scaling runs the kernel twice: pass 1 (statistics + amax, no
// output) and pass 2 (quantize with 448/amax from the saved mu / rsigma), the
// second launched as a programmatic dependent of the first and walking the
// rows backwards so that it starts on the rows pass 1 left in L2.
// MXFP8 calls that want the rowwise blocks only take this kernel too, in one
// pass: the 1x32 block maximum over the 4 (bf16) or 8 (fp32) lanes of a
// block, its E8M0 code, and E4M3 codes of y * 2^-e.
// NVFP4 output takes the same two passes; its pass 2 quantizes each run of 16
// elements of a row (the chunks of two adjacent lanes for bf16, four for
// fp32) with one E4M3 scale: the lanes of a block exchange their maxima with
// shuffles, convert A * S/6 to E4M3, look the element factor S / value(code)
// up in a 128-entry shared-memory table built once per CTA, and convert
// y * factor to E2M1 codes, two per byte.
#include <cuda_runtime.h>

#include "rn_device.cuh"
#include "rn_internal.h"

#ifndef RN_FWD_RES_TU
#define RN_FWD_RES_TU 0
#endif

// the (G, NC, ONE) row shapes compiled in
#ifndef RN_FWD_SHAPES
#define RN_FWD_SHAPES                                                              \
  RN_FWD_SHAPE(1, 4, false) RN_FWD_SHAPE(1, 8, false) RN_FWD_SHAPE(1, 16, false)    \
  RN_FWD_SHAPE(1, 16, true) RN_FWD_SHAPE(2, 8, false) RN_FWD_SHAPE(2, 8, true)      \
  RN_FWD_SHAPE(2, 16, true) RN_FWD_SHAPE(4, 16, true) RN_FWD_SHAPE(8, 16, true)
#endif

namespace rn {
namespace {

__device__ unsigned g_err_fwd;

// threads a CTA: the row part a lane holds (NC chunks of 16 bytes) sets the
// registers a thread needs: NC = 16 -> 512 threads (128 registers),
// NC = 8 -> 768 (80), NC = 4 -> 1024 (64)
template <int NC>
constexpr int max_threads() {
  return NC >= 16 ? 512 : (NC >= 8 ? 768 : 1024);
}
// named barriers: 1 .. kMaxGroups for the worker groups (G >= 2), 15 for
// all workers
constexpr int kMaxGroups = 14;
constexpr int kBarWorkers = 15;
// rows the producer issues before waiting for the first one to land
constexpr int kStartRows = 2;

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// store the PAIRS y pairs of one chunk in the output format; o points at the
// chunk's first output byte
template <int PAIRS, int QM>
__device__ __forceinline__ void store_chunk(unsigned char* o, int out_f32, const float2* y,
                                            float scale) {
  if constexpr (QM == kQNone) {
    if (out_f32) {
      float4* q = reinterpret_cast<float4*>(o);
#pragma unroll
      for (int i = 0; i < PAIRS / 2; ++i)
        q[i] = make_float4(y[2 * i].x, y[2 * i].y, y[2 * i + 1].x, y[2 * i + 1].y);
    } else if constexpr (PAIRS == 4) {
      *reinterpret_cast<uint4*>(o) =
          make_uint4(pack_bf16x2(y[0].x, y[0].y), pack_bf16x2(y[1].x, y[1].y),
                     pack_bf16x2(y[2].x, y[2].y), pack_bf16x2(y[3].x, y[3].y));
    } else {
      *reinterpret_cast<uint2*>(o) =
          make_uint2(pack_bf16x2(y[0].x, y[0].y), pack_bf16x2(y[1].x, y[1].y));
    }
  } else {
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

// value of a non-negative E4M3 code (0..0x7F), exact (through f16)
__device__ __forceinline__ float e4m3_code_value(uint32_t code) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)code));
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"((unsigned short)(h2 & 0xFFFFu)));
  return f;
}

// E2M1 codes of 2 * PAIRS values (round to nearest even, saturating at 6),
// element 0 in the low nibble; PAIRS = 4 fills a word, PAIRS = 2 its low half
template <int PAIRS>
__device__ __forceinline__ uint32_t pack_e2m1(const float2* q) {
  uint32_t r;
  if constexpr (PAIRS == 4) {
    // (the first source of the conversion lands in the high nibble)
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(q[0].x), "f"(q[0].y), "f"(q[1].x), "f"(q[1].y), "f"(q[2].x), "f"(q[2].y),
          "f"(q[3].x), "f"(q[3].y));
  } else {
    unsigned short h;
    asm("{\n\t.reg .b8 b0, b1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "mov.b16 %0, {b0, b1};\n\t}"
        : "=h"(h)
        : "f"(q[0].x), "f"(q[0].y), "f"(q[1].x), "f"(q[1].y));
    r = h;
  }
  return r;
}

// The row groups of this CTA: b, b + g, b + 2g, ... (b = blockIdx.x,
// g = gridDim.x), from the last one when reverse; group k holds rows
// k rps .. k rps + rps - 1 (the last group of all may be short).
template <bool ONE>
struct RowSeq {
  int first, step, count;
  __device__ __forceinline__ explicit RowSeq(const FwdParams& p) {
    const int b = blockIdx.x, g = gridDim.x;
    if constexpr (ONE) {
      count = b < p.N ? (p.N - b + g - 1) / g : 0;
    } else {
      const int ng = (p.N + (1 << p.rps_log2) - 1) >> p.rps_log2;
      count = b < ng ? (ng - b + g - 1) / g : 0;
    }
    first = p.reverse ? b + (count - 1) * g : b;
    step = p.reverse ? -g : g;
  }
  __device__ __forceinline__ int group(int i) const { return first + i * step; }
};

// sum of one value per warp over the G warps of a group, added in warp
// order (the same on every warp of the group); buf selects one of four
// exchange buffers so that consecutive exchanges never overwrite a value a
// slower warp of the group has yet to read
template <int G>
__device__ __forceinline__ float group_sum(float v, float* red, int group, int wg, int lane,
                                           int buf) {
  if constexpr (G == 1) {
    return v;
  } else {
    float* b = red + (group * 4 + buf) * 8;
    if (lane == 0) b[wg] = v;
    named_sync(1 + group, 32 * G);
    float s = b[0];
#pragma unroll
    for (int w = 1; w < G; ++w) s += b[w];
    return s;
  }
}

// ONE: one row a slot, fixed at compile time.  Rows of 8 KB or more never
// share a slot, and shorter ones only at large N; the general form (slot
// size, row group and position arithmetic at run time) cost the 8192 x 4096
// FP8 forwards ~1.7 us in generated code, so the shapes that meet one row a
// slot are also compiled this way.
template <typename TIn, int NK, int QM, int G, int NC, bool ONE, bool RES>
__global__ void __launch_bounds__(max_threads<NC>(), 1) rn_fwd_kernel(const FwdParams p) {
  constexpr int VEC = 16 / (int)sizeof(TIn);
  using V = Vec<TIn, VEC>;
  using Raw = typename V::Raw;
  constexpr int PAIRS = V::PAIRS;
  constexpr int F4 = VEC / 4;  // float4 of gamma per chunk
  constexpr bool LN = (NK == kLn);
  constexpr bool NORM = (NK != kIdentity);
  constexpr bool NV = (QM == kQNvfp4);
  constexpr bool MXR = (QM == kQMxRow);
  // pass 2 of current scaling / NVFP4 gets mu / rsigma with each row
  constexpr bool PASS2 = (QM == kQCurQuant || NV);
  constexpr bool META = (PASS2 && NORM);
  constexpr bool STATS = (!PASS2 && NORM);
  constexpr bool AMAX = (QM == kQDelayed || QM == kQCurAmax);
  constexpr bool GB_SMEM = NORM && G <= 2;
  extern __shared__ __align__(128) unsigned char smem[];

  const int W = p.workers;  // warps 0 .. W-1; producer: W
  const int H = p.H;
  const int nchunks = H / VEC;
  const uint32_t row_bytes = (uint32_t)H * sizeof(TIn);
  const int lg = ONE ? 0 : p.rps_log2;
  const int rps = 1 << lg;                             // rows a slot holds
  const uint32_t grp_bytes = ONE ? row_bytes : (uint32_t)rps * row_bytes;
  const uint32_t slot_bytes = RES ? 2 * grp_bytes : grp_bytes;  // x rows (then the residual rows)
  const uint32_t Q = (uint32_t)p.Q;
  const size_t gb_bytes = GB_SMEM ? (size_t)H * sizeof(float) * (LN ? 2 : 1) : 0;

  float4* gsm = reinterpret_cast<float4*>(smem);  // [F4][nchunks]: g of chunk c, part j
  float4* bsm = gsm + (size_t)F4 * nchunks;       // same for beta (LayerNorm)
  unsigned char* ring = smem + gb_bytes;
  float2* rstat = reinterpret_cast<float2*>(ring + (size_t)Q * slot_bytes);  // [Q][rps] (mu, rsigma)
  float* red = reinterpret_cast<float*>(ONE ? rstat + Q : rstat + (size_t)Q * rps);  // [kMaxGroups][4][8]
  uint32_t* red2 = reinterpret_cast<uint32_t*>(red + kMaxGroups * 4 * 8);  // [32]
  uint64_t* full = reinterpret_cast<uint64_t*>(red2 + 32);                  // row landed
  uint64_t* empty = full + Q;                                               // row read out
  float* nv_tbl = reinterpret_cast<float*>(empty + Q);  // NVFP4: [128] S / value(code)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (QM == kQCurAmax && threadIdx.x == 0) pdl_launch_dependents();

  for (uint32_t i = threadIdx.x; i < Q; i += blockDim.x) {
    mbar_init(smem_u32(&full[i]), META ? 2 : 1);
    mbar_init(smem_u32(&empty[i]), ONE ? G : G * rps);
    fence_barrier_init();
  }
  __syncthreads();

  const RowSeq<ONE> seq(p);

  if (warp == W) {
    // ------------------------------------------------------------ producer
    // (starts streaming rows while the workers stage gamma / beta)
    if (lane == 0) {
      if constexpr (META) pdl_wait();  // mu / rsigma come from pass 1
      const unsigned char* xb = static_cast<const unsigned char*>(p.x);
      RingPos pos{0u, 0u};
      for (int i = 0; i < seq.count; ++i) {
        int r0, nr;
        uint32_t bytes;
        if constexpr (ONE) {
          r0 = seq.group(i);
          nr = 1;
          bytes = row_bytes;
        } else {
          r0 = seq.group(i) << lg;
          nr = min(rps, p.N - r0);  // rows of this group
          bytes = (uint32_t)nr * row_bytes;
        }
        const uint32_t s = pos.slot;
        // a start-up burst of whole rings from every SM lands all at once,
        // late; instead the first kStartRows slots go out alone and the rest
        // of the ring once slot 0 is in, so that the workers start early
        if (i == kStartRows) mbar_wait(smem_u32(&full[0]), 0u, &g_err_fwd, kErrFullWait);
        if (i >= (int)Q) mbar_wait(smem_u32(&empty[s]), pos.phase ^ 1u, &g_err_fwd, kErrEmptyWait);
        const uint32_t bar = smem_u32(&full[s]);
        if constexpr (META) {
          if constexpr (ONE) {
            if (LN) cp_async4(smem_u32(&rstat[s].x), p.mu + r0);
            cp_async4(smem_u32(&rstat[s].y), p.rsigma + r0);
          } else {
            for (int j = 0; j < nr; ++j) {
              if (LN) cp_async4(smem_u32(&rstat[s * rps + j].x), p.mu + r0 + j);
              cp_async4(smem_u32(&rstat[s * rps + j].y), p.rsigma + r0 + j);
            }
          }
          cp_async_arrive(bar);
        }
        mbar_arrive_expect_tx(bar, RES ? 2 * bytes : bytes);
        bulk_g2s(smem_u32(ring + (size_t)s * slot_bytes), xb + (size_t)r0 * row_bytes, bytes, bar);
        if constexpr (RES)
          bulk_g2s(smem_u32(ring + (size_t)s * slot_bytes + grp_bytes),
                   static_cast<const unsigned char*>(p.residual) + (size_t)r0 * row_bytes, bytes,
                   bar);
        pos.advance(1, Q);
      }
      // every copy this CTA issued must have landed before it exits
      const int first = seq.count > (int)Q ? seq.count - (int)Q : 0;
      for (int k = first; k < seq.count; ++k)
        mbar_wait(smem_u32(&full[k % Q]), (uint32_t)(k / Q) & 1u, &g_err_fwd, kErrDrainWait);
    }
    return;
  }

  if constexpr (GB_SMEM) {
    // chunk c's gamma as F4 float4, part j at gsm[j * nchunks + c], so that a
    // warp's 16-byte reads of consecutive chunks are contiguous
    // a thread issues the loads of up to 4 items before its first store (one
    // trip to memory, not one per item): the first row lands ~1.6 us in, and
    // staged one item at a time the workers were not ready before ~1.8 us
    const int n4 = H / 4, NT = 32 * W;
    for (int u0 = threadIdx.x; u0 < n4; u0 += 4 * NT) {
      float4 gv[4], bv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int u = u0 + k * NT;
        if (u < n4) {
          gv[k] = reinterpret_cast<const float4*>(p.gamma)[u];
          if (LN)
            bv[k] = p.beta ? reinterpret_cast<const float4*>(p.beta)[u]
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int u = u0 + k * NT;
        if (u < n4) {
          const int c = u / F4, j = u - c * F4;
          gsm[j * nchunks + c] = p.zcg ? make_float4(1.0f + gv[k].x, 1.0f + gv[k].y,
                                                     1.0f + gv[k].z, 1.0f + gv[k].w)
                                       : gv[k];
          if (LN) bsm[j * nchunks + c] = bv[k];
        }
      }
    }
    named_sync(kBarWorkers, 32 * W);
  }

  // ---------------------------------------------------------- worker warps
  const int group = warp / G, wg = warp - group * G;
  const int NGR = W / G;  // groups; NGR < Q, NGR <= kMaxGroups when G > 1
  // this lane's chunks: cbase + k * CSTEP for k < nvalid
  const int cbase = wg * 32 + lane;
  constexpr int CSTEP = 32 * G;
  const int nv = cbase < nchunks ? (nchunks - cbase + CSTEP - 1) / CSTEP : 0;
  const int nvalid = nv < NC ? nv : NC;
  // the apply loop keeps a (then always true) test per chunk even for full
  // rows: with the chunks in one straight block the scheduler overlaps the
  // gamma / beta reads of many chunks and runs out of registers
  int nvalid_apply;
  asm volatile("mov.b32 %0, %1;" : "=r"(nvalid_apply) : "r"(nvalid));
  const float inv_h = 1.0f / (float)H;
  const int oesz = (QM == kQNone) ? (p.out_f32 ? 4 : 2) : 1;  // output bytes per element
  // output bytes from k to k + 1 (NVFP4: half a byte per element)
  const size_t ostep = NV ? (size_t)CSTEP * VEC / 2 : (size_t)CSTEP * VEC * oesz;

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
  float kq = 0.0f;  // NVFP4: S / 6
  if constexpr (NV) {
    pdl_wait();  // amax comes from pass 1
    const float am = *p.amax;
    float S = (am == 0.0f) ? 1.0f : __fdiv_rn(2688.0f, am);  // 448 * 6 / amax
    if (S > 3.402823466e38f) S = 3.402823466e38f;             // (NaN passes through)
    kq = __fdiv_rn(S, 6.0f);
    for (int c = threadIdx.x; c < 128; c += 32 * W)
      nv_tbl[c] = (c == 0) ? 0.0f : __fdiv_rn(S, e4m3_code_value((uint32_t)c));
    if (blockIdx.x == 0 && threadIdx.x == 0) {
      *p.scale_out = S;
      *p.scale_inv = __fdiv_rn(1.0f, S);
    }
    named_sync(kBarWorkers, 32 * W);
  }
  float ymax = 0.0f;  // running max |y| (NaN wins)

  // position i of the CTA's rows: row i & (rps - 1) of its group i >> lg,
  // whose slot and phase `pos` tracks (groups advance by less than Q per
  // step: NGR <= (Q - 1) rps)
  // (one row a slot: position i is slot use i, and pos advances by NGR
  // after each use)
  RingPos pos{ONE ? (uint32_t)group : 0u, 0u};
  int kgp = group >> lg;  // the previous position's row group
  if constexpr (!ONE) pos.advance((uint32_t)kgp, Q);
  int par = 0;
  for (int i = group; i < (ONE ? seq.count : seq.count << lg); i += NGR) {
    int kg, jr, r;
    if constexpr (ONE) {
      kg = i;
      jr = 0;
      r = seq.group(i);
    } else {
      pos.advance((uint32_t)((i >> lg) - kgp), Q);
      kg = kgp = i >> lg;
      jr = i & (rps - 1);
      r = (seq.group(kg) << lg) + jr;
      // the short last group of all: its missing rows are skipped by every
      // warp of the group (that slot is never used again)
      if (r >= p.N) continue;
    }
    const uint32_t s = pos.slot;
    // before waiting for this use of the slot, wait for the previous use to
    // be released: that use has then landed, so the parity wait below cannot
    // match a phase one lap old (alias-free since NGR <= (Q - 1) rps: a group
    // reaching this slot has already seen every earlier use of it issued)
    if (kg >= (int)Q) mbar_wait(smem_u32(&empty[s]), pos.phase ^ 1u, &g_err_fwd, kErrStatsWait);
    mbar_wait(smem_u32(&full[s]), pos.phase, &g_err_fwd, kErrFullWait);
    const unsigned char* rowp = ring + (size_t)s * slot_bytes + (size_t)jr * row_bytes;
    Raw raw[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k)
      if (k < nvalid) {
        raw[k] = V::load(rowp, cbase + k * CSTEP);
        if constexpr (RES) raw[k] = V::add_rn(raw[k], V::load(rowp + grp_bytes, cbase + k * CSTEP));
      }
    float mean = 0.0f, rs = 1.0f;
    if constexpr (META) {
      const float2 m = rstat[s * rps + jr];
      mean = LN ? m.x : 0.0f;
      rs = m.y;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    if constexpr (ONE) pos.advance((uint32_t)NGR, Q);
    if constexpr (RES) {
      // the new residual stream: h in the input dtype
      unsigned char* hrow = static_cast<unsigned char*>(p.residual_out) + (size_t)r * row_bytes;
#pragma unroll
      for (int k = 0; k < NC; ++k)
        if (k < nvalid) V::store(hrow, cbase + k * CSTEP, raw[k]);
    }

    if constexpr (STATS) {
      float2 a[PAIRS];
      if constexpr (LN) {
#pragma unroll
        for (int j = 0; j < PAIRS; ++j) a[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < NC; ++k)
          if (k < nvalid) {
#pragma unroll
            for (int j = 0; j < PAIRS; ++j) V::acc(a[j], raw[k], j);
          }
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < PAIRS; ++j) sum += a[j].x + a[j].y;
        mean = group_sum<G>(warp_sum(sum), red, group, wg, lane, 2 * par) * inv_h;
      }
#pragma unroll
      for (int j = 0; j < PAIRS; ++j) a[j] = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < NC; ++k)
        if (k < nvalid) {
#pragma unroll
          for (int j = 0; j < PAIRS; ++j) {
            if constexpr (LN) {
              const float2 d = V::sub(raw[k], j, mean);
              a[j] = fma2(d, d, a[j]);
            } else {
              V::sq_acc(a[j], raw[k], j);
            }
          }
        }
      float m2 = 0.f;
#pragma unroll
      for (int j = 0; j < PAIRS; ++j) m2 += a[j].x + a[j].y;
      m2 = group_sum<G>(warp_sum(m2), red, group, wg, lane, 2 * par + 1);
      rs = __frsqrt_rn(m2 * inv_h + p.eps);
      if (wg == 0 && lane == 0) {
        if constexpr (LN) p.mu[r] = mean;
        p.rsigma[r] = rs;
      }
      par ^= 1;
    }

    unsigned char* orow =
        NV ? static_cast<unsigned char*>(p.out) + ((size_t)r * H + (size_t)cbase * VEC) / 2
           : static_cast<unsigned char*>(p.out) + ((size_t)r * H + (size_t)cbase * VEC) * oesz;
    // NVFP4 / MXFP8 block scales: one byte per 16 / 32 elements, written by
    // the block's first lane
    uint8_t* srow = NV    ? p.scales + ((size_t)r * H + (size_t)cbase * VEC) / 16
                    : MXR ? p.scales + ((size_t)r * H + (size_t)cbase * VEC) / 32
                          : nullptr;
    const float2 rs2 = splat2(rs);
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      float2 y[PAIRS];
      float bm = 0.0f;  // NVFP4 / MXFP8 rowwise: max |y| of this lane's chunk
      if (k < nvalid_apply) {
        const int c = cbase + k * CSTEP;
        float4 gv[F4], bv[F4];
        if constexpr (NORM) {
#pragma unroll
          for (int j = 0; j < F4; ++j) {
            if constexpr (GB_SMEM) {
              gv[j] = gsm[j * nchunks + c];
              if (LN) bv[j] = bsm[j * nchunks + c];
            } else {
              gv[j] = __ldg(reinterpret_cast<const float4*>(p.gamma) + c * F4 + j);
              if (p.zcg)
                gv[j] = make_float4(1.0f + gv[j].x, 1.0f + gv[j].y, 1.0f + gv[j].z, 1.0f + gv[j].w);
              if (LN)
                bv[j] = p.beta ? __ldg(reinterpret_cast<const float4*>(p.beta) + c * F4 + j)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < PAIRS; ++j) {
          if constexpr (NORM) {
            const float4& g4 = gv[j / 2];
            const float2 gp = (j & 1) ? make_float2(g4.z, g4.w) : make_float2(g4.x, g4.y);
            if constexpr (LN) {
              const float4& b4 = bv[j / 2];
              const float2 bp = (j & 1) ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
              // x + (-mean): the same value as x - mean, written differently
              // so that the compiler does not keep the variance pass's
              // differences alive (128 registers) to reuse them here
              y[j] = fma2(mul2(V::add(raw[k], j, -mean), rs2), gp, bp);
            } else {
              y[j] = mul2(mul2(V::f32(raw[k], j), rs2), gp);
            }
          } else {
            y[j] = V::f32(raw[k], j);
          }
          if constexpr (AMAX) {
            ymax = amax_acc2(ymax, y[j]);  // one 3-input max on magnitudes a pair
          }
          if constexpr (NV) bm = fmaxf(bm, fmaxf(fabsf(y[j].x), fabsf(y[j].y)));
          if constexpr (MXR) bm = amax_acc2(bm, y[j]);  // NaN wins
        }
        if constexpr (QM != kQCurAmax && !NV && !MXR)
          store_chunk<PAIRS, QM>(orow + (size_t)k * ostep, p.out_f32, y, scale);
      }
      if constexpr (NV) {
        // a block of 16 elements spans 16 / VEC adjacent lanes (all of them
        // valid or none, since H % 16 == 0); every lane takes part in the
        // exchange
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
        if constexpr (VEC == 4) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
        if (k < nvalid_apply) {
          const uint32_t sc = pack_e4m3x2(__fmul_rn(bm, kq), 0.0f) & 0x7Fu;
          const float2 e2 = splat2(nv_tbl[sc]);
          float2 q[PAIRS];
#pragma unroll
          for (int j = 0; j < PAIRS; ++j) q[j] = mul2(y[j], e2);
          const uint32_t codes = pack_e2m1<PAIRS>(q);
          unsigned char* o = orow + (size_t)k * ostep;
          if constexpr (PAIRS == 4)
            *reinterpret_cast<uint32_t*>(o) = codes;
          else
            *reinterpret_cast<unsigned short*>(o) = (unsigned short)codes;
          if ((lane & (16 / VEC - 1)) == 0) srow[(size_t)k * (CSTEP * VEC / 16)] = (uint8_t)sc;
        }
      }
      if constexpr (MXR) {
        // a 1x32 block spans 32 / VEC adjacent lanes (all valid or none:
        // H % 32 == 0); E8M0 code of the block maximum, codes E4M3(y * 2^-e)
#pragma unroll
        for (int o = 1; o < 32 / VEC; o <<= 1) {
          const float w = __shfl_xor_sync(0xffffffffu, bm, o);
          asm("max.NaN.f32 %0, %0, %1;" : "+f"(bm) : "f"(w));
        }
        // (no rowwise output: the residual add's first kernel when only the
        // columnwise blocks are asked for)
        if (k < nvalid_apply && p.out != nullptr) {
          const uint32_t code = e8m0_code(bm);
          store_chunk<PAIRS, QM>(orow + (size_t)k * ostep, 0, y, e8m0_inv_scale(code));
          if ((lane & (32 / VEC - 1)) == 0) srow[(size_t)k * (CSTEP * VEC / 32)] = (uint8_t)code;
        }
      }
    }
  }

  if constexpr (AMAX) {
    const uint32_t b = warp_umax(abs_bits(ymax));
    if (lane == 0) red2[warp] = b;
    named_sync(kBarWorkers, 32 * W);
    if (threadIdx.x == 0) {
      uint32_t m = 0;
      for (int w = 0; w < W; ++w) m = max(m, red2[w]);
      pdl_wait();  // amax was zeroed by the kernel this one depends on
      atomicMax(reinterpret_cast<unsigned int*>(p.amax), m);
    }
  }
}

#if !RN_FWD_RES_TU
// zeroes amax (and forms scale_inv = 1/scale for delayed scaling) ahead of
// the forward, which is launched as its programmatic dependent
__global__ void rn_fwd_init_kernel(float* amax, const float* scale, float* scale_inv) {
  pdl_launch_dependents();
  *amax = 0.0f;
  if (scale != nullptr) *scale_inv = __fdiv_rn(1.0f, *scale);
}
#endif

template <typename TIn, int NK, int QM, int G, int NC, bool ONE>
rn_status launch_t(const FwdParams& p, const Launch& l, bool pdl, cudaStream_t s) {
  auto k = rn_fwd_kernel<TIn, NK, QM, G, NC, ONE, RN_FWD_RES_TU != 0>;
  if (ONE && p.rps_log2 != 0) return RN_ERR_UNSUPPORTED;
  // the shared-memory exchange buffers and named barriers exist for at most
  // kMaxGroups groups of G >= 2 warps and 31 worker warps
  const int workers = l.threads / 32 - 1;
  if (l.threads > max_threads<NC>() || workers != p.workers || workers % G != 0 || workers > 31 ||
      (G > 1 && workers / G > kMaxGroups))
    return RN_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l.smem) !=
      cudaSuccess)
    return RN_ERR_CUDA;
  int grid = 1;
  if (persistent_grid(k, l, &grid) != RN_OK) return RN_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)l.threads);
  cfg.dynamicSmemBytes = l.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, k, p) != cudaSuccess) return RN_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

// row shapes (G, NC, ONE); the planner picks one of these
template <typename TIn, int NK, int QM>
rn_status launch_shape(const FwdShape& sh, const FwdParams& p, const Launch& l, bool pdl,
                       cudaStream_t s) {
#define RN_FWD_SHAPE(G_, NC_, ONE_) \
  if (sh.g == G_ && sh.nc == NC_ && sh.one == ONE_) return launch_t<TIn, NK, QM, G_, NC_, ONE_>(p, l, pdl, s);
  RN_FWD_SHAPES
#undef RN_FWD_SHAPE
  return RN_ERR_UNSUPPORTED;
}

template <typename TIn, int NK>
rn_status launch_q(const FwdShape& sh, int qmode, const FwdParams& p, const Launch& l, bool pdl,
                   cudaStream_t s) {
  switch (qmode) {
    case kQNone:
      if constexpr (NK == kIdentity) return RN_ERR_UNSUPPORTED;
      else return launch_shape<TIn, NK, kQNone>(sh, p, l, pdl, s);
    case kQDelayed: return launch_shape<TIn, NK, kQDelayed>(sh, p, l, pdl, s);
    case kQCurAmax: return launch_shape<TIn, NK, kQCurAmax>(sh, p, l, pdl, s);
    case kQMxRow: return launch_shape<TIn, NK, kQMxRow>(sh, p, l, pdl, s);
#if !RN_FWD_RES_TU
    // (with a residual, the second passes read the stored sum as their x:
    // the plain kernel)
    case kQCurQuant: return launch_shape<TIn, NK, kQCurQuant>(sh, p, l, pdl, s);
    case kQNvfp4: return launch_shape<TIn, NK, kQNvfp4>(sh, p, l, pdl, s);
#endif
    default: return RN_ERR_INVALID;
  }
}

}  // namespace

#if RN_FWD_RES_TU

rn_status launch_fwd_res(int nk, bool bf16, const FwdShape& sh, int qmode, const FwdParams& p,
                         const Launch& l, bool pdl, cudaStream_t s) {
  if (nk == kIdentity || p.residual == nullptr || p.residual_out == nullptr) return RN_ERR_INVALID;
  if (bf16)
    return nk == kLn ? launch_q<uint16_t, kLn>(sh, qmode, p, l, pdl, s)
                     : launch_q<uint16_t, kRms>(sh, qmode, p, l, pdl, s);
  return nk == kLn ? launch_q<float, kLn>(sh, qmode, p, l, pdl, s)
                   : launch_q<float, kRms>(sh, qmode, p, l, pdl, s);
}

rn_status read_clear_error_fwd_res(unsigned* code) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_fwd, sizeof(v)) != cudaSuccess) return RN_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_err_fwd, &zero, sizeof(zero)) != cudaSuccess) return RN_ERR_CUDA;
  *code = v;
  return RN_OK;
}

#else

rn_status launch_fwd_init(float* amax, const float* scale, float* scale_inv, cudaStream_t s) {
  rn_fwd_init_kernel<<<1, 1, 0, s>>>(amax, scale, scale_inv);
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

rn_status launch_fwd(int nk, bool bf16, const FwdShape& sh, int qmode, const FwdParams& p,
                     const Launch& l, bool pdl, cudaStream_t s) {
  if (nk == kIdentity)
    return bf16 ? RN_ERR_UNSUPPORTED : launch_q<float, kIdentity>(sh, qmode, p, l, pdl, s);
  if (bf16)
    return nk == kLn ? launch_q<uint16_t, kLn>(sh, qmode, p, l, pdl, s)
                     : launch_q<uint16_t, kRms>(sh, qmode, p, l, pdl, s);
  return nk == kLn ? launch_q<float, kLn>(sh, qmode, p, l, pdl, s)
                   : launch_q<float, kRms>(sh, qmode, p, l, pdl, s);
}

rn_status read_clear_error_fwd(unsigned* code) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_err_fwd, sizeof(v)) != cudaSuccess) return RN_ERR_CUDA;
  if (cudaMemcpyToSymbol(g_err_fwd, &zero, sizeof(zero)) != cudaSuccess) return RN_ERR_CUDA;
  *code = v;
  return RN_OK;
}

#endif  // RN_FWD_RES_TU

}  // namespace rn
