// C ABI of the library (declared in include/rn.h): argument validation,
// launch planning and dispatch.  Everything here runs on the host and
// checks every argument before anything is enqueued.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "rn_internal.h"

namespace rn {
namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];
std::atomic<int> g_smem[kMaxDevices];
std::atomic<int> g_smem_sm[kMaxDevices];

constexpr int kMaxConsumers = 512;
constexpr int kBwdTileRows = 8;
constexpr int kBwdTargetChunks = 1024;  // chunks per call, roughly
constexpr int kBwdWideChunksPerCta = 3;  // wide shape: at most chunks a CTA at sm_margin 0

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int round_up(int v, int m) { return (v + m - 1) / m * m; }

int elem_size(rn_dtype d) { return d == RN_BF16 ? 2 : 4; }

bool dtype_ok(rn_dtype d) { return d == RN_BF16 || d == RN_F32; }

// x rows must be whole 16-byte chunks (bulk copies and vector loads)
bool row_ok(int64_t H, rn_dtype d) { return (H * elem_size(d)) % 16 == 0; }

// smallest group count in {1, 2, 4} that keeps the consumer threads <= cap
int pick_ng(int nchunks, int cap, int max_ng) {
  for (int ng = 1; ng <= max_ng; ng *= 2)
    if ((nchunks + ng - 1) / ng <= cap) return ng;
  return 0;
}

}  // namespace

rn_status device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return RN_ERR_UNSUPPORTED;
  int sms = g_sms[dev].load(std::memory_order_relaxed);
  int smem = g_smem[dev].load(std::memory_order_relaxed);
  int smem_sm = g_smem_sm[dev].load(std::memory_order_relaxed);
  if (sms <= 0 || smem <= 0 || smem_sm <= 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return RN_ERR_CUDA;
    if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return RN_ERR_CUDA;
    if (cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
        cudaSuccess)
      return RN_ERR_CUDA;
    g_sms[dev].store(sms, std::memory_order_relaxed);
    g_smem[dev].store(smem, std::memory_order_relaxed);
    g_smem_sm[dev].store(smem_sm, std::memory_order_relaxed);
  }
  out->sms = sms;
  out->smem_optin = smem;
  out->smem_per_sm = smem_sm;
  return RN_OK;
}

namespace {

// ---------------------------------------------------------------- planning

// shared memory one CTA may use when per_sm CTAs share an SM (the runtime
// reserves 1 KB per CTA)
size_t cta_smem_budget(const DeviceInfo& di, int per_sm) {
  const long long b = ((long long)di.smem_per_sm - 1024LL * per_sm) / per_sm;
  const long long cap = di.smem_optin;
  return (size_t)(b < cap ? b : cap);
}

// Warp roles of the row kernels: A apply warps (each thread owning NG
// 16-byte chunks of every row), S = max(2, A/2) stats warps (at most 3 in
// the compact shape; fewer than the ring's slots, which their pacing on slot
// releases relies on), one producer.  Compact shape: NG = 1 (A <= 8) or 4
// (A <= 4), two CTAs per SM when each still holds a ring of >= 6 slots.
// Otherwise the wide shape: one CTA per SM, NG 2 or 4 (4 when 2 would take
// the CTA past 512 threads: the 512-thread build has 128 registers a
// thread, the larger one 96), A <= 16, at most kBwdWideThreads threads.
struct Roles {
  int ng, A, S, per_sm, Q;
};

rn_status plan_roles(int nchunks, bool ln, size_t per_slot, size_t fixed, const DeviceInfo& di,
                     int q_cap, Roles* r) {
  // LayerNorm rows of more than 480 chunks (bf16 H > 3840) take the wide
  // shape, one CTA per SM with 8 apply and 4 stats warps at H = 4096: no SM
  // is left with one CTA running its last chunk alone (8192 x 4096: 39.2
  // against 41.2 us; 16384 x 4096: 70.7 against 73.7 us; 4096 x 4096: 26.8
  // against 27.4 us; sm_margin 16: 41.7 against 45.2 us).  Narrower
  // LayerNorm rows measured no better or worse that way (H = 2560: 53.4
  // against 49.4 us, 3072 even, 3584: 40.5 against 39.1 us at 12288 /
  // 8192 rows), and RMSNorm rows worse (8192 x 4096: 37.1 against 35.3 us;
  // with the wide shape's 2-3 chunks a CTA even, 35.1 against 35.4 us, but
  // 41.5 against 37.3 us at sm_margin 16).
  if (nchunks <= 512 && !(ln && nchunks > 480)) {
    // rows of 257 .. 512 chunks: 4 chunks a thread and 4 apply warps (the
    // per-row waits and addressing spread over twice the elements: 42.7 ->
    // 41.2 us at 8192 x 4096 LayerNorm bf16 against 2 chunks and 8 warps)
    const int ng = nchunks <= 256 ? 1 : 4;
    const size_t budget = cta_smem_budget(di, 2);
    int Q = budget > fixed ? (int)((budget - fixed) / per_slot) : 0;
    if (Q > q_cap) Q = q_cap;
    if (Q >= 6) {
      r->ng = ng;
      r->A = round_up((nchunks + ng - 1) / ng, 32) / 32;
      r->S = r->A / 2 > 2 ? r->A / 2 : 2;
      if (r->S > 3) r->S = 3;          // 12 warps a CTA: 80 registers a thread
      if (ng == 4) r->S = 3;           // 8 warps a CTA (2 stats warps: 43.4 us)
      if (r->S > Q - 1) r->S = Q - 1;  // stats warps must be fewer than slots
      r->per_sm = 2;
      r->Q = Q;
      return RN_OK;
    }
  }
  const size_t budget = cta_smem_budget(di, 1);
  int Q = budget > fixed ? (int)((budget - fixed) / per_slot) : 0;
  if (Q > q_cap) Q = q_cap;
  if (Q < 2) return RN_ERR_UNSUPPORTED;
  auto roles = [&](int ng, int* A, int* S) {
    *A = round_up((nchunks + ng - 1) / ng, 32) / 32;
    *S = *A / 2 > 2 ? *A / 2 : 2;
    if (*S > Q - 1) *S = Q - 1;  // stats warps must be fewer than slots
    const int cap = kBwdWideThreads / 32 - *A - 1;
    if (*S > cap) *S = cap;
  };
  int ng = 0, A = 0, S = 0;
  for (int g = 2; g <= 4 && ng == 0; g *= 2) {
    if ((nchunks + g - 1) / g > 512) continue;
    roles(g, &A, &S);
    if (32 * (A + S + 1) <= kBwdWideThreads512) ng = g;
  }
  if (ng == 0) {
    ng = (nchunks + 1) / 2 <= 512 ? 2 : 4;
    if ((nchunks + ng - 1) / ng > 512) return RN_ERR_UNSUPPORTED;
    roles(ng, &A, &S);
  }
  if (S < 1) return RN_ERR_UNSUPPORTED;
  r->ng = ng;
  r->A = A;
  r->S = S;
  r->per_sm = 1;
  r->Q = Q;
  return RN_OK;
}

// Row-wise forward: rows are taken by groups of G warps, the fewest that
// hold a row with <= 16 chunks of 16 bytes a lane (NC = 4 or 8 chunks for
// short rows; see plan_fwd for the bf16 LayerNorm exception); every chunk
// keeps its bounds test (variants without them needed more than the 128
// registers a thread of a 512-thread CTA has).  Threads a CTA follow from
// NC (512 for NC = 16, 768 for 8, 1024
// for 4: the registers of the row part); W = every warp but the producer, in whole
// groups, at most 14 groups of G >= 2; one CTA per SM; a ring of Q slots of
// 2^rps_log2 adjacent rows each, W / G <= (Q - 1) 2^rps_log2.
struct FwdPlan {
  FwdShape sh;
  int workers, Q, rps_log2;
  Launch l;
};

int fwd_max_threads(int nc) { return nc >= 16 ? 512 : (nc >= 8 ? 768 : 1024); }

rn_status plan_fwd(int nk, int H, int esz, int N, int sm_margin, const DeviceInfo& di,
                   FwdPlan* pl, int streams = 1, size_t extra_bytes = 0) {
  const int nchunks = H * esz / 16;
  FwdShape sh{1, 16, false};
  while (sh.g <= 8 && nchunks > 32 * sh.g * 16) sh.g *= 2;
  if (sh.g > 8) return RN_ERR_UNSUPPORTED;
  if (sh.g == 1 && nchunks <= 32 * 4) sh.nc = 4;
  // rows of 129 .. 256 chunks: 8 chunks a lane and 24 warps an SM (16 chunks
  // and 16 warps left half of each lane's registers idle: 65536 x 2048 bf16
  // FP8 delayed 97 -> 93 us, MXFP8 rowwise 111 -> 97 us)
  else if (sh.g == 1 && nchunks <= 32 * 8) sh.nc = 8;
  // bf16 LayerNorm rows of 257 .. 512 chunks: two warps a row, 8 chunks a
  // lane (24 warps an SM instead of 16 hide more of the two statistics
  // passes: 23.8 -> 22.8 us at 8192 x 4096; RMSNorm's single pass gains
  // nothing and pays the group exchange: 20.7 -> 22.7 us, so it keeps G = 1)
  if (nk == kLn && esz == 2 && sh.g == 1 && sh.nc == 16 && nchunks > 32 * 8) {
    sh.g = 2;
    sh.nc = 8;
  }
  const int g = sh.g;
  // gamma (and beta) staged in shared memory for G <= 2, read through L1
  // for longer rows
  const size_t gb =
      (nk != kIdentity && g <= 2) ? (size_t)H * sizeof(float) * (nk == kLn ? 2 : 1) : 0;
  // a slot holds 2^lg adjacent rows, moved by one copy (each copy request
  // costs the copy engine time of its own: 4 KB rows one a copy kept the
  // stream at two thirds of the HBM rate): copies of at least 8 KB, as long
  // as every SM still gets 4 groups or more
  const size_t row_bytes = (size_t)H * esz;
  const long long sms = di.sms - sm_margin;
  int lg = 0;
  while (lg < 3 && (row_bytes << lg) < 8192 && (long long)(N >> (lg + 1)) >= 4 * sms) ++lg;
  const int rps = 1 << lg;
  // one row a slot compiled as such: every shape but the two shortest-row
  // ones (1 x 4 and 1 x 8 chunks a lane, which group at large N) has that
  // instantiation
  sh.one = lg == 0 && !(sh.g == 1 && sh.nc < 16);
  // fixed: gamma/beta, group exchange (14 groups x 4 x 8 floats), amax words
  // (32), slack; per slot: the rows, their (mu, rsigma), two mbarriers
  // (+ extra_bytes after the barriers: the NVFP4 factor table)
  const size_t fixed = gb + 14 * 4 * 8 * sizeof(float) + 32 * sizeof(uint32_t) + 64 + extra_bytes;
  // (with a residual add a slot holds the x rows and the residual rows)
  const size_t per_slot = (size_t)rps * ((size_t)streams * row_bytes + sizeof(float2)) + 16;
  const size_t budget = cta_smem_budget(di, 1);
  int Q = budget > fixed ? (int)((budget - fixed) / per_slot) : 0;
  if (Q > 64) Q = 64;
  if (g >= 4) {
    // leave L1 room for gamma / beta (but keep two slots when they fit)
    int qmax = (int)((size_t(128) << 10) / per_slot);
    if (qmax < 2) qmax = 2;
    if (Q > qmax) Q = qmax;
  }
  if (Q < 2) return RN_ERR_UNSUPPORTED;
  int W = (fwd_max_threads(sh.nc) / 32 - 1) / g * g;
  // groups of several warps: at most 14 (their named barriers are 1 .. 14)
  if (g > 1 && W / g > 14) W = 14 * g;
  // rows in work at once (one a group) stay within Q - 1 slots, which keeps
  // the slot barriers' parity waits alias-free
  while (W > g && W / g > (Q - 1) * rps) W -= g;
  if (W / g > (Q - 1) * rps) return RN_ERR_UNSUPPORTED;
  pl->sh = sh;
  pl->workers = W;
  pl->Q = Q;
  pl->rps_log2 = lg;
  pl->l.threads = 32 * (W + 1);
  pl->l.smem = (size_t)Q * per_slot + fixed;
  pl->l.work = (N + rps - 1) / rps;
  pl->l.sms = di.sms - sm_margin;
  pl->l.per_sm = 1;
  return RN_OK;
}

// MXFP8: apply warps take 64-column sub-tiles of each 32-row tile (A <= 10
// warps, as few as give the same sub-tiles per warp), S = min(8, 15 - A)
// stats warps, a producer; one CTA per SM with a
// ring of at least 33 rows (a 32-row tile plus look-ahead) and gamma / beta
// staged in shared memory.
struct MxPlan {
  int Q, n_tbar, apply_warps, stats_warps;
  Launch l;
};

rn_status plan_mx(int nk, int H, int esz, int N, int sm_margin, const DeviceInfo& di,
                  MxPlan* pl) {
  const int nsub = (H + 63) / 64;
  // the largest A <= 10 that spreads the sub-tiles evenly
  int A = nsub < 10 ? nsub : 10;
  while (A > 1 && (nsub % A) != 0 && (nsub + A - 1) / A == (nsub + A - 2) / (A - 1)) --A;
  // stats warps: as many as fit beside the apply warps in 15 (a 32-row tile's
  // statistics should keep up with its apply work)
  int S = 15 - A;
  if (S > 8) S = 8;
  const size_t row_bytes = (size_t)H * esz;
  if (H / 8 > 32 * 16) return RN_ERR_UNSUPPORTED;  // a stats lane holds <= 16 chunks
  const size_t gb = nk == kIdentity ? 0 : (size_t)H * sizeof(float) * (nk == kLn ? 2 : 1);
  // per slot: the row, (mean, rsigma), two mbarriers; fixed: gamma / beta,
  // the tile barriers (at most 8), slack
  const size_t per_slot = row_bytes + sizeof(float2) + 16;
  const size_t fixed = gb + 8 * sizeof(uint64_t) + 64;
  const size_t budget = cta_smem_budget(di, 1);
  int Q = budget > fixed ? (int)((budget - fixed) / per_slot) : 0;
  if (Q > 128) Q = 128;
  if (Q < 33) return RN_ERR_UNSUPPORTED;
  pl->Q = Q;
  pl->n_tbar = (Q + 31) / 32 + 2;  // <= 8
  pl->apply_warps = A;
  pl->stats_warps = S;
  pl->l.threads = 32 * (A + S + 1);
  pl->l.smem = (size_t)Q * per_slot + fixed;
  pl->l.work = N / 32;
  pl->l.sms = di.sms - sm_margin;
  pl->l.per_sm = 1;
  return RN_OK;
}

// MXFP8 box kernel (bf16 H a multiple of 64, fp32 H of 32; N of 32): 16
// worker warps, one CTA per SM; fixed: 1 KB for aligning the box ring to
// 1024 bytes, the statistics partials of two tiles (2 x 2 nbox x 32
// float2), two tiles' (mean, rsigma), two barriers; per slot: a 16 KB box,
// an mbarrier, a ticket and a pending-read count.  At least 4 slots.
rn_status plan_mx_box(int nk, int H, int esz, int N, int sm_margin, const DeviceInfo& di,
                      MxPlan* pl) {
  const int c0 = 128 / esz;
  if (H % c0 != 0 || N % 32 != 0) return RN_ERR_UNSUPPORTED;
  const int nbox = (H / c0 + 3) / 4;
  const int nus = nk == kIdentity ? 0 : 2 * nbox;
  const size_t fixed = 1024 + 2 * (size_t)nus * 32 * sizeof(float2) + 2 * 32 * sizeof(float2) +
                       4 * sizeof(uint64_t) + 64;
  const size_t per_slot = kMxBoxBytes + sizeof(uint64_t) + 2 * sizeof(uint32_t);
  const size_t budget = cta_smem_budget(di, 1);
  int Q = budget > fixed ? (int)((budget - fixed) / per_slot) : 0;
  if (Q > 64) Q = 64;
  if (Q < 4) return RN_ERR_UNSUPPORTED;
  pl->Q = Q;
  pl->n_tbar = 2;
  pl->apply_warps = 16;
  pl->stats_warps = 0;
  pl->l.threads = kMxBoxThreads;
  pl->l.smem = fixed + (size_t)Q * per_slot;
  pl->l.work = N / 32;
  pl->l.sms = di.sms - sm_margin;
  pl->l.per_sm = 1;
  return RN_OK;
}

// backward chunking: a chunk is R_N = 8 * max(1, N / 8192) rows, a function
// of N only (the wide stats-warp shape takes longer chunks, a function of N
// and the device's SM count, in bwd_common), never of the grid or
// sm_margin, so the dgamma/dbeta partials and their sum are independent of
// sm_margin; the workspace is sized for R_N chunks, the most any shape uses
struct BwdShape {
  int chunk_rows, n_chunks;
};

rn_status bwd_shape(int64_t N, int64_t H, int esz, BwdShape* s) {
  if (pick_ng((int)(H * esz / 16), kMaxConsumers, 4) == 0) return RN_ERR_UNSUPPORTED;
  const int64_t m = N / (int64_t)(kBwdTileRows * kBwdTargetChunks);
  s->chunk_rows = kBwdTileRows * (int)(m < 1 ? 1 : m);
  s->n_chunks = (int)((N + s->chunk_rows - 1) / s->chunk_rows);
  return RN_OK;
}

size_t bwd_workspace(const BwdShape& s, int64_t H, bool ln) {
  return (size_t)s.n_chunks * (ln ? 2 : 1) * (size_t)H * sizeof(float);
}

// ---------------------------------------------------------------- checks
bool out_fields_only(const rn_output* o, bool data, bool rs, bool cd, bool cs, bool sc, bool so,
                     bool si, bool am) {
  return (o->data != nullptr) == data && (o->row_scales != nullptr) == rs &&
         (o->col_data != nullptr) == cd && (o->col_scales != nullptr) == cs &&
         (o->scale != nullptr) == sc && (o->scale_out != nullptr) == so &&
         (o->scale_inv != nullptr) == si && (o->amax != nullptr) == am;
}

rn_status check_out(rn_quant_mode mode, const rn_output* o, int64_t N, int64_t H) {
  if (o == nullptr) return RN_ERR_INVALID;
  if (N == 0) {
    // empty row tensors may have NULL data; only the scalar outputs matter
    if (mode == RN_QUANT_FP8_DELAYED)
      return (o->scale && o->scale_inv && o->amax) ? RN_OK : RN_ERR_INVALID;
    if (mode == RN_QUANT_FP8_CURRENT)
      return (o->scale_out && o->scale_inv && o->amax) ? RN_OK : RN_ERR_INVALID;
    if (mode == RN_QUANT_NONE)
      return (o->out_dtype == RN_BF16 || o->out_dtype == RN_F32) ? RN_OK : RN_ERR_INVALID;
    if (mode == RN_QUANT_MXFP8) return (H % 32 == 0) ? RN_OK : RN_ERR_UNSUPPORTED;
    if (mode == RN_QUANT_NVFP4) {
      if (!(o->scale_out && o->scale_inv && o->amax)) return RN_ERR_INVALID;
      return (H % 16 == 0) ? RN_OK : RN_ERR_UNSUPPORTED;
    }
    return RN_ERR_INVALID;
  }
  switch (mode) {
    case RN_QUANT_NONE:
      if (!out_fields_only(o, true, false, false, false, false, false, false, false))
        return RN_ERR_INVALID;
      if (o->out_dtype != RN_BF16 && o->out_dtype != RN_F32) return RN_ERR_INVALID;
      break;
    case RN_QUANT_FP8_DELAYED:
      if (!out_fields_only(o, true, false, false, false, true, false, true, true))
        return RN_ERR_INVALID;
      break;
    case RN_QUANT_FP8_CURRENT:
      if (!out_fields_only(o, true, false, false, false, false, true, true, true))
        return RN_ERR_INVALID;
      break;
    case RN_QUANT_MXFP8: {
      const bool rowwise = o->data != nullptr, colwise = o->col_data != nullptr;
      if (!rowwise && !colwise) return RN_ERR_INVALID;
      if (!out_fields_only(o, rowwise, rowwise, colwise, colwise, false, false, false, false))
        return RN_ERR_INVALID;
      if (H % 32 != 0 || N % 32 != 0) return RN_ERR_UNSUPPORTED;
      if (colwise && !aligned(o->col_data, 16)) return RN_ERR_UNSUPPORTED;
      break;
    }
    case RN_QUANT_NVFP4:
      if (!out_fields_only(o, true, true, false, false, false, true, true, true))
        return RN_ERR_INVALID;
      if (H % 16 != 0) return RN_ERR_UNSUPPORTED;
      break;
    default:
      return RN_ERR_INVALID;
  }
  if (o->data != nullptr && !aligned(o->data, 16)) return RN_ERR_UNSUPPORTED;
  if (o->amax && !aligned(o->amax, 4)) return RN_ERR_UNSUPPORTED;
  return RN_OK;
}

rn_status check_margin(int sm_margin, const DeviceInfo& di) {
  return (sm_margin < 0 || sm_margin >= di.sms) ? RN_ERR_INVALID : RN_OK;
}

// ---------------------------------------------------------------- forward
rn_status fwd_common(int nk, const void* x, rn_dtype dt, const float* gamma, const float* beta,
                     int64_t N, int64_t H, float eps, int zcg, int sm_margin, rn_quant_mode mode,
                     const rn_output* out, float* mu, float* rsigma, cudaStream_t stream,
                     bool res = false, const void* residual = nullptr,
                     void* residual_out = nullptr) {
  // with a residual add (res): residual and residual_out are [N, H] in x's
  // dtype; like the other row tensors they may be NULL when N == 0
  if (res && ((N > 0 && (residual == nullptr || residual_out == nullptr)) || nk == kIdentity))
    return RN_ERR_INVALID;
  if (res && N > 0 && (!aligned(residual, 16) || !aligned(residual_out, 16)))
    return RN_ERR_UNSUPPORTED;
  if ((x == nullptr && N > 0) || !dtype_ok(dt) || N < 0 || H < 1 || N > INT32_MAX ||
      H > INT32_MAX)
    return RN_ERR_INVALID;
  if (nk != kIdentity && (gamma == nullptr || (rsigma == nullptr && N > 0))) return RN_ERR_INVALID;
  if (nk == kLn && mu == nullptr && N > 0) return RN_ERR_INVALID;
  if (nk == kIdentity && mode == RN_QUANT_NONE) return RN_ERR_INVALID;
  rn_status st = check_out(mode, out, N, H);
  if (st != RN_OK) return st;
  if (!row_ok(H, dt) || !aligned(x, 16)) return RN_ERR_UNSUPPORTED;
  if ((gamma && !aligned(gamma, 16)) || (beta && !aligned(beta, 16)) ||
      (mu && !aligned(mu, 4)) || (rsigma && !aligned(rsigma, 4)))
    return RN_ERR_UNSUPPORTED;
  DeviceInfo di;
  if ((st = device_info(&di)) != RN_OK) return st;
  if ((st = check_margin(sm_margin, di)) != RN_OK) return st;
  if (N == 0 && mode == RN_QUANT_NONE) return RN_OK;
  if (N == 0 && mode == RN_QUANT_MXFP8) return RN_OK;
  const bool bf16 = dt == RN_BF16;
  const int esz = elem_size(dt);

  // the input of the two-direction MXFP8 kernels, and its rowwise outputs
  const void* mx_x = x;
  uint8_t* mx_data = mode == RN_QUANT_MXFP8 ? static_cast<uint8_t*>(out->data) : nullptr;
  uint8_t* mx_row_scales = mode == RN_QUANT_MXFP8 ? out->row_scales : nullptr;
  if (mode == RN_QUANT_MXFP8 && res && out->col_data != nullptr) {
    // residual add with the columnwise copy: the row kernel forms and stores
    // h = x + residual, the rowwise blocks (when asked for) and mu / rsigma in
    // one pass; the two-direction kernel below then reads h back for the
    // columnwise blocks (and writes mu / rsigma again, from the same h).
    // Both kernels are planned before the first is launched.
    MxPlan mp;
    if (plan_mx_box(nk, (int)H, esz, (int)N, sm_margin, di, &mp) != RN_OK &&
        (st = plan_mx(nk, (int)H, esz, (int)N, sm_margin, di, &mp)) != RN_OK)
      return st;
    FwdPlan pr;
    if ((st = plan_fwd(nk, (int)H, esz, (int)N, sm_margin, di, &pr, 2)) != RN_OK) return st;
    FwdParams p{};
    p.x = x;
    p.gamma = gamma;
    p.beta = beta;
    p.out = out->data;
    p.scales = out->data ? out->row_scales : nullptr;
    p.mu = mu;
    p.rsigma = rsigma;
    p.N = (int)N;
    p.H = (int)H;
    p.eps = eps;
    p.zcg = zcg ? 1 : 0;
    p.residual = residual;
    p.residual_out = residual_out;
    p.workers = pr.workers;
    p.Q = pr.Q;
    p.rps_log2 = pr.rps_log2;
    if ((st = launch_fwd_res(nk, bf16, pr.sh, kQMxRow, p, pr.l, false, stream)) != RN_OK) return st;
    mx_x = residual_out;
    mx_data = nullptr;
    mx_row_scales = nullptr;
  } else if (mode == RN_QUANT_MXFP8 && out->col_data == nullptr) {
    // rowwise blocks only: the row kernel in one pass (no 32-row tiles)
    FwdPlan pl;
    if ((st = plan_fwd(nk, (int)H, esz, (int)N, sm_margin, di, &pl)) != RN_OK) return st;
    FwdParams p{};
    p.x = x;
    p.gamma = gamma;
    p.beta = beta;
    p.out = out->data;
    p.scales = out->row_scales;
    p.mu = mu;
    p.rsigma = rsigma;
    p.N = (int)N;
    p.H = (int)H;
    p.eps = eps;
    p.zcg = zcg ? 1 : 0;
    p.workers = pl.workers;
    p.Q = pl.Q;
    p.rps_log2 = pl.rps_log2;
    if (res) {
      FwdPlan pr;
      if ((st = plan_fwd(nk, (int)H, esz, (int)N, sm_margin, di, &pr, 2)) != RN_OK) return st;
      p.residual = residual;
      p.residual_out = residual_out;
      p.workers = pr.workers;
      p.Q = pr.Q;
      p.rps_log2 = pr.rps_log2;
      return launch_fwd_res(nk, bf16, pr.sh, kQMxRow, p, pr.l, false, stream);
    }
    return launch_fwd(nk, bf16, pl.sh, kQMxRow, p, pl.l, false, stream);
  }
  if (mode == RN_QUANT_MXFP8) {
    MxPlan pl;
    // rows of whole 128-byte column blocks: the box kernel; other bf16 rows
    // (H of 32 mod 64 columns) the ring kernel, which holds a 32-row tile
    const bool box = plan_mx_box(nk, (int)H, esz, (int)N, sm_margin, di, &pl) == RN_OK;
    if (!box && (st = plan_mx(nk, (int)H, esz, (int)N, sm_margin, di, &pl)) != RN_OK) return st;
    MxParams p{};
    p.x = mx_x;
    p.gamma = gamma;
    p.beta = beta;
    p.data = mx_data;
    p.row_scales = mx_row_scales;
    p.col_data = out->col_data;
    p.col_scales = out->col_scales;
    p.mu = mu;
    p.rsigma = rsigma;
    p.N = (int)N;
    p.H = (int)H;
    p.eps = eps;
    p.zcg = zcg ? 1 : 0;
    p.Q = pl.Q;
    p.apply_warps = pl.apply_warps;
    p.stats_warps = pl.stats_warps;
    p.n_tiles = (int)(N / 32);
    p.n_tbar = pl.n_tbar;
    if (box) return launch_mx_box(nk, bf16, p, pl.l, stream);
    return launch_mx(nk, bf16, 1, p, pl.l, stream);
  }

  FwdPlan pl;
  if ((st = plan_fwd(nk, (int)H, esz, (int)N, sm_margin, di, &pl, res ? 2 : 1)) != RN_OK) return st;
  FwdParams p{};
  p.x = x;
  p.gamma = gamma;
  p.beta = beta;
  p.out = out->data;
  p.mu = mu;
  p.rsigma = rsigma;
  p.scale = out->scale;
  p.amax = out->amax;
  p.scale_inv = out->scale_inv;
  p.scale_out = out->scale_out;
  p.N = (int)N;
  p.H = (int)H;
  p.eps = eps;
  p.zcg = zcg ? 1 : 0;
  p.out_f32 = (mode == RN_QUANT_NONE && out->out_dtype == RN_F32) ? 1 : 0;
  p.residual = residual;
  p.residual_out = residual_out;
  p.workers = pl.workers;
  p.Q = pl.Q;
  p.rps_log2 = pl.rps_log2;
  p.reverse = 0;
  // pass 1 (or the only pass): with a residual, the kernel that adds it
  auto first = [&](int qmode, bool pdl) {
    return res ? launch_fwd_res(nk, bf16, pl.sh, qmode, p, pl.l, pdl, stream)
               : launch_fwd(nk, bf16, pl.sh, qmode, p, pl.l, pdl, stream);
  };

  switch (mode) {
    case RN_QUANT_NONE:
      return first(kQNone, false);
    case RN_QUANT_FP8_DELAYED:
      if ((st = launch_fwd_init(out->amax, out->scale, out->scale_inv, stream)) != RN_OK) return st;
      return first(kQDelayed, true);
    case RN_QUANT_FP8_CURRENT: {
      if ((st = launch_fwd_init(out->amax, nullptr, nullptr, stream)) != RN_OK) return st;
      if ((st = first(kQCurAmax, true)) != RN_OK) return st;
      // pass 2 normalizes the stored sum h (with a residual) or x again
      FwdPlan p2 = pl;
      if (res && (st = plan_fwd(nk, (int)H, esz, (int)N, sm_margin, di, &p2, 1)) != RN_OK) return st;
      FwdParams q = p;
      if (res) q.x = residual_out;
      q.residual = nullptr;
      q.residual_out = nullptr;
      q.workers = p2.workers;
      q.Q = p2.Q;
      q.rps_log2 = p2.rps_log2;
      q.reverse = 1;
      return launch_fwd(nk, bf16, p2.sh, kQCurQuant, q, p2.l, true, stream);
    }
    case RN_QUANT_NVFP4: {
      // the same two passes; pass 2 needs room for its factor table
      if ((st = launch_fwd_init(out->amax, nullptr, nullptr, stream)) != RN_OK) return st;
      if ((st = first(kQCurAmax, true)) != RN_OK) return st;
      FwdPlan p2;
      if ((st = plan_fwd(nk, (int)H, esz, (int)N, sm_margin, di, &p2, 1, kNvTableBytes)) != RN_OK)
        return st;
      FwdParams q = p;
      if (res) q.x = residual_out;
      q.residual = nullptr;
      q.residual_out = nullptr;
      q.scales = out->row_scales;
      q.workers = p2.workers;
      q.Q = p2.Q;
      q.rps_log2 = p2.rps_log2;
      q.reverse = 1;
      return launch_fwd(nk, bf16, p2.sh, kQNvfp4, q, p2.l, true, stream);
    }
    default:
      return RN_ERR_INVALID;
  }
}

// ---------------------------------------------------------------- backward
rn_status bwd_common(bool ln, const void* dz, const void* x, rn_dtype dt, const float* mu,
                     const float* rsigma, const float* gamma, int64_t N, int64_t H, int zcg,
                     int sm_margin, void* dx, float* dgamma, float* dbeta, void* ws,
                     size_t* ws_bytes, cudaStream_t stream) {
  if (!dtype_ok(dt) || N < 0 || H < 1 || N > INT32_MAX || H > INT32_MAX) return RN_ERR_INVALID;
  BwdShape sh;
  rn_status st;
  if (!row_ok(H, dt)) return RN_ERR_UNSUPPORTED;
  if ((st = bwd_shape(N, H, elem_size(dt), &sh)) != RN_OK) return st;
  const size_t need = bwd_workspace(sh, H, ln);
  if (ws == nullptr) {
    if (ws_bytes == nullptr) return RN_ERR_INVALID;
    *ws_bytes = need;
    return RN_OK;
  }
  // with N == 0 the row tensors are empty and may be NULL
  if (((dz == nullptr || x == nullptr || rsigma == nullptr || dx == nullptr) && N > 0) ||
      gamma == nullptr || dgamma == nullptr)
    return RN_ERR_INVALID;
  if (ln && ((mu == nullptr && N > 0) || dbeta == nullptr)) return RN_ERR_INVALID;
  if (ws_bytes == nullptr || *ws_bytes < need) return RN_ERR_WORKSPACE;
  if (!aligned(dz, 16) || !aligned(x, 16) || !aligned(dx, 16) || !aligned(ws, 16) ||
      !aligned(gamma, 4) || !aligned(rsigma, 4) || (mu && !aligned(mu, 4)) ||
      !aligned(dgamma, 4) || (dbeta && !aligned(dbeta, 4)))
    return RN_ERR_UNSUPPORTED;
  DeviceInfo di;
  if ((st = device_info(&di)) != RN_OK) return st;
  if ((st = check_margin(sm_margin, di)) != RN_OK) return st;
  if (N == 0) {
    if (cudaMemsetAsync(dgamma, 0, H * sizeof(float), stream) != cudaSuccess) return RN_ERR_CUDA;
    if (ln && cudaMemsetAsync(dbeta, 0, H * sizeof(float), stream) != cudaSuccess)
      return RN_ERR_CUDA;
    return RN_OK;
  }
  const int esz = elem_size(dt);
  const size_t row_bytes = (size_t)H * esz;
  const int nch = (int)(H * esz / 16);
  BwdParams p{};
  p.dz = dz;
  p.x = x;
  p.mu = mu;
  p.rsigma = rsigma;
  p.gamma = gamma;
  p.dx = dx;
  p.part = static_cast<float*>(ws);
  p.N = (int)N;
  p.H = (int)H;
  p.zcg = zcg ? 1 : 0;
  p.chunk_rows = sh.chunk_rows;
  p.n_chunks = sh.n_chunks;
  Launch l;
  l.work = sh.n_chunks;
  l.sms = di.sms - sm_margin;

  // fp32 rows that 16 warps cover with 16 elements (4 chunks) a thread take
  // the kernel without stats or producer warps: A warps, up to 8 with as
  // many CTAs per SM (<= 4) as keep a ring of >= 6 slots and 128 registers a
  // thread, else one CTA per SM with up to 16.  (bf16 rows stay with the
  // stats-warp kernel: with its more warps per SM it is the faster of the
  // two there, 44.5 vs 47.3 us for 8192 x 4096.)  per slot: the x and dz
  // rows, (mu, rsigma), an mbarrier; fixed: the warp-sum exchange (2 x 16
  // float2) + slack.
  const int ngf = 4;
  const int Af = (nch + 32 * ngf - 1) / (32 * ngf);
  if (dt == RN_F32 && Af <= 16) {
    const size_t per_slot = 2 * row_bytes + sizeof(float2) + 8;
    const size_t fixed = 32 * sizeof(float2) + 64;
    const bool big = Af > 8;
    int per_sm = 0, Q = 0;
    for (int k = big ? 1 : 4; k >= 1 && per_sm == 0; --k) {
      if (k * 32 * Af > 512 && k > 1) continue;
      const size_t b = cta_smem_budget(di, k);
      int q = b > fixed ? (int)((b - fixed) / per_slot) : 0;
      if (q > 64) q = 64;
      if (q >= (k > 1 ? 6 : 3)) {
        per_sm = k;
        Q = q;
      }
    }
    if (per_sm == 0) return RN_ERR_UNSUPPORTED;
    p.apply_warps = Af;
    p.stats_warps = 0;
    p.Q = Q;
    l.threads = 32 * Af;
    l.smem = (size_t)Q * per_slot + fixed;
    l.per_sm = per_sm;
    if ((st = launch_bwd_fused(ln, big, p, l, stream)) != RN_OK) return st;
  } else {
    // longer rows: stats warps + apply warps (roles as in plan_roles).
    // fixed: g [H] (as float4 parts of each chunk) + slack; per slot: the x
    // and dz rows, (mu, rsigma) as loaded, (mu, rsigma, c1, c2), three
    // mbarriers.
    const size_t fixed = (size_t)H * sizeof(float) + 64;
    const size_t per_slot = 2 * row_bytes + sizeof(float2) + sizeof(float4) + 24;
    Roles ro;
    if ((st = plan_roles(nch, ln, per_slot, fixed, di, 64, &ro)) != RN_OK) return st;
    p.apply_warps = ro.A;
    p.stats_warps = ro.S;
    p.Q = ro.Q;
    l.threads = 32 * (ro.A + ro.S + 1);
    l.smem = (size_t)ro.Q * per_slot + fixed;
    l.per_sm = ro.per_sm;
    if (ro.per_sm == 1) {
      // one CTA per SM: chunks of R = max(R_N, ceil(N / (k SMs))) rows with
      // k = 3 or 2 chunks a CTA at sm_margin 0, whichever leaves the
      // busiest CTA fewer rows (3 on a tie), so that the CTAs hold
      // near-equal rows, with fewer partials.  8192 x 4096 LayerNorm: 456
      // chunks of 18 rows, 35.9 against 39.2 us with 1024 of 8 (sm_margin
      // 16: 42.8 against 41.6 us; 2 a CTA: 34.9 / 45.1 us, 4: 37.0 / 42.9,
      // 6: 38.8 / 41.3); 3000 x 5120: 300 chunks of 10 rows, LayerNorm 24.7
      // against 27.1 us, RMSNorm 22.7 against 24.8 us (sm_margin 16: 28.7
      // against 26.8, 26.4 against 24.0 us).  R depends on N and the
      // device, never on sm_margin, and is never below R_N, so the
      // workspace the query reports (for R_N) covers it.
      int64_t R = 0, busiest = -1;
      for (int k = kBwdWideChunksPerCta; k >= 2; --k) {
        const int64_t per = (int64_t)k * di.sms;
        int64_t r = (N + per - 1) / per;
        if (r < sh.chunk_rows) r = sh.chunk_rows;
        const int64_t rows = ((N + r - 1) / r + di.sms - 1) / di.sms * r;
        if (busiest < 0 || rows < busiest) {
          busiest = rows;
          R = r;
        }
      }
      p.chunk_rows = (int)R;
      p.n_chunks = (int)((N + R - 1) / R);
      l.work = p.n_chunks;
    }
    if ((st = launch_bwd(ln, dt == RN_BF16, ro.ng, p, l, stream)) != RN_OK) return st;
  }
  ColReduceParams c{};
  c.part = p.part;
  c.dgamma = dgamma;
  c.dbeta = dbeta;
  c.H = (int)H;
  c.n_chunks = p.n_chunks;
  c.nacc = ln ? 2 : 1;
  return launch_colreduce(c, stream);
}

}  // namespace
}  // namespace rn

using namespace rn;

extern "C" {

rn_status rn_layernorm_fwd(const void* x, rn_dtype x_dtype, const float* gamma, const float* beta,
                           int64_t N, int64_t H, float eps, int zero_centered_gamma, int sm_margin,
                           rn_quant_mode mode, const rn_output* out, float* mu, float* rsigma,
                           void* stream) {
  return fwd_common(kLn, x, x_dtype, gamma, beta, N, H, eps, zero_centered_gamma, sm_margin, mode,
                    out, mu, rsigma, static_cast<cudaStream_t>(stream));
}

rn_status rn_rmsnorm_fwd(const void* x, rn_dtype x_dtype, const float* gamma, int64_t N, int64_t H,
                         float eps, int zero_centered_gamma, int sm_margin, rn_quant_mode mode,
                         const rn_output* out, float* rsigma, void* stream) {
  return fwd_common(kRms, x, x_dtype, gamma, nullptr, N, H, eps, zero_centered_gamma, sm_margin,
                    mode, out, nullptr, rsigma, static_cast<cudaStream_t>(stream));
}

rn_status rn_layernorm_add_fwd(const void* x, const void* residual, rn_dtype dtype,
                               const float* gamma, const float* beta, int64_t N, int64_t H,
                               float eps, int zero_centered_gamma, int sm_margin,
                               rn_quant_mode mode, const rn_output* out, void* residual_out,
                               float* mu, float* rsigma, void* stream) {
  return fwd_common(kLn, x, dtype, gamma, beta, N, H, eps, zero_centered_gamma, sm_margin, mode,
                    out, mu, rsigma, static_cast<cudaStream_t>(stream), true, residual,
                    residual_out);
}

rn_status rn_rmsnorm_add_fwd(const void* x, const void* residual, rn_dtype dtype,
                             const float* gamma, int64_t N, int64_t H, float eps,
                             int zero_centered_gamma, int sm_margin, rn_quant_mode mode,
                             const rn_output* out, void* residual_out, float* rsigma,
                             void* stream) {
  return fwd_common(kRms, x, dtype, gamma, nullptr, N, H, eps, zero_centered_gamma, sm_margin,
                    mode, out, nullptr, rsigma, static_cast<cudaStream_t>(stream), true, residual,
                    residual_out);
}

rn_status rn_layernorm_bwd(const void* dz, const void* x, rn_dtype dtype, const float* mu,
                           const float* rsigma, const float* gamma, int64_t N, int64_t H,
                           int zero_centered_gamma, int sm_margin, void* dx, float* dgamma,
                           float* dbeta, void* workspace, size_t* workspace_bytes, void* stream) {
  return bwd_common(true, dz, x, dtype, mu, rsigma, gamma, N, H, zero_centered_gamma, sm_margin, dx,
                    dgamma, dbeta, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

rn_status rn_rmsnorm_bwd(const void* dz, const void* x, rn_dtype dtype, const float* rsigma,
                         const float* gamma, int64_t N, int64_t H, int zero_centered_gamma,
                         int sm_margin, void* dx, float* dgamma, void* workspace,
                         size_t* workspace_bytes, void* stream) {
  return bwd_common(false, dz, x, dtype, nullptr, rsigma, gamma, N, H, zero_centered_gamma,
                    sm_margin, dx, dgamma, nullptr, workspace, workspace_bytes,
                    static_cast<cudaStream_t>(stream));
}

rn_status rn_delayed_scaling_update(float* amax_history, int64_t history_len, const float* amax,
                                    float* scale, float* scale_inv, void* stream) {
  if (amax_history == nullptr || amax == nullptr || scale == nullptr || scale_inv == nullptr ||
      history_len < 1)
    return RN_ERR_INVALID;
  if (history_len > kMaxHistory) return RN_ERR_UNSUPPORTED;
  if (!aligned(amax_history, 4) || !aligned(amax, 4) || !aligned(scale, 4) || !aligned(scale_inv, 4))
    return RN_ERR_UNSUPPORTED;
  return launch_amax_history(amax_history, (int)history_len, amax, scale, scale_inv,
                             static_cast<cudaStream_t>(stream));
}

rn_status rn_quantize_only(const float* y, int64_t N, int64_t H, rn_quant_mode mode,
                           const rn_output* out, void* stream) {
  if (mode != RN_QUANT_FP8_DELAYED && mode != RN_QUANT_FP8_CURRENT && mode != RN_QUANT_MXFP8 &&
      mode != RN_QUANT_NVFP4)
    return RN_ERR_INVALID;
  return fwd_common(kIdentity, y, RN_F32, nullptr, nullptr, N, H, 0.0f, 0, 0, mode, out, nullptr,
                    nullptr, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------ scaled activations
static rn_status act_common_checks(rn_act act, const void* x, rn_dtype dt, const float* scales,
                                   int64_t N, int64_t H, float limit, float alpha) {
  if (act != RN_ACT_SRELU && act != RN_ACT_SWIGLU && act != RN_ACT_CLAMPED_SWIGLU)
    return RN_ERR_INVALID;
  if ((x == nullptr && N > 0) || !dtype_ok(dt) || N < 0 || H < 1 || N > INT32_MAX ||
      H > INT32_MAX / 2)
    return RN_ERR_INVALID;
  if (act == RN_ACT_CLAMPED_SWIGLU && (!(limit >= 0.0f) || !(alpha == alpha) ||
                                       alpha > 3.4e38f || alpha < -3.4e38f))
    return RN_ERR_INVALID;
  if (!row_ok(H, dt) || !aligned(x, 16) || (scales && !aligned(scales, 4)))
    return RN_ERR_UNSUPPORTED;
  return RN_OK;
}

rn_status rn_scaled_act_fwd(rn_act act, const void* x, rn_dtype dtype, const float* scales,
                            int64_t N, int64_t H, float limit, float alpha, rn_quant_mode mode,
                            const rn_output* out, void* stream) {
  rn_status st = act_common_checks(act, x, dtype, scales, N, H, limit, alpha);
  if (st != RN_OK) return st;
  if (mode == RN_QUANT_NVFP4) return RN_ERR_UNSUPPORTED;
  if (mode == RN_QUANT_MXFP8 && out != nullptr &&
      (out->col_data != nullptr || out->col_scales != nullptr))
    return RN_ERR_UNSUPPORTED;  // rowwise blocks only
  if (mode == RN_QUANT_MXFP8) {
    if (out == nullptr) return RN_ERR_INVALID;
    if (N > 0 && !out_fields_only(out, true, true, false, false, false, false, false, false))
      return RN_ERR_INVALID;
    if (H % 32 != 0) return RN_ERR_UNSUPPORTED;
    if (N > 0 && !aligned(out->data, 16)) return RN_ERR_UNSUPPORTED;
  } else if ((st = check_out(mode, out, N, H)) != RN_OK) {
    return st;
  }
  DeviceInfo di;
  if ((st = device_info(&di)) != RN_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0 && (mode == RN_QUANT_NONE || mode == RN_QUANT_MXFP8)) return RN_OK;
  ActParams p{};
  p.x = x;
  p.out = out->data;
  p.row_scales = mode == RN_QUANT_MXFP8 ? out->row_scales : nullptr;
  p.scales = scales;
  p.scale = out->scale;
  p.amax = out->amax;
  p.scale_inv = out->scale_inv;
  p.scale_out = out->scale_out;
  p.N = (int)N;
  p.H = (int)H;
  p.limit = limit;
  p.alpha = alpha;
  p.out_f32 = (mode == RN_QUANT_NONE && out->out_dtype == RN_F32) ? 1 : 0;
  const bool bf16 = dtype == RN_BF16;
  switch (mode) {
    case RN_QUANT_NONE:
    case RN_QUANT_MXFP8:
      return launch_act_fwd(act, bf16, kQNone, p, di.sms, false, s);
    case RN_QUANT_FP8_DELAYED:
      if ((st = launch_fwd_init(out->amax, out->scale, out->scale_inv, s)) != RN_OK) return st;
      return launch_act_fwd(act, bf16, kQDelayed, p, di.sms, true, s);
    case RN_QUANT_FP8_CURRENT:
      if ((st = launch_fwd_init(out->amax, nullptr, nullptr, s)) != RN_OK) return st;
      if ((st = launch_act_fwd(act, bf16, kQCurAmax, p, di.sms, true, s)) != RN_OK) return st;
      return launch_act_fwd(act, bf16, kQCurQuant, p, di.sms, true, s);
    default:
      return RN_ERR_INVALID;
  }
}

rn_status rn_scaled_act_bwd(rn_act act, const void* dy, const void* x, rn_dtype dtype,
                            const float* scales, int64_t N, int64_t H, float limit, float alpha,
                            void* dx, float* dscales, void* stream) {
  rn_status st = act_common_checks(act, x, dtype, scales, N, H, limit, alpha);
  if (st != RN_OK) return st;
  if (N > 0 && (dy == nullptr || dx == nullptr)) return RN_ERR_INVALID;
  if ((dy && !aligned(dy, 16)) || (dx && !aligned(dx, 16)) || (dscales && !aligned(dscales, 4)))
    return RN_ERR_UNSUPPORTED;
  DeviceInfo di;
  if ((st = device_info(&di)) != RN_OK) return st;
  if (N == 0) return RN_OK;
  ActParams p{};
  p.x = x;
  p.dy = dy;
  p.out = dx;
  p.scales = scales;
  p.dscales = dscales;
  p.N = (int)N;
  p.H = (int)H;
  p.limit = limit;
  p.alpha = alpha;
  return launch_act_bwd(act, dtype == RN_BF16, p, di.sms, static_cast<cudaStream_t>(stream));
}

const char* rn_status_str(rn_status s) {
  switch (s) {
    case RN_OK: return "ok";
    case RN_ERR_INVALID: return "invalid argument";
    case RN_ERR_UNSUPPORTED: return "unsupported shape, dtype or alignment";
    case RN_ERR_WORKSPACE: return "workspace missing or too small";
    case RN_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

rn_status rn_device_error(unsigned int* code) {
  if (code == nullptr) return RN_ERR_INVALID;
  if (cudaDeviceSynchronize() != cudaSuccess) return RN_ERR_CUDA;
  unsigned a = 0, b = 0, c = 0;
  rn_status st;
  unsigned a2 = 0;
  if ((st = read_clear_error_fwd(&a)) != RN_OK) return st;
  if ((st = read_clear_error_fwd_res(&a2)) != RN_OK) return st;
  if (a == 0) a = a2;
  if ((st = read_clear_error_mx(&b)) != RN_OK) return st;
  if ((st = read_clear_error_bwd(&c)) != RN_OK) return st;
  *code = a ? a : (b ? b : c);
  return RN_OK;
}

int rn_abi_version(void) { return 1; }

}  // extern "C"

// ------------------------------------------ LayerNorm backward, no allocation
// rn_layernorm_bwd needs a caller-allocated workspace for its dgamma/dbeta
// partial sums.  Callers that cannot allocate device memory where they run
// the backward get rn_layernorm_bwd_noalloc instead: the partials live in a
// fixed array that is part of the library's device image.
namespace rn {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device

// Loaded with the library on every device that runs its kernels and held
// until the process exits.  Host code must not pass this symbol to a kernel:
// on the host it is only a stand-in; the device address comes from
// cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::atomic<void*> g_noalloc_addr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
rn_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return RN_ERR_UNSUPPORTED;
  void* p = g_noalloc_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return RN_ERR_CUDA;
    g_noalloc_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return RN_OK;
}

}  // namespace
}  // namespace rn

extern "C" rn_status rn_layernorm_bwd_noalloc(const void* dz, const void* x, rn_dtype dtype,
                                              const float* mu, const float* rsigma,
                                              const float* gamma, int64_t N, int64_t H,
                                              int zero_centered_gamma, int sm_margin, void* dx,
                                              float* dgamma, float* dbeta, void* stream) {
  size_t need = 0;
  rn_status st = bwd_common(true, nullptr, nullptr, dtype, nullptr, nullptr, nullptr, N, H, 0, 0,
                            nullptr, nullptr, nullptr, nullptr, &need, nullptr);
  if (st != RN_OK) return st;
  if (need > kNoAllocScratchBytes) return RN_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != RN_OK) return st;
  size_t cap = kNoAllocScratchBytes;
  return bwd_common(true, dz, x, dtype, mu, rsigma, gamma, N, H, zero_centered_gamma, sm_margin,
                    dx, dgamma, dbeta, scratch, &cap, static_cast<cudaStream_t>(stream));
}
