// Device-side building blocks shared by the normalization kernels:
// mbarrier + bulk-copy (TMA engine, non-tensor form) pipeline primitives with
// bounded waits, numeric conversions (bf16, E4M3, E8M0) and reductions.
//
// Every wait here has a time limit: on expiry the kernel records an error
// code in its translation unit's device error word and carries on, so that a
// logic error can never hang the GPU.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rn {

// error codes recorded in the device error word
enum : unsigned {
  kErrFullWait = 1,    // an apply warp gave up waiting for a row to land
  kErrEmptyWait = 2,   // the producer gave up waiting for a slot to free
  kErrDrainWait = 3,   // the producer gave up waiting for its last copies
  kErrReadyWait = 4,   // an apply warp gave up waiting for a row's statistics
  kErrStatsWait = 5,   // a stats warp gave up waiting for a row to land
};

// wait limit in SM clock cycles (about 4 s at 1 GHz, 2 s at 2 GHz); the
// per-SM cycle counter is monotonic, unlike a wall-clock timer
constexpr long long kWaitLimitCycles = 4000000000ll;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// `count` arrivals at once
__device__ __forceinline__ void mbar_arrive_cnt(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// One bounded test of a phase: the thread may sleep until the phase
// completes or about kSuspendHintNs pass, so that waiting costs few issue
// slots.
constexpr uint32_t kSuspendHintNs = 20000;

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Wait until the phase with `parity` of barrier `bar` has completed, for at
// most kWaitLimitCycles; on expiry record `code` in *err and return false.
// Once an error is recorded (checked only after kErrorCheckCycles of
// waiting, so that the spin itself touches no global memory), later waits
// give up too, so a kernel that lost its pipeline finishes quickly (its
// results are then meaningless; the host reads the error word).
constexpr long long kErrorCheckCycles = 100000;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned* err,
                                          unsigned code) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    const long long dt = clock64() - t0;
    if (dt > kErrorCheckCycles &&
        (dt > kWaitLimitCycles || *reinterpret_cast<volatile unsigned*>(err) != 0u)) {
      atomicCAS(err, 0u, code);
      return false;
    }
  }
  return true;
}

// A slot ticket: a shared-memory word the producer of a ring sets to the
// use number of a slot (st.release) just before it refills the slot, which it
// does only once the slot's previous use was released.  A consumer that finds
// ticket == its use (ld.acquire) knows every earlier use of the slot has
// completed, so the parity wait on the slot's "full" barrier that follows
// cannot match an older phase, however far ahead of the slot the consumer
// is.  Bounded like mbar_wait.
__device__ __forceinline__ void ticket_set(uint32_t addr, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ticket_get(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ bool ticket_wait(uint32_t addr, uint32_t want, unsigned* err,
                                            unsigned code) {
  if (ticket_get(addr) == want) return true;
  const long long t0 = clock64();
  while (ticket_get(addr) != want) {
    __nanosleep(32);
    const long long dt = clock64() - t0;
    if (dt > kErrorCheckCycles &&
        (dt > kWaitLimitCycles || *reinterpret_cast<volatile unsigned*>(err) != 0u)) {
      atomicCAS(err, 0u, code);
      return false;
    }
  }
  return true;
}

// One contiguous global -> shared copy by the bulk-copy engine; completion
// is signalled on `bar` as `bytes` transaction bytes.  dst, src 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// L2 eviction-priority policies (createpolicy), used as cache hints
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// bulk copy as bulk_g2s, with an L2 cache-eviction hint for the source
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// 16-byte global store with an L2 cache-eviction hint
__device__ __forceinline__ void st_hint_f4(float* p, float4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w), "l"(pol)
               : "memory");
}

// 8-byte global load with an L2 cache-eviction hint
__device__ __forceinline__ float2 ld_hint_f2(const float* p, uint64_t pol) {
  float2 v;
  asm volatile("ld.global.L2::cache_hint.v2.f32 {%0, %1}, [%2], %3;" : "=f"(v.x), "=f"(v.y) : "l"(p), "l"(pol));
  return v;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel of its stream still
// runs; griddepcontrol.wait blocks until that kernel has completed and its
// memory operations are visible.  launch_dependents lets the next such
// kernel start before this one ends.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 4-byte asynchronous global -> shared copy (cp.async); completion is
// tracked by cp_async_arrive on an mbarrier
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// the barrier receives one arrival once every cp.async this thread issued
// so far has landed (the arrival is counted in the barrier's init count)
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Position in a ring of q slots: slot index and the parity of its use.
// Advancing by n <= q rows needs no division.
struct RingPos {
  uint32_t slot, phase;
  __device__ __forceinline__ void advance(uint32_t n, uint32_t q) {
    slot += n;
    if (slot >= q) {
      slot -= q;
      phase ^= 1u;
    }
  }
  // position k rows ahead (k < q)
  __device__ __forceinline__ RingPos ahead(uint32_t k, uint32_t q) const {
    RingPos r = *this;
    r.advance(k, q);
    return r;
  }
};

// named barrier over the consumer warps only (id 1; id 0 is __syncthreads)
__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// ------------------------------------------------------------ conversions
// 8 bf16 (one 16-byte chunk) -> fp32; exact.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void bf16x4_to_f32(const uint2& v, float* f) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xFFFF0000u);
}

// two fp32 -> packed bf16x2 (round to nearest even); lo in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// two fp32 -> two E4M3 codes (nearest even, saturating); lo in the low byte
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// four fp32 -> four E4M3 codes in one word, element 0 in the low byte (the
// two halves joined by the register move)
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// |v| as ordered bits: for non-negative floats and NaN the unsigned order of
// the bit patterns is the numeric order, with NaN above +inf.
__device__ __forceinline__ uint32_t abs_bits(float v) {
  return __float_as_uint(v) & 0x7FFFFFFFu;
}

// max that lets NaN win (max.NaN), on magnitudes
__device__ __forceinline__ float amax_acc(float acc, float v) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(acc), "f"(fabsf(v)));
  return r;
}

// E8M0 shared-scale code of a block with absolute maximum `amax`
// (OCP MX v1.0 rule for E4M3 elements): e = floor(log2 amax) - 8 clamped to
// [-127, 127], code = e + 127.  floor(log2) of a normal fp32 is its biased
// exponent field minus 127, so code = field - 8, clamped to [0, 254]; zero
// and subnormal amax give 0; NaN gives 0xFF; +inf (field 255) gives 247.
__device__ __forceinline__ uint32_t e8m0_code(float amax) {
  const uint32_t b = __float_as_uint(amax) & 0x7FFFFFFFu;
  if (b > 0x7F800000u) return 0xFFu;
  const int field = static_cast<int>(b >> 23);
  const int c = field - 8;
  return static_cast<uint32_t>(c < 0 ? 0 : c);
}

// 2^-e for an E8M0 code (e = code - 127), as the fp32 with exponent field
// 254 - code; codes 0..247 give normal values 2^127 .. 2^-120.  NaN code
// gives NaN so that the whole block quantizes to NaN.
__device__ __forceinline__ float e8m0_inv_scale(uint32_t code) {
  if (code == 0xFFu) return __uint_as_float(0x7FC00000u);
  return __uint_as_float((254u - code) << 23);
}

// ------------------------------------------------- packed fp32 pairs (f32x2)
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 splat2(float v) { return make_float2(v, v); }

// ------------------------------------- bf16 pairs with fp32 arithmetic
// A 32-bit word holds two bf16 values, element 0 in the low half.  The
// mixed-precision forms take the bf16 operands directly; every result is the
// same single-rounded fp32 value as converting first (bf16 -> fp32 is exact).

// exact fp32 values of the pair
__device__ __forceinline__ float2 bf16x2_f32(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// (x0 - m, x1 - m), each rounded once
__device__ __forceinline__ float2 bf16x2_sub(uint32_t w, float m) {
  float2 d;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "sub.rn.f32.bf16 %0, l, %3;\n\tsub.rn.f32.bf16 %1, h, %3;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "r"(w), "f"(m));
  return d;
}

// (x0 + c, x1 + c), each rounded once
__device__ __forceinline__ float2 bf16x2_add(uint32_t w, float c) {
  float2 d;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "add.rn.f32.bf16 %0, l, %3;\n\tadd.rn.f32.bf16 %1, h, %3;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "r"(w), "f"(c));
  return d;
}

// acc += (x0, x1)
__device__ __forceinline__ void bf16x2_acc(float2& acc, uint32_t w) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "add.rn.f32.bf16 %0, l, %0;\n\tadd.rn.f32.bf16 %1, h, %1;\n\t}"
      : "+f"(acc.x), "+f"(acc.y)
      : "r"(w));
}

// acc += (x0 * x0, x1 * x1)  (the products are exact in fp32)
__device__ __forceinline__ void bf16x2_sq_acc(float2& acc, uint32_t w) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "fma.rn.f32.bf16 %0, l, l, %0;\n\tfma.rn.f32.bf16 %1, h, h, %1;\n\t}"
      : "+f"(acc.x), "+f"(acc.y)
      : "r"(w));
}

// running maximum and minimum over two more values (3-input forms); NaN
// wins.  max|y| = max(hi, -lo) at the end.
__device__ __forceinline__ float max3(float acc, float2 v) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(acc), "f"(v.x), "f"(v.y));
  return r;
}
__device__ __forceinline__ float min3(float acc, float2 v) {
  float r;
  asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(acc), "f"(v.x), "f"(v.y));
  return r;
}

// running max of magnitudes over two more values; NaN wins
__device__ __forceinline__ float amax_acc2(float acc, float2 v) {
  float r;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(acc), "f"(fabsf(v.x)), "f"(fabsf(v.y)));
  return r;
}

// ------------------------------------------------------- row chunks
// A chunk is VEC consecutive elements of a row (VEC/2 pairs), loaded from
// shared memory with one vector load.
template <typename TIn, int VEC>
struct Vec;

template <>
struct Vec<uint16_t, 8> {  // bf16, 16 bytes
  static constexpr int PAIRS = 4;
  struct Raw {
    uint32_t w[4];
  };
  __device__ __forceinline__ static Raw load(const unsigned char* p, int c) {
    const uint4 v = *reinterpret_cast<const uint4*>(p + (size_t)c * 16);
    return Raw{{v.x, v.y, v.z, v.w}};
  }
  __device__ __forceinline__ static void store(unsigned char* p, int c, const Raw& r) {
    *reinterpret_cast<uint4*>(p + (size_t)c * 16) = make_uint4(r.w[0], r.w[1], r.w[2], r.w[3]);
  }
  // element-wise a + b, each rounded once to bf16 (nearest even)
  __device__ __forceinline__ static Raw add_rn(const Raw& a, const Raw& b) {
    Raw r;
#pragma unroll
    for (int i = 0; i < 4; ++i) asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r.w[i]) : "r"(a.w[i]), "r"(b.w[i]));
    return r;
  }
  __device__ __forceinline__ static float2 f32(const Raw& r, int i) { return bf16x2_f32(r.w[i]); }
  __device__ __forceinline__ static float2 sub(const Raw& r, int i, float m) {
    return bf16x2_sub(r.w[i], m);
  }
  __device__ __forceinline__ static float2 add(const Raw& r, int i, float c) {
    return bf16x2_add(r.w[i], c);
  }
  __device__ __forceinline__ static void acc(float2& a, const Raw& r, int i) { bf16x2_acc(a, r.w[i]); }
  __device__ __forceinline__ static void sq_acc(float2& a, const Raw& r, int i) {
    bf16x2_sq_acc(a, r.w[i]);
  }
};

template <>
struct Vec<uint16_t, 4> {  // bf16, 8 bytes
  static constexpr int PAIRS = 2;
  struct Raw {
    uint32_t w[2];
  };
  __device__ __forceinline__ static Raw load(const unsigned char* p, int c) {
    const uint2 v = *reinterpret_cast<const uint2*>(p + (size_t)c * 8);
    return Raw{{v.x, v.y}};
  }
  __device__ __forceinline__ static float2 f32(const Raw& r, int i) { return bf16x2_f32(r.w[i]); }
  __device__ __forceinline__ static float2 sub(const Raw& r, int i, float m) {
    return bf16x2_sub(r.w[i], m);
  }
  __device__ __forceinline__ static float2 add(const Raw& r, int i, float c) {
    return bf16x2_add(r.w[i], c);
  }
  __device__ __forceinline__ static void acc(float2& a, const Raw& r, int i) { bf16x2_acc(a, r.w[i]); }
  __device__ __forceinline__ static void sq_acc(float2& a, const Raw& r, int i) {
    bf16x2_sq_acc(a, r.w[i]);
  }
};

template <>
struct Vec<float, 4> {  // fp32, 16 bytes
  static constexpr int PAIRS = 2;
  struct Raw {
    float2 p[2];
  };
  __device__ __forceinline__ static Raw load(const unsigned char* p, int c) {
    const float4 v = *reinterpret_cast<const float4*>(p + (size_t)c * 16);
    return Raw{{make_float2(v.x, v.y), make_float2(v.z, v.w)}};
  }
  __device__ __forceinline__ static void store(unsigned char* p, int c, const Raw& r) {
    *reinterpret_cast<float4*>(p + (size_t)c * 16) = make_float4(r.p[0].x, r.p[0].y, r.p[1].x, r.p[1].y);
  }
  __device__ __forceinline__ static Raw add_rn(const Raw& a, const Raw& b) {
    return Raw{{add2(a.p[0], b.p[0]), add2(a.p[1], b.p[1])}};
  }
  __device__ __forceinline__ static float2 f32(const Raw& r, int i) { return r.p[i]; }
  __device__ __forceinline__ static float2 sub(const Raw& r, int i, float m) {
    return sub2(r.p[i], splat2(m));
  }
  __device__ __forceinline__ static float2 add(const Raw& r, int i, float c) {
    return add2(r.p[i], splat2(c));
  }
  __device__ __forceinline__ static void acc(float2& a, const Raw& r, int i) { a = add2(a, r.p[i]); }
  __device__ __forceinline__ static void sq_acc(float2& a, const Raw& r, int i) {
    a = fma2(r.p[i], r.p[i], a);
  }
};

template <>
struct Vec<float, 8> {  // fp32, 32 bytes
  static constexpr int PAIRS = 4;
  struct Raw {
    float2 p[4];
  };
  __device__ __forceinline__ static Raw load(const unsigned char* p, int c) {
    const float4* q = reinterpret_cast<const float4*>(p + (size_t)c * 32);
    const float4 a = q[0], b = q[1];
    return Raw{{make_float2(a.x, a.y), make_float2(a.z, a.w), make_float2(b.x, b.y),
                make_float2(b.z, b.w)}};
  }
  __device__ __forceinline__ static float2 f32(const Raw& r, int i) { return r.p[i]; }
  __device__ __forceinline__ static float2 sub(const Raw& r, int i, float m) {
    return sub2(r.p[i], splat2(m));
  }
  __device__ __forceinline__ static float2 add(const Raw& r, int i, float c) {
    return add2(r.p[i], splat2(c));
  }
  __device__ __forceinline__ static void acc(float2& a, const Raw& r, int i) { a = add2(a, r.p[i]); }
  __device__ __forceinline__ static void sq_acc(float2& a, const Raw& r, int i) {
    a = fma2(r.p[i], r.p[i], a);
  }
};

// ------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

__device__ __forceinline__ uint32_t warp_umax(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

}  // namespace rn
