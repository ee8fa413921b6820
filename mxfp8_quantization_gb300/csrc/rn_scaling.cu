// Delayed-scaling recipe step: the bookkeeping that closes the loop around
// the delayed-scaling FP8 forward (page "Implementation:NVIDIA
// TransformerEngine PyTorch Ext Normalization", section "Description": FP8
// output with a scale chosen from earlier steps).  The history keeps the most
// recent amax at index 0; a step shifts it by one place and puts the new amax
// first; the next scale is fp32(448 / max(history)) by one IEEE division,
// unless that maximum is 0 or not finite (then the previous scale is kept);
// scale_inv = fp32(1 / scale).
//
// One CTA: every thread holds one history entry; the old entries are staged
// in shared memory before any is rewritten; the maximum is a block reduction
// with NaN winning.
#include <cuda_runtime.h>

#include "rn_device.cuh"
#include "rn_internal.h"

namespace rn {
namespace {

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

__global__ void __launch_bounds__(kMaxHistory) rn_amax_history_kernel(float* hist, int L,
                                                                        const float* amax,
                                                                        float* scale,
                                                                        float* scale_inv) {
  __shared__ float old[kMaxHistory];
  __shared__ float wmax[kMaxHistory / 32];
  const int t = threadIdx.x;
  if (t < L) old[t] = hist[t];
  __syncthreads();
  float v = 0.0f;
  if (t < L) {
    v = (t == 0) ? *amax : old[t - 1];
    hist[t] = v;
  }
  float m = v;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((t & 31) == 0) wmax[t >> 5] = m;
  __syncthreads();
  if (t == 0) {
    float mm = wmax[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) mm = max_nan(mm, wmax[w]);
    // keep the previous scale when the maximum is 0, negative or not finite
    const bool usable = mm > 0.0f && mm <= 3.402823466e38f;
    const float s = usable ? __fdiv_rn(448.0f, mm) : *scale;
    *scale = s;
    *scale_inv = __fdiv_rn(1.0f, s);
  }
}

}  // namespace

rn_status launch_amax_history(float* hist, int L, const float* amax, float* scale,
                              float* scale_inv, cudaStream_t s) {
  const int threads = (L + 31) / 32 * 32;
  rn_amax_history_kernel<<<1, threads, 0, s>>>(hist, L, amax, scale, scale_inv);
  return cudaGetLastError() == cudaSuccess ? RN_OK : RN_ERR_CUDA;
}

}  // namespace rn
