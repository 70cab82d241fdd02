// Device helpers shared by the scan kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssd {

__device__ __forceinline__ float ld(const float* p, size_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p, size_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st(float* p, size_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st(__nv_bfloat16* p, size_t i, float v) { p[i] = __float2bfloat16_rn(v); }

// dt' = softplus(z) = max(z, 0) + log1p(exp(-|z|)), no threshold.
__device__ __forceinline__ float softplus_f(float z) { return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z))); }

// d softplus / dz = sigmoid(z), evaluated without overflow for either sign.
__device__ __forceinline__ float sigmoid_f(float z) {
  const float e = expf(-fabsf(z));
  return z >= 0.f ? 1.f / (1.f + e) : e / (1.f + e);
}

// The same two functions on the approximate hardware exp2 / log2 units, for the
// bf16 tensor-core kernels: a few instructions each instead of the inlined
// accurate versions, which keeps the warp-specialized kernels' code (and their
// instruction-cache footprint) small.  Relative error about 1e-6 over the
// range the scan meets, far inside the bf16 path's tolerance.
__device__ __forceinline__ float softplus_fast(float z) { return fmaxf(z, 0.f) + __logf(1.f + __expf(-fabsf(z))); }
__device__ __forceinline__ float sigmoid_fast(float z) { return __fdividef(1.f, 1.f + __expf(-z)); }

// Deterministic block-wide sum: fixed shuffle tree inside each warp, then the
// warp totals added in warp order by thread 0.  `red` holds >= 32 floats.
// Every thread of the block must call it; the result is valid in thread 0.
__device__ __forceinline__ float block_sum_t0(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float tot = 0.f;
  if (threadIdx.x == 0)
    for (int i = 0; i < nw; ++i) tot += red[i];
  return tot;
}

}  // namespace ssd
