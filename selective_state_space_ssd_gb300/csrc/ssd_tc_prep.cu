// Pieces shared by the tensor-core forward and backward: the K2 pre-pass
// (C B^T per chunk and group, fp32) and the shapes the tcgen05 kernels serve.
#include "ssd_device.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kL = 64, kN = 128;

// CB[b][c][g][t][s] = sum_n C[b, c*L+t, g, n] B[b, c*L+s, g, n]  (fp32)
__global__ void __launch_bounds__(256) k_cb(const __nv_bfloat16* B, const __nv_bfloat16* C, float* CB, int T, int G,
                                            int nc) {
  __shared__ float sC[kL][kN + 1];
  __shared__ float sB[kL][kN + 1];
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  for (int e = threadIdx.x; e < kL * kN; e += blockDim.x) {
    const int t = e / kN, n = e % kN;
    const size_t gi = (((size_t)b * T + c * kL + t) * G + g) * kN + n;
    sC[t][n] = __bfloat162float(C[gi]);
    sB[t][n] = __bfloat162float(B[gi]);
  }
  __syncthreads();
  const int t = threadIdx.x >> 2, s0 = threadIdx.x & 3;
  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.f;
  for (int n = 0; n < kN; ++n) {
    const float cv = sC[t][n];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] += cv * sB[s0 + 4 * j][n];
  }
  float* out = CB + ((((size_t)b * nc + c) * G + g) * kL + t) * kL;
#pragma unroll
  for (int j = 0; j < 16; ++j) out[s0 + 4 * j] = acc[j];
}

}  // namespace

// The tensor-core kernels serve Mamba-2 with bf16 io, chunk 64, head dim 64
// and state 128 (the 130M and 2.7B layer shapes); everything else runs on the
// CUDA-core kernels.  Their (chunk, head) items are indexed with 32-bit integers.
bool tc_forward_supported(const Dims& d) {
  return d.variant == kMamba2 && d.bf16 && d.L == kL && d.P == 64 && d.N == kN &&
         (long long)d.b * d.nc * d.H < (1ll << 31);
}
bool tc_backward_supported(const Dims& d) { return tc_forward_supported(d); }

cudaError_t tc_cb_prepass(const Dims& d, const void* B, const void* C, float* CB, cudaStream_t st) {
  SSD_LAUNCH("k_cb", st,
             k_cb<<<dim3(d.nc, d.G, d.b), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(B),
                                                        static_cast<const __nv_bfloat16*>(C), CB, d.T, d.G, d.nc));
  return cudaGetLastError();
}

}  // namespace ssd
