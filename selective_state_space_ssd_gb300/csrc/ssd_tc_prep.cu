// Pieces shared by the tensor-core forward and backward: the K2 pre-pass
// (C B^T per chunk and group, fp32) and the shapes the tcgen05 kernels serve.
#include "ssd_device.cuh"
#include "ssd_internal.h"
#include "tc_common.cuh"

namespace ssd {
namespace {
using namespace tc;

constexpr int kL = 64, kN = 128;

// CB[b][c][g][t][s] = sum_n C[b, c*L+t, g, n] B[b, c*L+s, g, n]  (fp32), on the
// tensor cores: one CTA per (chunk, group) loads the C and B tiles with TMA
// (two 64-column atoms each, K-major), issues the eight K = 16 steps of one
// M = 64, N = 64 MMA, and its four warps write the accumulator rows out.
struct alignas(1024) CbSmem {
  uint8_t C[2][kL * 64 * 2];  // [atom][t][64 n] bf16, SW128
  uint8_t B[2][kL * 64 * 2];  // [atom][s][64 n]
  uint64_t full, done;
  uint32_t tmem_slot;
};

__global__ void __launch_bounds__(128) k_cb(const __grid_constant__ CUtensorMap tm_c,
                                            const __grid_constant__ CUtensorMap tm_b, float* __restrict__ CB, int T,
                                            int G, int nc, int* status) {
  extern __shared__ uint8_t smem_raw[];
  CbSmem& sm = *reinterpret_cast<CbSmem*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5;
  const long long k = blockIdx.x;  // (b * nc + c) * G + g
  const int g = (int)(k % G);
  const long long bc = k / G;
  const int c = (int)(bc % nc), b = (int)(bc / nc);
  const int row = b * T + c * kL;
  if (tid == 0) {
    mbar_init(&sm.full, 1);
    mbar_init(&sm.done, 1);
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(&sm.tmem_slot, 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  if (tid == 0) {
    mbar_expect_tx(&sm.full, 4 * kL * 64 * 2);
    for (int a = 0; a < 2; ++a) {
      tma_load_3d(sm.C[a], &tm_c, 64 * a, g, row, &sm.full);
      tma_load_3d(sm.B[a], &tm_b, 64 * a, g, row, &sm.full);
    }
    if (mbar_wait(&sm.full, 0, status, 61)) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kN; kk += 16)
        mma_bf16(tmem, kdesc(sm.C[0], kL, kk), kdesc(sm.B[0], kL, kk), idesc_bf16(64, 64, false, false), kk > 0);
    }
    mma_commit(&sm.done);
  }
  __syncwarp();
  const bool ok = mbar_wait(&sm.done, 0, status, 62);
  tc_fence_after();
  if (ok && *status == 0) {
    // M = 64 accumulator: row t = 16 warp + (lane & 15) in lane 32 warp + (lane & 15); lanes 16-31 take columns 32-63
    const int lane = tid & 31, t = 16 * warp + (lane & 15), s0 = 32 * (lane >> 4);
    uint32_t v[32];
    tmem_ld_pair32(taddr(tmem, 32 * warp, 0), v);
    tmem_wait_ld();
    float4* out = reinterpret_cast<float4*>(CB + ((size_t)k * kL + t) * kL + s0);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      out[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]), __uint_as_float(v[4 * e + 2]),
                           __uint_as_float(v[4 * e + 3]));
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

}  // namespace

// The tensor-core kernels serve Mamba-2 with bf16 io, chunk 64, head dim 64
// and state 128 (the 130M and 2.7B layer shapes); everything else runs on the
// CUDA-core kernels.  Their (chunk, head) items are indexed with 32-bit integers.
bool tc_forward_supported(const Dims& d) {
  return d.variant == kMamba2 && d.bf16 && d.L == kL && d.P == 64 && d.N == kN &&
         (long long)d.b * d.nc * d.H < (1ll << 31) && d.b <= 65535 && d.G <= 65535;
}
bool tc_backward_supported(const Dims& d) { return tc_forward_supported(d); }

cudaError_t tc_cb_prepass(const Dims& d, const void* B, const void* C, float* CB, int* status, cudaStream_t st) {
  const uint64_t rows = (uint64_t)d.b * d.T;
  CUtensorMap tb, tcm;
  cudaError_t e = make_tmap_3d_bf16(&tb, B, d.N, d.G, rows, 64, 1, 64);
  if (e == cudaSuccess) e = make_tmap_3d_bf16(&tcm, C, d.N, d.G, rows, 64, 1, 64);
  if (e != cudaSuccess) return e;
  const long long nchunks = (long long)d.b * d.nc * d.G;
  if (nchunks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  const int smem = (int)sizeof(CbSmem) + 1024;
  e = cudaFuncSetAttribute(k_cb, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  SSD_LAUNCH("k_cb", st, k_cb<<<(unsigned)nchunks, 128, smem, st>>>(tcm, tb, CB, d.T, d.G, d.nc, status));
  return cudaGetLastError();
}

}  // namespace ssd
