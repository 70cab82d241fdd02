// The device status word, read from the host, and a self-test of the bounded
// waits that set it.
//
// Every wait of the tensor-core kernels on an mbarrier or a named barrier is
// bounded: when it runs out, the kernel writes a nonzero code into the status
// word (the first 4 bytes of the call's workspace, or of the fixed scratch of
// ssd_forward_static), stops issuing work and returns, so the context stays
// usable and the host learns of it by reading the word.  ssd_wait_selftest
// makes one such wait run out on purpose: one thread waits on an mbarrier that
// nothing ever arrives on, with a short limit the caller picks.  No copy, MMA
// or TMEM allocation is in flight when it gives up.
#include <stdint.h>

#include "../../include/ssd.h"
#include "ssd_internal.h"
#include "tc_common.cuh"

namespace ssd {
namespace {

constexpr int kSelftestCode = 1;

__global__ void __launch_bounds__(32) k_wait_selftest(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t never;  // initialised for one arrival, which never comes
  if (threadIdx.x == 0) {
    tc::mbar_init(&never, 1);
    tc::mbar_init_fence();
  }
  __syncwarp();
  if (threadIdx.x == 0) tc::mbar_wait_loop(&never, 0, status, kSelftestCode, limit_ns);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ssd_status read_word(const void* word, int32_t* code, cudaStream_t st) {
  if (cudaMemcpyAsync(code, word, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess) return SSD_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return SSD_ERR_CUDA;
  return *code == 0 ? SSD_OK : SSD_ERR_TIMEOUT;
}

}  // namespace
}  // namespace ssd

extern "C" {

ssd_status ssd_read_status(const void* ws, int32_t* code, void* cuda_stream) {
  if (!ws || !code) return SSD_ERR_INVALID_ARG;
  return ssd::read_word(ws, code, static_cast<cudaStream_t>(cuda_stream));
}

ssd_status ssd_wait_selftest(void* ws, uint32_t limit_us, void* cuda_stream) {
  if (!ws) return SSD_ERR_INVALID_ARG;
  if (limit_us < 1 || limit_us > 2000000u) return SSD_ERR_INVALID_ARG;
  if (!ssd::aligned16(ws)) return SSD_ERR_ALIGNMENT;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return SSD_ERR_CUDA;
  ssd::k_wait_selftest<<<1, 32, 0, st>>>(static_cast<int*>(ws), 1000ull * limit_us);
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
