// ssd_forward_static: the forward scan for callers that must not allocate
// device memory.  Instead of a caller-provided workspace it uses one fixed,
// file-scope device array as its scratch.
#include <stdint.h>

#include "../../include/ssd.h"
#include "ssd_internal.h"

namespace ssd {
namespace {

// The scratch array.  Every GPU that loads this library's module holds it
// until the process exits; its size is the hard limit on the workspace of the
// problems this entry point accepts.
constexpr size_t kStaticScratchBytes = (size_t)32 << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of the array on the current device.  In host code the symbol
// g_static_scratch is only a host-side stand-in, so the address a kernel may
// use comes from cudaGetSymbolAddress with that device current.  It is looked
// up on every call (no cache that a device reset or a new context would leave
// stale); once the module is loaded on the device the lookup allocates
// nothing.
ssd_status static_scratch_ptr(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return SSD_ERR_CUDA;
  *out = p;
  return SSD_OK;
}

}  // namespace
}  // namespace ssd

extern "C" {

ssd_status ssd_forward_static(const ssd_problem* prob, const void* x, const float* dt_raw, const float* A,
                              const void* B, const void* C, const float* s0, void* y, float* s_final,
                              void* cuda_stream) {
  size_t need = 0;
  ssd_status s = ssd_workspace_size(prob, 0, &need);
  if (s != SSD_OK) return s;
  if (need > ssd::kStaticScratchBytes) return SSD_ERR_TOO_LARGE;
  void* scratch = nullptr;
  s = ssd::static_scratch_ptr(&scratch);
  if (s != SSD_OK) return s;
  // The same validation, kernels and status-word reset as ssd_forward; only
  // the scratch differs.
  return ssd_forward(prob, x, dt_raw, A, B, C, s0, y, s_final, scratch, ssd::kStaticScratchBytes, cuda_stream);
}

ssd_status ssd_forward_static_status(int32_t* code, void* cuda_stream) {
  void* scratch = nullptr;
  ssd_status s = ssd::static_scratch_ptr(&scratch);
  if (s != SSD_OK || !code) return s;
  if (cudaMemcpyAsync(code, scratch, sizeof(int32_t), cudaMemcpyDeviceToHost, static_cast<cudaStream_t>(cuda_stream)) !=
          cudaSuccess ||
      cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
    return SSD_ERR_CUDA;
  return *code == 0 ? SSD_OK : SSD_ERR_TIMEOUT;
}

}  // extern "C"
