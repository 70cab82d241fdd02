// Host-side creation of TMA tensor maps (128-byte swizzled bf16 tiles).  The
// driver's cuTensorMapEncodeTiled is reached through the runtime's
// entry-point query, so the library does not link libcuda directly.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "ssd_internal.h"

namespace ssd {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

cudaError_t encode(CUtensorMap* m, const void* base, cuuint32_t rank, const cuuint64_t* dims,
                   const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides_bytes, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t make_tmap_2d_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                              uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  return encode(m, base, 2, dims, strides, box);
}

cudaError_t make_tmap_3d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0,
                              uint32_t b1, uint32_t b2) {
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {b0, b1, b2};
  return encode(m, base, 3, dims, strides, box);
}

cudaError_t make_tmap_4d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3,
                              uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  const cuuint64_t dims[4] = {d0, d1, d2, d3};
  const cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
  const cuuint32_t box[4] = {b0, b1, b2, b3};
  return encode(m, base, 4, dims, strides, box);
}

cudaError_t make_tmap_seq_bf16(CUtensorMap* m, const void* base, const Dims& d, uint64_t width) {
  return make_tmap_3d_bf16(m, base, width, (uint64_t)d.T, (uint64_t)d.b, 64, 64, 1);
}

cudaError_t make_tmap_bc_bf16(CUtensorMap* m, const void* base, const Dims& d) {
  return make_tmap_4d_bf16(m, base, (uint64_t)d.N, (uint64_t)d.G, (uint64_t)d.T, (uint64_t)d.b, 64, 1, 64, 1);
}

}  // namespace ssd
