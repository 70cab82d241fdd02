// Internal host/device interface of the scan library (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ssd {

enum Variant { kMamba2 = 0, kMamba1 = 1, kMimo = 2 };

// Validated sizes of one problem.  All counts fit in int; element offsets are
// computed in size_t.
struct Dims {
  int variant;
  bool bf16;  // io dtype
  int b, T, H, P, N, G, L, R;
  int nc;   // T / L
  int LR;   // fused chunk length L * R
  int hpg;  // heads per group (Mamba-2)
  int rs = 0;  // tensor-core kernels on a MIMO problem: log2 R (their T is then the fused length T * R)
};

struct FwdArgs {
  const void* x;
  const float* dt_raw;
  const float* A;
  const void* B;
  const void* C;
  const float* s0;
  void* y;
  float* s_final;
  __nv_bfloat16* states_out = nullptr;  // tensor-core path: chunk states to this caller buffer, not the workspace
  float* ckpt_out = nullptr;            // tensor-core path: fp32 checkpoints every ckpt_every chunks
  int ckpt_every = 0;
};

struct BwdArgs {
  const void* dy;
  const float* ds_final;
  const void* x;
  const float* dt_raw;
  const float* A;
  const void* B;
  const void* C;
  const float* s0;
  void* dx;
  float* ddt_raw;
  float* dA;
  void* dB;
  void* dC;
  float* ds0;
  const __nv_bfloat16* states_in = nullptr;  // tensor-core path: stashed chunk states (no forward replay)
  const float* ckpt_in = nullptr;            // tensor-core path: replay in segments from these checkpoints
  int ckpt_every = 0;
};

// The first kStatusBytes of every workspace hold the device status word
// (int32 at offset 0): each call resets it to 0, and a kernel whose bounded
// wait gives up writes a nonzero code there.
constexpr size_t kStatusBytes = 256;

// Carves a caller-owned workspace into 256-byte aligned pieces after the
// status word.  The same code sizes the workspace (base == nullptr) and hands
// out the pointers.
struct Carver {
  char* base;
  size_t off = kStatusBytes;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    off = (off + 255) & ~size_t(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

// Chunked SIMT path (Mamba-2 and MIMO; fp32 arithmetic, fp32 or bf16 io).
size_t simt_forward_ws(const Dims& d);
size_t simt_backward_ws(const Dims& d);
cudaError_t simt_forward(const Dims& d, const FwdArgs& a, void* ws, cudaStream_t st);
cudaError_t simt_backward(const Dims& d, const BwdArgs& a, void* ws, cudaStream_t st);

// Tensor-core path (bf16 io, P = 64, N = 128): Mamba-2 with chunk 64, and MIMO
// with a power-of-two rank R <= 64 as a Mamba-2 scan over the fused sequence
// t * R + r (see tc_dims).
bool tc_forward_supported(const Dims& d);
// The sizes the tensor-core kernels run: the problem itself for Mamba-2; for
// MIMO the fused sequence of T * R positions in chunks of 64 (16 steps of R =
// 4), one group per head, and rs = log2 R.
Dims tc_dims(const Dims& d);
// Chunk-parallel forward (ssd_tc_fwdc.cu): the state scan, then every (chunk, head) output at once.
size_t tc_forward_ws(const Dims& d);
cudaError_t tc_forward(const Dims& d, const FwdArgs& a, void* ws, cudaStream_t st);
// Sequential state scans and the K2 tiles, in one launch (ssd_tc_scan.cu).
// The forward scan (u = x, with B) writes S_c for every chunk (bf16
// [b,H,nc][N][P]) and S_nc into fin (if not null); the reverse scan (u = dy,
// with C) writes dS_{c+1} for every chunk and dS_0 into fin.  init = s0 (may
// be null) or ds_final.  Either side may be absent (null); CB[b, c, g] =
// C B^T of every chunk and group (fp32) is always written.
// Forward side only: ckpt_out (not null) receives the fp32 state entering
// every `every`-th chunk, [b,H,nk][P][N] with nk = ceil(nc / every) (entry 0 =
// s0); with ckpt_in (not null) the forward scan runs as b*H*nk independent
// segments of `every` chunks, each started from its entry, and writes the same
// S_c tiles as the whole-sequence scan (init and fin unused).
struct ScanSide {
  const void* u;
  const float* init;
  float* fin;
  __nv_bfloat16* states;
  float* ckpt_out = nullptr;
  const float* ckpt_in = nullptr;
  int every = 0;
};
size_t tc_scan_states_bytes(const Dims& d);
size_t tc_checkpoints_bytes(const Dims& d, int every);
cudaError_t tc_scans(const Dims& d, const ScanSide* fwd, const ScanSide* rev, const void* B, const void* C,
                     const float* dt_raw, const float* A, float* CB, int* status, cudaStream_t st);
// Chunk-parallel backward (ssd_tc_bwdc.cu): both scans, then every (chunk, head) at once.
size_t tc_backward_ws(const Dims& d);
cudaError_t tc_backward(const Dims& d, const BwdArgs& a, void* ws, cudaStream_t st);
bool tc_backward_supported(const Dims& d);

// TMA tensor maps over bf16 tensors with 128-byte swizzle (tma_host.cu).
cudaError_t make_tmap_2d_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                              uint32_t box_outer);
cudaError_t make_tmap_3d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0,
                              uint32_t b1, uint32_t b2);
cudaError_t make_tmap_4d_bf16(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3,
                              uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3);
// The per-token tensors seen by the chunk tiles, with the sequence dimension
// kept apart from the batch: a tile of the last, partial chunk of a sequence
// (T not a multiple of 64) reads zeros past the sequence end and a store of
// it writes nothing there.
//   [b, T, width] bf16 (x, y, dy, dx with width = H*P): 64 x 64 boxes, coordinates (col, t, b);
//   [b, T, G, N] bf16 (B, C): 64 x 1 x 64 x 1 boxes, coordinates (n, g, t, b).
cudaError_t make_tmap_seq_bf16(CUtensorMap* m, const void* base, const Dims& d, uint64_t width);
cudaError_t make_tmap_bc_bf16(CUtensorMap* m, const void* base, const Dims& d);

// Mamba-1 path (fp32).
size_t m1_forward_ws(const Dims& d);
size_t m1_backward_ws(const Dims& d);
cudaError_t m1_forward(const Dims& d, const FwdArgs& a, void* ws, cudaStream_t st);
cudaError_t m1_backward(const Dims& d, const BwdArgs& a, void* ws, cudaStream_t st);

// Launches `kernel` with programmatic stream serialization: it may be scheduled
// while the previous kernel on `st` finishes, and must call pdl_wait() (the
// device side, tc_common.cuh) before it touches global memory.  Used for the
// second and later kernels of one call, whose prologue (barrier set-up, TMEM
// allocation) then overlaps the previous kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                         Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Per-launch event timing (see ssd_profile_start in ssd.h).  SSD_LAUNCH wraps
// every kernel launch of the library.
void prof_begin(const char* name, cudaStream_t st);
void prof_end(cudaStream_t st);

}  // namespace ssd

#define SSD_LAUNCH(name, st, ...)     \
  do {                                \
    ::ssd::prof_begin((name), (st));  \
    __VA_ARGS__;                      \
    ::ssd::prof_end((st));            \
  } while (0)
