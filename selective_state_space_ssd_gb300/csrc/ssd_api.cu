// C ABI of the scan library: argument validation, workspace sizing and
// dispatch to the kernels.  Validation completes before anything is enqueued;
// a call that returns an error has launched nothing.
#include <stdint.h>

#include <initializer_list>
#include <mutex>
#include <vector>

#include "../../include/ssd.h"
#include "ssd_internal.h"

namespace ssd {
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ssd_status make_dims(const ssd_problem* pr, Dims* d) {
  if (!pr) return SSD_ERR_INVALID_ARG;
  if (pr->variant < SSD_MAMBA2 || pr->variant > SSD_MIMO) return SSD_ERR_INVALID_ARG;
  if (pr->io_dtype != SSD_F32 && pr->io_dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
  if (pr->batch < 1 || pr->seqlen < 1 || pr->nheads < 1 || pr->headdim < 1 || pr->dstate < 1 || pr->chunk < 1 ||
      pr->mimo_rank < 1)
    return SSD_ERR_SHAPE;
  const int64_t kMax = (int64_t)1 << 30;
  if (pr->batch > kMax || pr->seqlen > kMax || pr->nheads > kMax) return SSD_ERR_SHAPE;
  d->variant = pr->variant;
  d->bf16 = pr->io_dtype == SSD_BF16;
  d->b = (int)pr->batch;
  d->T = (int)pr->seqlen;
  d->H = (int)pr->nheads;
  d->P = (int)pr->headdim;
  d->N = (int)pr->dstate;
  d->R = (int)pr->mimo_rank;
  if (pr->chunk > 256) return SSD_ERR_SHAPE;
  // nc chunks of `chunk` steps; the last holds the remaining T - (nc - 1) * chunk steps
  d->L = (int)pr->chunk;
  d->nc = (int)((pr->seqlen + pr->chunk - 1) / pr->chunk);
  switch (pr->variant) {
    case SSD_MAMBA2:
      if (pr->ngroups < 1 || pr->nheads % pr->ngroups != 0) return SSD_ERR_SHAPE;
      if (pr->mimo_rank != 1) return SSD_ERR_SHAPE;
      d->G = (int)pr->ngroups;
      break;
    case SSD_MIMO:
      d->G = d->H;  // B and C per head
      break;
    case SSD_MAMBA1:
      if (pr->headdim != 1 || pr->mimo_rank != 1) return SSD_ERR_SHAPE;
      if (pr->dstate > 32) return SSD_ERR_SHAPE;
      if (pr->io_dtype != SSD_F32) return SSD_ERR_DTYPE;
      d->G = 1;
      break;
  }
  if (pr->variant != SSD_MAMBA1) {
    if (pr->headdim > 256 || pr->dstate > 256) return SSD_ERR_SHAPE;
    if (pr->chunk * pr->mimo_rank > 256) return SSD_ERR_SHAPE;
  }
  d->LR = d->L * d->R;
  d->hpg = d->H / d->G;
  // element counts of the largest tensors must fit in int32 indexing of a dimension
  const double big = (double)pr->batch * pr->seqlen * pr->nheads * pr->mimo_rank *
                     (double)(pr->headdim > pr->dstate ? pr->headdim : pr->dstate);
  if (big > 4.0e12) return SSD_ERR_SHAPE;
  return SSD_OK;
}

size_t ws_bytes(const Dims& d, bool backward) {
  if (d.variant == kMamba1) return backward ? m1_backward_ws(d) : m1_forward_ws(d);
  if (!backward && tc_forward_supported(d)) return tc_forward_ws(d);
  if (backward && tc_backward_supported(d)) return tc_backward_ws(d);
  return backward ? simt_backward_ws(d) : simt_forward_ws(d);
}

ssd_status check_ptrs(std::initializer_list<const void*> required, std::initializer_list<const void*> optional) {
  for (const void* p : required) {
    if (!p) return SSD_ERR_INVALID_ARG;
    if (!aligned16(p)) return SSD_ERR_ALIGNMENT;
  }
  for (const void* p : optional)
    if (p && !aligned16(p)) return SSD_ERR_ALIGNMENT;
  return SSD_OK;
}

struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};

std::mutex g_prof_mu;
bool g_prof_on = false;
int g_prof_cap = 0;
std::vector<ProfRec> g_prof;
thread_local int t_prof_open = -1;  // record opened by this thread's last prof_begin

// Validation shared by the checkpoint calls: the problem, then 1 <= every <= 2^30 (SSD_ERR_INVALID_ARG),
// then the tensor-core Mamba-2 path (SSD_ERR_SHAPE otherwise).
ssd_status checkpoint_dims(const ssd_problem* prob, int64_t every, Dims* d) {
  ssd_status s = make_dims(prob, d);
  if (s != SSD_OK) return s;
  if (every < 1 || every > (int64_t)1 << 30) return SSD_ERR_INVALID_ARG;
  if (d->variant != kMamba2 || !tc_forward_supported(*d)) return SSD_ERR_SHAPE;
  return SSD_OK;
}

}  // namespace

void prof_begin(const char* name, cudaStream_t st) {
  t_prof_open = -1;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on || (int)g_prof.size() >= g_prof_cap) return;
  ProfRec r{name, nullptr, nullptr};
  if (cudaEventCreate(&r.a) != cudaSuccess) return;
  if (cudaEventCreate(&r.b) != cudaSuccess) {
    cudaEventDestroy(r.a);
    return;
  }
  cudaEventRecord(r.a, st);
  g_prof.push_back(r);
  t_prof_open = (int)g_prof.size() - 1;
}

void prof_end(cudaStream_t st) {
  if (t_prof_open < 0) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (t_prof_open < (int)g_prof.size()) cudaEventRecord(g_prof[t_prof_open].b, st);
  t_prof_open = -1;
}

}  // namespace ssd

using namespace ssd;

extern "C" {

int ssd_version(void) { return 100; }

ssd_status ssd_profile_start(int capacity) {
  if (capacity < 1) return SSD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = true;
  g_prof_cap = capacity;
  return SSD_OK;
}

ssd_status ssd_profile_stop(ssd_kernel_time* out, int capacity, int* count) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = false;
  ssd_status st = SSD_OK;
  int n = 0;
  for (size_t i = 0; i < g_prof.size(); ++i) {
    ProfRec& r = g_prof[i];
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
      st = SSD_ERR_CUDA;
    if (out && n < capacity) out[n++] = ssd_kernel_time{r.name, ms};
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  g_prof.clear();
  if (count) *count = n;
  return st;
}

const char* ssd_status_string(ssd_status s) {
  switch (s) {
    case SSD_OK: return "SSD_OK";
    case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG: missing buffer or unknown enum value";
    case SSD_ERR_SHAPE: return "SSD_ERR_SHAPE: sizes not allowed (H % G, limits of this build)";
    case SSD_ERR_DTYPE: return "SSD_ERR_DTYPE: io dtype not supported for this variant";
    case SSD_ERR_ALIGNMENT: return "SSD_ERR_ALIGNMENT: a pointer is not 16-byte aligned";
    case SSD_ERR_WORKSPACE: return "SSD_ERR_WORKSPACE: workspace smaller than ssd_workspace_size()";
    case SSD_ERR_CUDA: return "SSD_ERR_CUDA: a CUDA call or kernel launch failed";
    case SSD_ERR_TIMEOUT: return "SSD_ERR_TIMEOUT: a bounded device-side wait gave up";
    case SSD_ERR_INTERNAL: return "SSD_ERR_INTERNAL: device-side consistency check failed";
    case SSD_ERR_TOO_LARGE:
      return "SSD_ERR_TOO_LARGE: the problem needs more scratch than the fixed 32 MiB array of ssd_forward_static";
  }
  return "SSD_ERR_UNKNOWN";
}

ssd_status ssd_workspace_size(const ssd_problem* prob, int backward, size_t* bytes) {
  if (!bytes) return SSD_ERR_INVALID_ARG;
  Dims d;
  ssd_status s = make_dims(prob, &d);
  if (s != SSD_OK) return s;
  *bytes = ws_bytes(d, backward != 0);
  return SSD_OK;
}

ssd_status ssd_forward(const ssd_problem* prob, const void* x, const float* dt_raw, const float* A, const void* B,
                       const void* C, const float* s0, void* y, float* s_final, void* ws, size_t ws_bytes_given,
                       void* cuda_stream) {
  Dims d;
  ssd_status s = make_dims(prob, &d);
  if (s != SSD_OK) return s;
  if (d.variant == kMimo) {
    if (A) return SSD_ERR_INVALID_ARG;
    s = check_ptrs({x, dt_raw, B, C, y, s_final}, {s0});
  } else {
    s = check_ptrs({x, dt_raw, A, B, C, y, s_final}, {s0});
  }
  if (s != SSD_OK) return s;
  const size_t need = ws_bytes(d, false);
  if (ws_bytes_given < need) return SSD_ERR_WORKSPACE;
  if (!ws) return SSD_ERR_INVALID_ARG;
  if (!aligned16(ws)) return SSD_ERR_ALIGNMENT;
  FwdArgs a{x, dt_raw, A, B, C, s0, y, s_final};
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return SSD_ERR_CUDA;
  cudaError_t e = d.variant == kMamba1        ? m1_forward(d, a, ws, st)
                  : tc_forward_supported(d) ? tc_forward(d, a, ws, st)
                                            : simt_forward(d, a, ws, st);
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_backward(const ssd_problem* prob, const void* dy, const float* ds_final, const void* x,
                        const float* dt_raw, const float* A, const void* B, const void* C, const float* s0, void* dx,
                        float* ddt_raw, float* dA, void* dB, void* dC, float* ds0, void* ws, size_t ws_bytes_given,
                        void* cuda_stream) {
  Dims d;
  ssd_status s = make_dims(prob, &d);
  if (s != SSD_OK) return s;
  if (d.variant == kMimo) {
    if (A || dA) return SSD_ERR_INVALID_ARG;
    s = check_ptrs({dy, ds_final, x, dt_raw, B, C, dx, ddt_raw, dB, dC, ds0}, {s0});
  } else {
    s = check_ptrs({dy, ds_final, x, dt_raw, A, B, C, dx, ddt_raw, dA, dB, dC, ds0}, {s0});
  }
  if (s != SSD_OK) return s;
  const size_t need = ws_bytes(d, true);
  if (ws_bytes_given < need) return SSD_ERR_WORKSPACE;
  if (!ws) return SSD_ERR_INVALID_ARG;
  if (!aligned16(ws)) return SSD_ERR_ALIGNMENT;
  BwdArgs a{dy, ds_final, x, dt_raw, A, B, C, s0, dx, ddt_raw, dA, dB, dC, ds0};
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return SSD_ERR_CUDA;
  cudaError_t e = d.variant == kMamba1         ? m1_backward(d, a, ws, st)
                  : tc_backward_supported(d) ? tc_backward(d, a, ws, st)
                                             : simt_backward(d, a, ws, st);
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_states_size(const ssd_problem* prob, size_t* bytes) {
  if (!bytes) return SSD_ERR_INVALID_ARG;
  Dims d;
  ssd_status s = make_dims(prob, &d);
  if (s != SSD_OK) return s;
  if (d.variant != kMamba2 || !tc_forward_supported(d)) return SSD_ERR_SHAPE;
  *bytes = tc_scan_states_bytes(d);
  return SSD_OK;
}

ssd_status ssd_forward_stash(const ssd_problem* prob, const void* x, const float* dt_raw, const float* A,
                             const void* B, const void* C, const float* s0, void* y, float* s_final, void* states,
                             size_t states_bytes, void* ws, size_t ws_bytes_given, void* cuda_stream) {
  Dims d;
  ssd_status s = make_dims(prob, &d);
  if (s != SSD_OK) return s;
  if (d.variant != kMamba2 || !tc_forward_supported(d)) return SSD_ERR_SHAPE;
  s = check_ptrs({x, dt_raw, A, B, C, y, s_final, states}, {s0});
  if (s != SSD_OK) return s;
  if (states_bytes < tc_scan_states_bytes(d) || ws_bytes_given < ws_bytes(d, false)) return SSD_ERR_WORKSPACE;
  if (!ws) return SSD_ERR_INVALID_ARG;
  if (!aligned16(ws)) return SSD_ERR_ALIGNMENT;
  FwdArgs a{x, dt_raw, A, B, C, s0, y, s_final, static_cast<__nv_bfloat16*>(states)};
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return SSD_ERR_CUDA;
  return tc_forward(d, a, ws, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_backward_stashed(const ssd_problem* prob, const void* dy, const float* ds_final, const void* x,
                                const float* dt_raw, const float* A, const void* B, const void* C,
                                const void* states, size_t states_bytes, void* dx, float* ddt_raw, float* dA,
                                void* dB, void* dC, float* ds0, void* ws, size_t ws_bytes_given, void* cuda_stream) {
  Dims d;
  ssd_status s = make_dims(prob, &d);
  if (s != SSD_OK) return s;
  if (d.variant != kMamba2 || !tc_backward_supported(d)) return SSD_ERR_SHAPE;
  s = check_ptrs({dy, ds_final, x, dt_raw, A, B, C, states, dx, ddt_raw, dA, dB, dC, ds0}, {});
  if (s != SSD_OK) return s;
  if (states_bytes < tc_scan_states_bytes(d) || ws_bytes_given < ws_bytes(d, true)) return SSD_ERR_WORKSPACE;
  if (!ws) return SSD_ERR_INVALID_ARG;
  if (!aligned16(ws)) return SSD_ERR_ALIGNMENT;
  BwdArgs a{dy, ds_final, x, dt_raw, A, B, C, nullptr, dx, ddt_raw, dA, dB, dC, ds0,
            static_cast<const __nv_bfloat16*>(states)};
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return SSD_ERR_CUDA;
  return tc_backward(d, a, ws, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_checkpoints_size(const ssd_problem* prob, int64_t every, size_t* bytes) {
  if (!bytes) return SSD_ERR_INVALID_ARG;
  Dims d;
  ssd_status s = checkpoint_dims(prob, every, &d);
  if (s != SSD_OK) return s;
  *bytes = tc_checkpoints_bytes(d, (int)every);
  return SSD_OK;
}

ssd_status ssd_forward_checkpointed(const ssd_problem* prob, const void* x, const float* dt_raw, const float* A,
                                    const void* B, const void* C, const float* s0, void* y, float* s_final,
                                    int64_t every, float* ckpt, size_t ckpt_bytes, void* ws, size_t ws_bytes_given,
                                    void* cuda_stream) {
  Dims d;
  ssd_status s = checkpoint_dims(prob, every, &d);
  if (s != SSD_OK) return s;
  s = check_ptrs({x, dt_raw, A, B, C, y, s_final, ckpt}, {s0});
  if (s != SSD_OK) return s;
  if (ckpt_bytes < tc_checkpoints_bytes(d, (int)every) || ws_bytes_given < ws_bytes(d, false))
    return SSD_ERR_WORKSPACE;
  if (!ws) return SSD_ERR_INVALID_ARG;
  if (!aligned16(ws)) return SSD_ERR_ALIGNMENT;
  FwdArgs a{x, dt_raw, A, B, C, s0, y, s_final};
  a.ckpt_out = ckpt;
  a.ckpt_every = (int)every;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return SSD_ERR_CUDA;
  return tc_forward(d, a, ws, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_backward_checkpointed(const ssd_problem* prob, const void* dy, const float* ds_final, const void* x,
                                     const float* dt_raw, const float* A, const void* B, const void* C,
                                     int64_t every, const float* ckpt, size_t ckpt_bytes, void* dx, float* ddt_raw,
                                     float* dA, void* dB, void* dC, float* ds0, void* ws, size_t ws_bytes_given,
                                     void* cuda_stream) {
  Dims d;
  ssd_status s = checkpoint_dims(prob, every, &d);
  if (s != SSD_OK) return s;
  s = check_ptrs({dy, ds_final, x, dt_raw, A, B, C, ckpt, dx, ddt_raw, dA, dB, dC, ds0}, {});
  if (s != SSD_OK) return s;
  if (ckpt_bytes < tc_checkpoints_bytes(d, (int)every) || ws_bytes_given < ws_bytes(d, true))
    return SSD_ERR_WORKSPACE;
  if (!ws) return SSD_ERR_INVALID_ARG;
  if (!aligned16(ws)) return SSD_ERR_ALIGNMENT;
  BwdArgs a{dy, ds_final, x, dt_raw, A, B, C, nullptr, dx, ddt_raw, dA, dB, dC, ds0};
  a.ckpt_in = ckpt;
  a.ckpt_every = (int)every;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return SSD_ERR_CUDA;
  return tc_backward(d, a, ws, st) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
