// Mamba-1 branch (one decay per state), fp32.  One lane per (batch, channel,
// state): the recurrence s_t[n] = exp(dt'_t A[d,n]) s_{t-1}[n] + dt'_t x_t B_t[n]
// runs serially in t on that lane, and y_t = sum_n s_t[n] C_t[n] is a shuffle
// reduction over the W >= N lanes of the channel ("S1-31: SSM_SCAN_BACK —
// Mamba has a backward", opening paragraph: the Mamba-1 branch has one decay
// per state).
//
// The backward replays the forward, keeping the state at the start of every
// segment of K = chunk steps, then walks the segments in reverse: each is
// replayed from its checkpoint into shared memory and walked backwards,
// carrying dS from the ds_final seed (the same page, "Two things that are
// easy to get wrong": the nonzero seed, and s_{t-1} recomputed for d(dt)).
// dB and dC (shared by every channel) are written per channel and then summed
// over channels in ascending order; dA over batches in ascending order.
#include "ssd_device.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kM1Threads = 128;

struct M1 {
  const float *x, *dt, *A, *B, *C, *s0;
  int b, T, D, N, W, K;  // W: lanes per channel (power of two >= N, <= 32)
};

__device__ __forceinline__ float group_sum(float v, int W) {
  for (int o = W >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o, W);
  return v;
}

__global__ void __launch_bounds__(kM1Threads) k_m1_forward(M1 m, float* y, float* s_final) {
  const int lane = threadIdx.x % m.W;
  const long unit = ((long)blockIdx.x * blockDim.x + threadIdx.x) / m.W;
  const bool valid = unit < (long)m.b * m.D;
  const bool act = valid && lane < m.N;
  const int bb = valid ? (int)(unit / m.D) : 0, d = valid ? (int)(unit % m.D) : 0;
  const float a_n = act ? m.A[(size_t)d * m.N + lane] : 0.f;
  float s = (act && m.s0) ? m.s0[((size_t)bb * m.D + d) * m.N + lane] : 0.f;
  for (int t = 0; t < m.T; ++t) {
    const size_t td = ((size_t)bb * m.T + t) * m.D + d;
    const size_t tn = ((size_t)bb * m.T + t) * m.N + lane;
    const float dtp = valid ? softplus_f(m.dt[td]) : 0.f;
    const float xv = valid ? m.x[td] : 0.f;
    if (act) s = expf(dtp * a_n) * s + dtp * xv * m.B[tn];
    const float yv = group_sum(act ? s * m.C[tn] : 0.f, m.W);
    if (valid && lane == 0) y[td] = yv;
  }
  if (act) s_final[((size_t)bb * m.D + d) * m.N + lane] = s;
}

// Per lane: checkpoints ck[unit][seg][n]; parts dB/dC [b,T,D,N]; dA part [b,D,N].
__global__ void __launch_bounds__(kM1Threads)
    k_m1_backward(M1 m, const float* dy, const float* ds_final, float* ck, float* dx, float* ddt_raw,
                  float* dB_part, float* dC_part, float* dA_part, float* ds0) {
  extern __shared__ float seg_states[];  // [(K+1)][blockDim.x]
  const int lane = threadIdx.x % m.W;
  const long unit = ((long)blockIdx.x * blockDim.x + threadIdx.x) / m.W;
  const bool valid = unit < (long)m.b * m.D;
  const bool act = valid && lane < m.N;
  const int bb = valid ? (int)(unit / m.D) : 0, d = valid ? (int)(unit % m.D) : 0;
  const float a_n = act ? m.A[(size_t)d * m.N + lane] : 0.f;
  const int nseg = (m.T + m.K - 1) / m.K;  // the last segment may be shorter (T not a multiple of K)
  const size_t ck_base = ((size_t)unit * nseg) * m.N + lane;
  // forward replay: the state entering each segment
  float s = (act && m.s0) ? m.s0[((size_t)bb * m.D + d) * m.N + lane] : 0.f;
  for (int k = 0; k < nseg; ++k) {
    if (act) ck[ck_base + (size_t)k * m.N] = s;
    const int len = min(m.K, m.T - k * m.K);
    for (int j = 0; j < len; ++j) {
      const int t = k * m.K + j;
      const size_t td = ((size_t)bb * m.T + t) * m.D + d;
      if (act) {
        const float dtp = softplus_f(m.dt[td]);
        s = expf(dtp * a_n) * s + dtp * m.x[td] * m.B[((size_t)bb * m.T + t) * m.N + lane];
      }
    }
  }
  float dS = act ? ds_final[((size_t)bb * m.D + d) * m.N + lane] : 0.f;
  float dA_acc = 0.f;
  float* mine = seg_states + threadIdx.x;
  const int stride = blockDim.x;
  for (int k = nseg - 1; k >= 0; --k) {
    float r = act ? ck[ck_base + (size_t)k * m.N] : 0.f;
    mine[0] = r;
    const int len = min(m.K, m.T - k * m.K);
    for (int j = 0; j < len; ++j) {
      const int t = k * m.K + j;
      const size_t td = ((size_t)bb * m.T + t) * m.D + d;
      if (act) {
        const float dtp = softplus_f(m.dt[td]);
        r = expf(dtp * a_n) * r + dtp * m.x[td] * m.B[((size_t)bb * m.T + t) * m.N + lane];
      }
      mine[(j + 1) * stride] = r;
    }
    for (int j = len - 1; j >= 0; --j) {
      const int t = k * m.K + j;
      const size_t td = ((size_t)bb * m.T + t) * m.D + d;
      const size_t tn = ((size_t)bb * m.T + t) * m.N + lane;
      const float z = valid ? m.dt[td] : 0.f;
      const float dtp = softplus_f(z);
      const float xv = valid ? m.x[td] : 0.f;
      const float dyv = valid ? dy[td] : 0.f;
      const float Bn = act ? m.B[tn] : 0.f;
      const float Cn = act ? m.C[tn] : 0.f;
      const float s_cur = mine[(j + 1) * stride], s_prev = mine[j * stride];
      const float a = act ? expf(dtp * a_n) : 0.f;
      dS += dyv * Cn;                                   // y_t = s_t . C_t
      const size_t part = (((size_t)bb * m.T + t) * m.D + d) * m.N + lane;
      if (act) dC_part[part] = dyv * s_cur;
      const float u = group_sum(dS * Bn, m.W);          // d(dt' x) direction
      if (act) dB_part[part] = dtp * xv * dS;
      const float dda = a * dS * s_prev;                // the decay path
      dA_acc += dtp * dda;
      const float dd = u * xv + group_sum(a_n * dda, m.W);
      if (valid && lane == 0) {
        dx[td] = dtp * u;
        ddt_raw[td] = dd * sigmoid_f(z);
      }
      dS *= a;
    }
  }
  if (act) {
    ds0[((size_t)bb * m.D + d) * m.N + lane] = dS;
    dA_part[((size_t)bb * m.D + d) * m.N + lane] = dA_acc;
  }
}

// out[b,t,n] = sum over channels d (ascending) of part[b,t,d,n].
__global__ void k_m1_channel_sum(const float* part, float* out, int b, int T, int D, int N) {
  const size_t total = (size_t)b * T * N;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const size_t bt = e / N;
    const int n = e % N;
    float acc = 0.f;
    for (int d = 0; d < D; ++d) acc += part[(bt * D + d) * N + n];
    out[e] = acc;
  }
}

__global__ void k_m1_dA_sum(const float* part, float* dA, int b, int DN) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= DN) return;
  float acc = 0.f;
  for (int bb = 0; bb < b; ++bb) acc += part[(size_t)bb * DN + i];
  dA[i] = acc;
}

int lanes_for(int N) {
  int w = 1;
  while (w < N) w <<= 1;
  return w;
}

M1 make_m1(const Dims& d, const void* x, const float* dt, const float* A, const void* B, const void* C,
           const float* s0) {
  M1 m;
  m.x = static_cast<const float*>(x);
  m.dt = dt;
  m.A = A;
  m.B = static_cast<const float*>(B);
  m.C = static_cast<const float*>(C);
  m.s0 = s0;
  m.b = d.b; m.T = d.T; m.D = d.H; m.N = d.N; m.W = lanes_for(d.N); m.K = d.L;
  return m;
}

struct M1Ws {
  float *ck, *dB_part, *dC_part, *dA_part;
};

M1Ws carve_m1(const Dims& d, Carver& cv) {
  M1Ws w;
  const size_t units = (size_t)d.b * d.H;
  w.ck = cv.take<float>(units * d.nc * d.N);
  w.dB_part = cv.take<float>((size_t)d.b * d.T * d.H * d.N);
  w.dC_part = cv.take<float>((size_t)d.b * d.T * d.H * d.N);
  w.dA_part = cv.take<float>((size_t)d.b * d.H * d.N);
  return w;
}

}  // namespace

size_t m1_forward_ws(const Dims&) { return kStatusBytes; }

size_t m1_backward_ws(const Dims& d) {
  Carver cv(nullptr);
  carve_m1(d, cv);
  return cv.off;
}

cudaError_t m1_forward(const Dims& d, const FwdArgs& a, void*, cudaStream_t st) {
  M1 m = make_m1(d, a.x, a.dt_raw, a.A, a.B, a.C, a.s0);
  const long lanes = (long)d.b * d.H * m.W;
  const int blocks = (int)((lanes + kM1Threads - 1) / kM1Threads);
  SSD_LAUNCH("k_m1_forward", st,
             k_m1_forward<<<blocks, kM1Threads, 0, st>>>(m, static_cast<float*>(a.y), a.s_final));
  return cudaGetLastError();
}

cudaError_t m1_backward(const Dims& d, const BwdArgs& a, void* ws, cudaStream_t st) {
  Carver cv(ws);
  M1Ws w = carve_m1(d, cv);
  M1 m = make_m1(d, a.x, a.dt_raw, a.A, a.B, a.C, a.s0);
  const long lanes = (long)d.b * d.H * m.W;
  const int blocks = (int)((lanes + kM1Threads - 1) / kM1Threads);
  const size_t smem = (size_t)(m.K + 1) * kM1Threads * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k_m1_backward, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  SSD_LAUNCH("k_m1_backward", st,
             k_m1_backward<<<blocks, kM1Threads, smem, st>>>(m, static_cast<const float*>(a.dy), a.ds_final, w.ck,
                                                  static_cast<float*>(a.dx), a.ddt_raw, w.dB_part, w.dC_part,
                                                  w.dA_part, a.ds0));
  const size_t tot = (size_t)d.b * d.T * d.N;
  const int rb = (int)((tot + 255) / 256 < 65535 ? (tot + 255) / 256 : 65535);
  SSD_LAUNCH("k_m1_channel_sum", st,
             k_m1_channel_sum<<<rb, 256, 0, st>>>(w.dB_part, static_cast<float*>(a.dB), d.b, d.T, d.H, d.N));
  SSD_LAUNCH("k_m1_channel_sum", st,
             k_m1_channel_sum<<<rb, 256, 0, st>>>(w.dC_part, static_cast<float*>(a.dC), d.b, d.T, d.H, d.N));
  SSD_LAUNCH("k_m1_dA_sum", st,
             k_m1_dA_sum<<<(d.H * d.N + 255) / 256, 256, 0, st>>>(w.dA_part, a.dA, d.b, d.H * d.N));
  return cudaGetLastError();
}

}  // namespace ssd
