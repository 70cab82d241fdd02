// Mamba-1 branch (one decay per state), fp32 ("S1-31: SSM_SCAN_BACK — Mamba
// has a backward", opening paragraph: the Mamba-1 branch has one decay per
// state).  Per (batch, channel d, state n):
//     s_t[n] = exp(dt'_t A[d,n]) s_{t-1}[n] + dt'_t x_t B_t[n],   y_t = sum_n s_t[n] C_t[n],
// a serial recurrence in t with no chunkwise shortcut (the decay differs per
// state), so the work is laid out for latency and issue: one thread carries
// kS = 4 states of one channel (the step's shared-memory loads and the lane
// shuffles of a channel serve four states; with two a thread both kernels were
// issue-bound), the Wc threads of a channel are adjacent lanes (y and the other
// sums over n are Wc-lane shuffles), and a block of 128 threads holds cpb =
// 128 / Wc consecutive channels of one sequence.  The block walks the sequence
// in chunks (32 steps in the forward and the backward's replay, 8 in its
// reverse walk) whose inputs (x, dt, dy for its channels; B, C of the step)
// are staged in shared memory by cp.async kStages - 1 chunks ahead, so a step
// reads shared memory only.
//
// The backward replays the forward once to keep the state entering every
// chunk (a checkpoint in global memory), then walks the chunks in reverse:
// each is replayed from its checkpoint into registers (the states of its 8
// steps; the walk recomputes each decay, with the same bits, rather than keep
// 32 of them in registers) and walked backwards, carrying dS from the ds_final seed (the
// same page, "Two things that are easy to get wrong": the nonzero seed, and
// s_{t-1} recomputed for d(dt)).  dB_t and dC_t are sums over every channel:
// each block adds its channels in ascending order in shared memory and writes
// one partial per (step, state); a second kernel adds the blocks' partials in
// ascending order.  dA adds the batches in ascending order.
//
// Steps past the end of the sequence (a partial last chunk) are staged as
// dt_raw = -inf and x = dy = B = C = 0: dt' = 0, so they leave the state as it
// is and add nothing; nothing is stored for them.
#include "ssd_device.cuh"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kThreads = 128;
constexpr int kS = 4;        // states per thread
constexpr int kTcF = 32;     // steps per chunk, forward
constexpr int kTc = 8;       // steps per chunk, backward (its replay keeps a chunk's states in registers)
constexpr int kStages = 3;   // chunk buffers: the one in use and two in flight
constexpr float kLog2e = 1.4426950408889634f;

// exp(dp * A) as 2^(dp * A2) with A2 = A log2(e) formed once per state, on the
// hardware's approximate exp2 (ex2.approx.ftz: relative error about 2^-22; the
// decays lie in (2^-8, 1], far from the flushed subnormals).  The exponent's
// rounding adds a relative error below 1e-6 over the arguments the scan meets
// (|dp A| <= 5), far inside the fp32 path's 1e-4 bound, for two instructions
// instead of an accurate expf or the subnormal-safe exp2f.
__device__ __forceinline__ float decay(float dp, float A2) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(dp * A2));
  return r;
}

struct M1 {
  const float *x, *dt, *A, *B, *C, *s0;
  int b, T, D, N;
  int Wc;    // threads per channel: the power of two >= ceil(N / kS) (the kernels' template argument)
  int nblk;  // channel blocks per sequence: ceil(D / (kThreads / Wc))
  int nck;   // backward chunks: ceil(T / kTc)
  int nckf;  // forward chunks: ceil(T / kTcF)
};

__device__ __forceinline__ void cp_async4(float* smem, const float* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// the group of the chunk about to be used has landed (kStages - 1 younger groups may still be in flight)
__device__ __forceinline__ void cp_async_wait_stages() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kStages - 1) : "memory");
}

template <int kWc>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = kWc >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o, kWc);
  return v;
}

// Block geometry for kWc threads per channel: cpb channels, NP states per channel as laid out.
template <int kWc>
struct Geo {
  static constexpr int cpb = kThreads / kWc, NP = kS * kWc;
};

// kS consecutive floats of shared memory (16-byte aligned)
__device__ __forceinline__ void ldsk(const float* p, float (&v)[kS]) {
  const float4 w = *reinterpret_cast<const float4*>(p);
  v[0] = w.x;
  v[1] = w.y;
  v[2] = w.z;
  v[3] = w.w;
}
__device__ __forceinline__ void stsk(float* p, const float (&v)[kS]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}

// One chunk's inputs in shared memory: per step t of the chunk, the block's
// channels ([t][cpb]) and the step's states ([t][NP]).
struct Stage {
  float *x, *dt, *dy, *B, *C;
};

__host__ __device__ constexpr size_t stage_floats(int cpb, int NP, int tc, bool bwd) {
  return (size_t)tc * ((bwd ? 3 : 2) * cpb + 2 * NP);
}

template <int kWc, int kT, bool kBwd>
__device__ __forceinline__ Stage stage_at(float* base) {
  constexpr int cpb = Geo<kWc>::cpb, NP = Geo<kWc>::NP;
  Stage s;
  s.x = base;
  s.dt = s.x + kT * cpb;
  s.dy = kBwd ? s.dt + kT * cpb : nullptr;
  s.B = (kBwd ? s.dy : s.dt) + kT * cpb;
  s.C = s.B + kT * NP;
  return s;
}

// Starts the copies of chunk k into st (dy only when given, C only when
// wanted); positions outside the sequence, the channels or the states are
// filled directly.
template <int kWc, int kT>
__device__ __forceinline__ void stage_load(const Stage& st, const M1& m, const float* dy, int b, int d0, int k,
                                           bool want_c) {
  constexpr int cpb = Geo<kWc>::cpb, NP = Geo<kWc>::NP;
  const int t0 = k * kT;
#pragma unroll
  for (int i = threadIdx.x; i < kT * cpb; i += kThreads) {
    const int t = t0 + i / cpb, d = d0 + i % cpb;
    if (t < m.T && d < m.D) {
      const size_t o = ((size_t)b * m.T + t) * m.D + d;
      cp_async4(st.x + i, m.x + o);
      cp_async4(st.dt + i, m.dt + o);
      if (dy) cp_async4(st.dy + i, dy + o);
    } else {
      st.x[i] = 0.f;
      st.dt[i] = -INFINITY;
      if (dy) st.dy[i] = 0.f;
    }
  }
#pragma unroll
  for (int i = threadIdx.x; i < kT * NP; i += kThreads) {
    const int t = t0 + i / NP, n = i % NP;
    if (t < m.T && n < m.N) {
      const size_t o = ((size_t)b * m.T + t) * m.N + n;
      cp_async4(st.B + i, m.B + o);
      if (want_c) cp_async4(st.C + i, m.C + o);
    } else {
      st.B[i] = 0.f;
      if (want_c) st.C[i] = 0.f;
    }
  }
}

template <int kWc>
__global__ void __launch_bounds__(kThreads) k_m1_forward(M1 m, float* y, float* s_final) {
  constexpr int cpb = Geo<kWc>::cpb, NP = Geo<kWc>::NP;
  constexpr size_t sf = stage_floats(cpb, NP, kTcF, false);
  extern __shared__ float smf[];
  const int tid = threadIdx.x, c = tid / kWc, l = tid % kWc;
  const int b = blockIdx.x / m.nblk, d0 = (blockIdx.x % m.nblk) * cpb, d = d0 + c;
  float* dtp = smf + kStages * sf;  // [kTcF][cpb] dt' of the chunk
  float* ys = dtp + kTcF * cpb;     // [kTcF][cpb] y of the chunk
  float A2[kS], s[kS];
#pragma unroll
  for (int j = 0; j < kS; ++j) {
    const int n = kS * l + j;
    const bool ok = d < m.D && n < m.N;
    A2[j] = ok ? m.A[(size_t)d * m.N + n] * kLog2e : 0.f;  // A log2(e)
    s[j] = ok && m.s0 ? m.s0[((size_t)b * m.D + d) * m.N + n] : 0.f;
  }
  for (int k = 0; k < kStages - 1; ++k) {
    if (k < m.nckf) stage_load<kWc, kTcF>(stage_at<kWc, kTcF, false>(smf + k * sf), m, nullptr, b, d0, k, true);
    cp_async_commit();
  }
  for (int k = 0; k < m.nckf; ++k) {
    const int kf = k + kStages - 1;
    if (kf < m.nckf)
      stage_load<kWc, kTcF>(stage_at<kWc, kTcF, false>(smf + (kf % kStages) * sf), m, nullptr, b, d0, kf, true);
    cp_async_commit();
    cp_async_wait_stages();
    __syncthreads();
    const Stage cur = stage_at<kWc, kTcF, false>(smf + (k % kStages) * sf);
#pragma unroll
    for (int i = tid; i < kTcF * cpb; i += kThreads) dtp[i] = softplus_f(cur.dt[i]);
    __syncthreads();
#pragma unroll
    for (int tt = 0; tt < kTcF; ++tt) {
      const float dp = dtp[tt * cpb + c], u = dp * cur.x[tt * cpb + c];
      float Bj[kS], Cj[kS];
      ldsk(cur.B + tt * NP + kS * l, Bj);
      ldsk(cur.C + tt * NP + kS * l, Cj);
      float yp = 0.f;
#pragma unroll
      for (int j = 0; j < kS; ++j) {
        s[j] = decay(dp, A2[j]) * s[j] + u * Bj[j];
        yp += s[j] * Cj[j];
      }
      yp = group_sum<kWc>(yp);
      if (l == 0) ys[tt * cpb + c] = yp;
    }
    __syncthreads();  // also: the chunk's buffers are free for the copies issued next
    const int t0 = k * kTcF;
#pragma unroll
    for (int i = tid; i < kTcF * cpb; i += kThreads) {
      const int t = t0 + i / cpb, dd = d0 + i % cpb;
      if (t < m.T && dd < m.D) y[((size_t)b * m.T + t) * m.D + dd] = ys[i];
    }
  }
#pragma unroll
  for (int j = 0; j < kS; ++j) {
    const int n = kS * l + j;
    if (d < m.D && n < m.N) s_final[((size_t)b * m.D + d) * m.N + n] = s[j];
  }
}

struct M1Bwd {
  const float* dy;
  const float* ds_final;
  float* ck;  // [b][nck][D][N]: the state entering every chunk
  float* dx;
  float* ddt_raw;
  float* dB_part;  // [b][T][nblk][N]
  float* dC_part;
  float* dA_part;  // [b][D][N]
  float* ds0;
};

template <int kWc>
__global__ void __launch_bounds__(kThreads, 4) k_m1_backward(M1 m, M1Bwd g) {
  constexpr int cpb = Geo<kWc>::cpb, NP = Geo<kWc>::NP;
  constexpr size_t sf = stage_floats(cpb, NP, kTc, true);
  extern __shared__ float smf[];
  const int tid = threadIdx.x, c = tid / kWc, l = tid % kWc;
  const int blk = blockIdx.x % m.nblk;
  const int b = blockIdx.x / m.nblk, d0 = blk * cpb, d = d0 + c;
  float* dtp = smf + kStages * sf;  // [kTc][cpb]
  float* sig = dtp + kTc * cpb;     // [kTc][cpb] sigmoid(dt_raw)
  float* dxs = sig + kTc * cpb;     // [kTc][cpb]
  float* dds = dxs + kTc * cpb;     // [kTc][cpb]
  float* rB = dds + kTc * cpb;      // [kTc][cpb][NP] per-channel dB terms
  float* rC = rB + kTc * cpb * NP;  // [kTc][cpb][NP] per-channel dC terms
  float A[kS], A2[kS], s[kS];
  bool act[kS];
#pragma unroll
  for (int j = 0; j < kS; ++j) {
    const int n = kS * l + j;
    act[j] = d < m.D && n < m.N;
    A[j] = act[j] ? m.A[(size_t)d * m.N + n] : 0.f;
    A2[j] = A[j] * kLog2e;
    s[j] = act[j] && m.s0 ? m.s0[((size_t)b * m.D + d) * m.N + n] : 0.f;
  }
  auto ck_at = [&](int k, int j) { return g.ck + (((size_t)b * m.nck + k) * m.D + d) * m.N + kS * l + j; };

  // ---- forward replay: the state entering every kTc-step chunk (its checkpoint), walking the sequence in
  //      staged chunks of kTcF steps as the forward does (a quarter of the barriers and dt' passes of kTc-step
  //      chunks); its buffers alias the reverse walk's, which are not in use yet
  {
    constexpr size_t sfr = stage_floats(cpb, NP, kTcF, false);
    float* dtr = smf + kStages * sfr;  // [kTcF][cpb] dt' of the chunk
    for (int k = 0; k < kStages - 1; ++k) {
      if (k < m.nckf) stage_load<kWc, kTcF>(stage_at<kWc, kTcF, false>(smf + k * sfr), m, nullptr, b, d0, k, false);
      cp_async_commit();
    }
    for (int k = 0; k < m.nckf; ++k) {
      const int kf = k + kStages - 1;
      if (kf < m.nckf)
        stage_load<kWc, kTcF>(stage_at<kWc, kTcF, false>(smf + (kf % kStages) * sfr), m, nullptr, b, d0, kf, false);
      cp_async_commit();
      cp_async_wait_stages();
      __syncthreads();
      const Stage cur = stage_at<kWc, kTcF, false>(smf + (k % kStages) * sfr);
#pragma unroll
      for (int i = tid; i < kTcF * cpb; i += kThreads) dtr[i] = softplus_f(cur.dt[i]);
      __syncthreads();
#pragma unroll
      for (int tt = 0; tt < kTcF; ++tt) {
        if (tt % kTc == 0) {  // the state entering backward chunk ck (chunks past the sequence are not stored)
          const int ck = (k * kTcF + tt) / kTc;
          if (ck < m.nck) {
#pragma unroll
            for (int j = 0; j < kS; ++j)
              if (act[j]) *ck_at(ck, j) = s[j];
          }
        }
        const float dp = dtr[tt * cpb + c], u = dp * cur.x[tt * cpb + c];
        float Bj[kS];
        ldsk(cur.B + tt * NP + kS * l, Bj);
#pragma unroll
        for (int j = 0; j < kS; ++j) s[j] = decay(dp, A2[j]) * s[j] + u * Bj[j];
      }
      __syncthreads();  // the chunk's buffers are free for the copies issued next
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
  }

  // ---- reverse walk over the chunks
  float dS[kS], dA[kS];
#pragma unroll
  for (int j = 0; j < kS; ++j) {
    dS[j] = act[j] ? g.ds_final[((size_t)b * m.D + d) * m.N + kS * l + j] : 0.f;
    dA[j] = 0.f;
  }
  for (int r = 0; r < kStages - 1; ++r) {
    const int k = m.nck - 1 - r;
    if (k >= 0) stage_load<kWc, kTc>(stage_at<kWc, kTc, true>(smf + r * sf), m, g.dy, b, d0, k, true);
    cp_async_commit();
  }
  for (int r = 0; r < m.nck; ++r) {
    const int k = m.nck - 1 - r, kf = k - (kStages - 1);
    if (kf >= 0)
      stage_load<kWc, kTc>(stage_at<kWc, kTc, true>(smf + ((r + kStages - 1) % kStages) * sf), m, g.dy, b, d0, kf,
                           true);
    cp_async_commit();
    // the chunk's entering state, from its checkpoint
    float S[kTc + 1][kS];
#pragma unroll
    for (int j = 0; j < kS; ++j) S[0][j] = act[j] ? *ck_at(k, j) : 0.f;
    cp_async_wait_stages();
    __syncthreads();
    const Stage cur = stage_at<kWc, kTc, true>(smf + (r % kStages) * sf);
#pragma unroll
    for (int i = tid; i < kTc * cpb; i += kThreads) {
      const float z = cur.dt[i];
      dtp[i] = softplus_f(z);
      sig[i] = sigmoid_f(z);
    }
    __syncthreads();
    // replay the chunk: states and decays of its steps, in registers
#pragma unroll
    for (int tt = 0; tt < kTc; ++tt) {
      const float dp = dtp[tt * cpb + c], u = dp * cur.x[tt * cpb + c];
      float Bj[kS];
      ldsk(cur.B + tt * NP + kS * l, Bj);
#pragma unroll
      for (int j = 0; j < kS; ++j) {
        S[tt + 1][j] = decay(dp, A2[j]) * S[tt][j] + u * Bj[j];
      }
    }
    // walk it backwards
#pragma unroll
    for (int tt = kTc - 1; tt >= 0; --tt) {
      const int ic = tt * cpb + c;
      const float dp = dtp[ic], xv = cur.x[ic], dyv = cur.dy[ic];
      float Bj[kS], Cj[kS];
      ldsk(cur.B + tt * NP + kS * l, Bj);
      ldsk(cur.C + tt * NP + kS * l, Cj);
      float up = 0.f, ddp = 0.f, tB[kS], tC[kS];
#pragma unroll
      for (int j = 0; j < kS; ++j) {
        const float aj = decay(dp, A2[j]);  // recomputed (the same bits as the replay's): registers for 4 states
        dS[j] += dyv * Cj[j];        // y_t = s_t . C_t
        tC[j] = dyv * S[tt + 1][j];  // dC_t uses s_t
        up += dS[j] * Bj[j];         // d(dt' x) direction
        tB[j] = dp * xv * dS[j];
        const float dda = aj * dS[j] * S[tt][j];  // the decay path, with s_{t-1}
        dA[j] += dp * dda;
        ddp += A[j] * dda;
        dS[j] *= aj;
      }
      const float u = group_sum<kWc>(up);
      const float dd = u * xv + group_sum<kWc>(ddp);
      if (l == 0) {
        dxs[ic] = dp * u;
        dds[ic] = dd * sig[ic];
      }
      stsk(rB + (size_t)ic * NP + kS * l, tB);
      stsk(rC + (size_t)ic * NP + kS * l, tC);
    }
    __syncthreads();  // also: the chunk's buffers are free for the copies issued next
    const int t0 = k * kTc;
    // dB, dC: this block's channels added in ascending order, one partial per (step, state)
#pragma unroll
    for (int i = tid; i < kTc * NP; i += kThreads) {
      const int tt = i / NP, n = i % NP, t = t0 + tt;
      float sb = 0.f, sc = 0.f;
#pragma unroll 8
      for (int cc = 0; cc < cpb; ++cc) {
        sb += rB[(tt * cpb + cc) * NP + n];
        sc += rC[(tt * cpb + cc) * NP + n];
      }
      if (t < m.T && n < m.N) {
        const size_t o = (((size_t)b * m.T + t) * m.nblk + blk) * m.N + n;
        g.dB_part[o] = sb;
        g.dC_part[o] = sc;
      }
    }
#pragma unroll
    for (int i = tid; i < kTc * cpb; i += kThreads) {
      const int t = t0 + i / cpb, dd = d0 + i % cpb;
      if (t < m.T && dd < m.D) {
        const size_t o = ((size_t)b * m.T + t) * m.D + dd;
        g.dx[o] = dxs[i];
        g.ddt_raw[o] = dds[i];
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kS; ++j) {
    if (!act[j]) continue;
    const size_t o = ((size_t)b * m.D + d) * m.N + kS * l + j;
    g.ds0[o] = dS[j];
    g.dA_part[o] = dA[j];
  }
}

// out[b,t,n] = sum over the channel blocks (ascending) of part[b,t,blk,n].
__global__ void k_m1_channel_sum(const float* part, float* out, int b, int T, int nblk, int N) {
  const size_t total = (size_t)b * T * N;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const size_t bt = e / N;
    const int n = e % N;
    float acc = 0.f;
    for (int k = 0; k < nblk; ++k) acc += part[(bt * nblk + k) * N + n];
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
  const int need = (N + kS - 1) / kS;
  int w = 1;
  while (w < need) w <<= 1;
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
  m.b = d.b;
  m.T = d.T;
  m.D = d.H;
  m.N = d.N;
  m.Wc = lanes_for(d.N);
  const int cpb = kThreads / m.Wc;
  m.nblk = (d.H + cpb - 1) / cpb;
  m.nck = (d.T + kTc - 1) / kTc;
  m.nckf = (d.T + kTcF - 1) / kTcF;
  return m;
}

template <int kWc>
size_t fwd_smem() {
  constexpr int cpb = Geo<kWc>::cpb, NP = Geo<kWc>::NP;
  return (kStages * stage_floats(cpb, NP, kTcF, false) + 2 * (size_t)kTcF * cpb) * sizeof(float);
}
template <int kWc>
size_t bwd_smem() {
  constexpr int cpb = Geo<kWc>::cpb, NP = Geo<kWc>::NP;
  // the reverse walk's buffers, or the forward replay's (kTcF-step stages and their dt'), which alias them
  const size_t walk = kStages * stage_floats(cpb, NP, kTc, true) + 4 * (size_t)kTc * cpb + 2 * (size_t)kTc * cpb * NP;
  const size_t replay = kStages * stage_floats(cpb, NP, kTcF, false) + (size_t)kTcF * cpb;
  return (walk > replay ? walk : replay) * sizeof(float);
}

template <int kWc>
cudaError_t launch_fwd(const M1& m, float* y, float* s_final, cudaStream_t st) {
  const size_t smem = fwd_smem<kWc>();
  cudaError_t e = cudaFuncSetAttribute(k_m1_forward<kWc>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned blocks = (unsigned)((long long)m.b * m.nblk);
  SSD_LAUNCH("k_m1_forward", st, k_m1_forward<kWc><<<blocks, kThreads, smem, st>>>(m, y, s_final));
  return cudaGetLastError();
}

template <int kWc>
cudaError_t launch_bwd(const M1& m, const M1Bwd& g, cudaStream_t st) {
  const size_t smem = bwd_smem<kWc>();
  cudaError_t e = cudaFuncSetAttribute(k_m1_backward<kWc>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned blocks = (unsigned)((long long)m.b * m.nblk);
  SSD_LAUNCH("k_m1_backward", st, k_m1_backward<kWc><<<blocks, kThreads, smem, st>>>(m, g));
  return cudaGetLastError();
}

struct M1Ws {
  float *ck, *dB_part, *dC_part, *dA_part;
};

M1Ws carve_m1(const Dims& d, Carver& cv) {
  const M1 m = make_m1(d, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
  M1Ws w;
  w.ck = cv.take<float>((size_t)d.b * m.nck * d.H * d.N);
  w.dB_part = cv.take<float>((size_t)d.b * d.T * m.nblk * d.N);
  w.dC_part = cv.take<float>((size_t)d.b * d.T * m.nblk * d.N);
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
  const M1 m = make_m1(d, a.x, a.dt_raw, a.A, a.B, a.C, a.s0);
  if ((long long)m.b * m.nblk > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  float* y = static_cast<float*>(a.y);
  switch (m.Wc) {  // N <= 32 and four states a thread: 1 to 8 threads a channel
    case 1: return launch_fwd<1>(m, y, a.s_final, st);
    case 2: return launch_fwd<2>(m, y, a.s_final, st);
    case 4: return launch_fwd<4>(m, y, a.s_final, st);
    case 8: return launch_fwd<8>(m, y, a.s_final, st);
    case 16: return launch_fwd<16>(m, y, a.s_final, st);
  }
  return cudaErrorInvalidConfiguration;
}

cudaError_t m1_backward(const Dims& d, const BwdArgs& a, void* ws, cudaStream_t st) {
  Carver cv(ws);
  M1Ws w = carve_m1(d, cv);
  const M1 m = make_m1(d, a.x, a.dt_raw, a.A, a.B, a.C, a.s0);
  if ((long long)m.b * m.nblk > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  M1Bwd g{static_cast<const float*>(a.dy), a.ds_final, w.ck, static_cast<float*>(a.dx), a.ddt_raw,
          w.dB_part, w.dC_part, w.dA_part, a.ds0};
  cudaError_t e = cudaErrorInvalidConfiguration;
  switch (m.Wc) {
    case 1: e = launch_bwd<1>(m, g, st); break;
    case 2: e = launch_bwd<2>(m, g, st); break;
    case 4: e = launch_bwd<4>(m, g, st); break;
    case 8: e = launch_bwd<8>(m, g, st); break;
    case 16: e = launch_bwd<16>(m, g, st); break;
  }
  if (e != cudaSuccess) return e;
  const size_t tot = (size_t)d.b * d.T * d.N;
  const int rb = (int)((tot + 255) / 256 < 65535 ? (tot + 255) / 256 : 65535);
  SSD_LAUNCH("k_m1_channel_sum", st,
             k_m1_channel_sum<<<rb, 256, 0, st>>>(w.dB_part, static_cast<float*>(a.dB), d.b, d.T, m.nblk, d.N));
  SSD_LAUNCH("k_m1_channel_sum", st,
             k_m1_channel_sum<<<rb, 256, 0, st>>>(w.dC_part, static_cast<float*>(a.dC), d.b, d.T, m.nblk, d.N));
  SSD_LAUNCH("k_m1_dA_sum", st,
             k_m1_dA_sum<<<(d.H * d.N + 255) / 256, 256, 0, st>>>(w.dA_part, a.dA, d.b, d.H * d.N));
  return cudaGetLastError();
}

}  // namespace ssd
