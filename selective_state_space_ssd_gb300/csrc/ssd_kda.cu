// The KDA delta-rule recurrence and its BPTT backward (the notes page
// "sec-10.tex", section "反向传播推导": forward F1-F6, reverse steps 1-6), fp32.
//
// Per batch element b and value head hv (query / key head h = hv / G), the
// state S is K x V.  Each warp owns 4 value columns of one (b, hv) and keeps
// its K x 4 slice of S in registers: lane l holds rows l, l + 32, l + 64,
// l + 96.  Column work (p = k^T S_dec, o = q^T S, dr) reduces over the key
// rows of a column: a warp reduction.  Row work of the backward (dq, da, dk,
// dg) reduces over the value columns: each warp's 4-column partial sums are
// added over the warps of its CTA in warp order (shared memory, one barrier
// per step), then over the CTAs of the (b, hv) in CTA order (a small kernel).
// Every warp loads the next step's inputs while it computes the current one,
// so their global latency is off the recurrence's critical path.
//
//   forward   k_kda_forward<false>: o and s_final, every warp on its own.
//   backward  1. k_kda_forward<true> replays the forward from the leaf inputs
//                and keeps the state entering every 8th step (checkpoints,
//                stored lane-major so every store is one coalesced line);
//             2. k_kda_backward, CTAs of up to eight column warps of one
//                (b, hv), walks the 8-step segments from the last: it replays
//                the segment from its checkpoint (S_dec and r of every step to
//                shared memory), then runs steps 1-6 backwards through it,
//                carrying dS_acc in registers across segments, and writes the
//                CTA's row sums per step;
//             3. k_kda_rows adds the CTAs' row sums in CTA order (dq, dk, dg,
//                dbeta per value head);
//             4. k_kda_gva adds the per-value-head dq, dk onto their query /
//                key head in a fixed order (the page's view + sum) and scales
//                dq.
#include <math.h>
#include <stdint.h>

#include <initializer_list>

#include "../../include/ssd.h"
#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kRows = 4;       // key rows per lane: K <= 128
constexpr int kCols = 4;       // value columns per warp: V <= 128 in at most 32 warps
constexpr int kSeg = 8;        // steps per checkpoint segment
constexpr int kMaxWarps = 32;  // column warps of a (b, hv)
constexpr int kCtaWarps = 8;   // column warps of a backward CTA
constexpr int kSlice = 32 * kRows * kCols;  // floats of one warp's state slice
// dynamic shared memory of a backward CTA: the replay scratch of a segment for kCtaWarps warps
constexpr size_t kBwdSmem = (size_t)kSeg * (kCtaWarps * kSlice + kCols * kCtaWarps) * sizeof(float);

struct KdaDims {
  int b, T, H, HV, G, K, V;
  int nw;     // column warps per (b, hv): ceil(V / 8)
  int nseg;   // checkpoint segments: ceil(T / 16)
  int wpc;    // column warps per backward CTA: min(nw, 4)
  int nsplit; // backward CTAs per (b, hv): ceil(nw / wpc)
};

struct KdaIn {
  const float* q;     // [b,T,H,K]
  const float* k;     // [b,T,H,K]
  const float* v;     // [b,T,HV,V]
  const float* g;     // [b,T,HV,K]
  const float* beta;  // [b,T,HV]
  float scale;
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// The per-step inputs of one warp: its rows of q, k, g, beta, and its columns of v, as loaded (load_step), then
// finished (finish_step: q scaled, g -> exp(g)).  Rows and columns outside K, V read 0 (exp(0) = 1 keeps those
// state entries at 0).
struct StepIn {
  float q[kRows], k[kRows], eg[kRows], v[kCols], beta;
};

__device__ __forceinline__ void load_step(const KdaIn& in, const KdaDims& d, int b, int hv, int t, int lane, int col0,
                                          StepIn& s) {
  const int h = hv / d.G;
  const size_t qk = ((size_t)b * d.T + t) * d.H + h, gv = ((size_t)b * d.T + t) * d.HV + hv;
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int r = lane + 32 * i;
    const bool ok = r < d.K;
    s.q[i] = ok ? in.q[qk * d.K + r] : 0.f;
    s.k[i] = ok ? in.k[qk * d.K + r] : 0.f;
    s.eg[i] = ok ? in.g[gv * d.K + r] : 0.f;
  }
#pragma unroll
  for (int j = 0; j < kCols; ++j) s.v[j] = col0 + j < d.V ? in.v[gv * d.V + col0 + j] : 0.f;
  s.beta = in.beta[gv];
}

__device__ __forceinline__ void finish_step(StepIn& s, float scale) {
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    s.q[i] *= scale;
    s.eg[i] = __expf(s.eg[i]);
  }
}

// F1-F5 on this warp's slice: S <- S_dec + beta k (x) (v - k^T S_dec); returns r (all lanes).
__device__ __forceinline__ void delta_step(float (&S)[kRows][kCols], const StepIn& s, float (&r)[kCols]) {
#pragma unroll
  for (int i = 0; i < kRows; ++i)
#pragma unroll
    for (int j = 0; j < kCols; ++j) S[i][j] *= s.eg[i];  // F1
#pragma unroll
  for (int j = 0; j < kCols; ++j) {
    float p = 0.f;
#pragma unroll
    for (int i = 0; i < kRows; ++i) p = fmaf(s.k[i], S[i][j], p);
    r[j] = s.v[j] - warp_sum(p);  // F2, F3
  }
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const float a = s.beta * s.k[i];  // F4
#pragma unroll
    for (int j = 0; j < kCols; ++j) S[i][j] = fmaf(a, r[j], S[i][j]);  // F5
  }
}

// F1-F6 on this warp's slice for the forward, with o_j = q^T S_t[:, j] = q^T S_dec[:, j] + (q . a) r_j (F5): the
// column sums q^T S_dec reduce beside k^T S_dec and q . k needs no state, so the only work after the state update
// is one FMA per column (reduced after F5, o's warp sums had held each step up).  Lanes 0 .. kCols - 1 return
// o[col0 + lane].
__device__ __forceinline__ float delta_step_o(float (&S)[kRows][kCols], const StepIn& s, int lane) {
  float qk = 0.f;
#pragma unroll
  for (int i = 0; i < kRows; ++i) qk = fmaf(s.q[i], s.k[i], qk);
#pragma unroll
  for (int i = 0; i < kRows; ++i)
#pragma unroll
    for (int j = 0; j < kCols; ++j) S[i][j] *= s.eg[i];  // F1
  float p[kCols], qs[kCols];
#pragma unroll
  for (int j = 0; j < kCols; ++j) {
    p[j] = 0.f, qs[j] = 0.f;
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      p[j] = fmaf(s.k[i], S[i][j], p[j]);
      qs[j] = fmaf(s.q[i], S[i][j], qs[j]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    qk += __shfl_xor_sync(0xffffffffu, qk, o);
#pragma unroll
    for (int j = 0; j < kCols; ++j) {
      p[j] += __shfl_xor_sync(0xffffffffu, p[j], o);
      qs[j] += __shfl_xor_sync(0xffffffffu, qs[j], o);
    }
  }
  const float qa = s.beta * qk;  // q . a with a = beta k (F4)
  float out = 0.f;
#pragma unroll
  for (int j = 0; j < kCols; ++j) {
    const float r = s.v[j] - p[j];  // F2, F3
#pragma unroll
    for (int i = 0; i < kRows; ++i) S[i][j] = fmaf(s.beta * s.k[i], r, S[i][j]);  // F5
    const float oj = fmaf(qa, r, qs[j]);                                           // F6
    if (lane == j) out = oj;
  }
  return out;
}

// Checkpoint slot of warp w's slice: [unit][seg][w][i * kCols + j][lane] (lane-major: one coalesced line per store)
__device__ __forceinline__ size_t ckpt_slot(const KdaDims& d, int unit, int seg, int w) {
  return (((size_t)unit * d.nseg + seg) * d.nw + w) * kSlice;
}

// Forward: one warp per 4 columns of one (b, hv); grid (b * HV, ceil(nw / 2)), two warps per CTA.
// kCkpt: the backward's replay, which writes only the state entering every kSeg-th step (checkpoints);
// otherwise o [b,T,HV,V] and s_final [b,HV,K,V].
template <bool kCkpt>
__global__ void __launch_bounds__(64) k_kda_forward(KdaIn in, KdaDims d, const float* __restrict__ s0, float* o,
                                                    float* s_final, float* ckpt) {
  const int lane = threadIdx.x & 31;
  const int w = blockIdx.y * 2 + (threadIdx.x >> 5);
  if (w >= d.nw) return;
  const int unit = blockIdx.x, b = unit / d.HV, hv = unit - b * d.HV;
  const int col0 = kCols * w;
  const size_t sbase = (size_t)unit * d.K * d.V;
  float S[kRows][kCols];
#pragma unroll
  for (int i = 0; i < kRows; ++i)
#pragma unroll
    for (int j = 0; j < kCols; ++j) {
      const int r = lane + 32 * i, c = col0 + j;
      S[i][j] = s0 && r < d.K && c < d.V ? s0[sbase + (size_t)r * d.V + c] : 0.f;
    }
  StepIn nx;
  load_step(in, d, b, hv, 0, lane, col0, nx);
  auto step = [&](int t) {
    if (kCkpt && t % kSeg == 0) {
      float* dst = ckpt + ckpt_slot(d, unit, t / kSeg, w);
#pragma unroll
      for (int i = 0; i < kRows; ++i)
#pragma unroll
        for (int j = 0; j < kCols; ++j) dst[(i * kCols + j) * 32 + lane] = S[i][j];
    }
    StepIn s = nx;
    if (t + 1 < d.T) load_step(in, d, b, hv, t + 1, lane, col0, nx);
    finish_step(s, in.scale);
    if (kCkpt) {
      float r[kCols];
      delta_step(S, s, r);
    } else {
      const float out = delta_step_o(S, s, lane);  // o[col0 + lane] for lanes 0 .. kCols - 1
      if (lane < kCols && col0 + lane < d.V) o[(((size_t)b * d.T + t) * d.HV + hv) * d.V + col0 + lane] = out;
    }
  };
  if (kCkpt) {
    // the replay unrolled by two: a step's loads and exponentials overlap the previous step's reductions (the
    // forward with o measured slower unrolled)
#pragma unroll 2
    for (int t = 0; t < d.T; ++t) step(t);
  } else {
    for (int t = 0; t < d.T; ++t) step(t);
  }
  if (!kCkpt) {
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < kCols; ++j) {
        const int r = lane + 32 * i, c = col0 + j;
        if (r < d.K && c < d.V) s_final[sbase + (size_t)r * d.V + c] = S[i][j];
      }
  }
}

struct KdaBwdOut {
  const float* dout;      // do [b,T,HV,V]
  const float* ds_final;  // [b,HV,K,V]
  float* part;            // [b,T,HV][nsplit][dq, da, dk_r, dg rows (4 K), then dbeta]: row sums of each CTA
  float* dv;              // [b,T,HV,V]
  float* ds0;             // [b,HV,K,V]
  const float* ckpt;      // checkpoints (ckpt_slot)
};

// Backward: CTA (unit, split) runs column warps split * wpc .. + wpc - 1 of (b, hv) = unit (the warps past nw
// only join the barriers).  Static shared memory: the per-step row partials of its warps, double-buffered,
// [buf][warp][dq, da, dk_r, dg][row 0..127], and their dbeta partials [buf][warp].
__global__ void __launch_bounds__(32 * kCtaWarps) k_kda_backward(KdaIn in, KdaDims d, KdaBwdOut out) {
  constexpr int kPartRow = 32 * kRows;
  __shared__ float part[2][kCtaWarps][4][kPartRow];
  __shared__ float dbp[2][kCtaWarps];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int unit = blockIdx.x, split = blockIdx.y, b = unit / d.HV, hv = unit - b * d.HV;
  const int w = split * d.wpc + wl;  // the warp's column block of the (b, hv)
  const bool live = wl < d.wpc && w < d.nw;
  const int nlive = min(d.wpc, d.nw - split * d.wpc);
  const int col0 = kCols * w;
  const size_t sbase = (size_t)unit * d.K * d.V;
  // the replay scratch, in shared memory: kSeg steps x (wpc slices of S_dec, then kCols wpc values of r)
  extern __shared__ float scr[];
  const size_t step_floats = (size_t)d.wpc * kSlice + kCols * d.wpc;  // one step of the scratch
  auto sd_at = [&](float* st, int i, int j) -> float& { return st[(size_t)wl * kSlice + (i * kCols + j) * 32 + lane]; };
  auto r_at = [&](float* st, int j) -> float& { return st[(size_t)d.wpc * kSlice + kCols * wl + j]; };
  const int rstride = 4 * d.K + 1;
  float dS[kRows][kCols];  // dS_acc, seeded with ds_final
#pragma unroll
  for (int i = 0; i < kRows; ++i)
#pragma unroll
    for (int j = 0; j < kCols; ++j) {
      const int r = lane + 32 * i, c = col0 + j;
      dS[i][j] = live && r < d.K && c < d.V ? out.ds_final[sbase + (size_t)r * d.V + c] : 0.f;
    }
  int step = 0;  // steps done, for the double buffer
  for (int sg = d.nseg - 1; sg >= 0; --sg) {
    const int t0 = sg * kSeg, t1 = min(d.T, t0 + kSeg);
    // replay the segment from its checkpoint: S_dec and r of every step to the scratch
    if (live) {
      float S[kRows][kCols];
      const float* src = out.ckpt + ckpt_slot(d, unit, sg, w);
#pragma unroll
      for (int i = 0; i < kRows; ++i)
#pragma unroll
        for (int j = 0; j < kCols; ++j) S[i][j] = src[(i * kCols + j) * 32 + lane];
      StepIn nx;
      load_step(in, d, b, hv, t0, lane, col0, nx);
      for (int t = t0; t < t1; ++t) {
        StepIn s = nx;
        if (t + 1 < t1) load_step(in, d, b, hv, t + 1, lane, col0, nx);
        finish_step(s, in.scale);
        float r[kCols];
        float* st = scr + (size_t)(t - t0) * step_floats;
#pragma unroll
        for (int i = 0; i < kRows; ++i)
#pragma unroll
          for (int j = 0; j < kCols; ++j) sd_at(st, i, j) = S[i][j] * s.eg[i];
        delta_step(S, s, r);
        float rv = r[0];
#pragma unroll
        for (int j = 1; j < kCols; ++j)
          if (lane == j) rv = r[j];
        if (lane < kCols) r_at(st, lane) = rv;
      }
    }
    __syncwarp();  // the r values of the warp's columns, written by lanes 0 .. kCols - 1, are read by every lane
    // steps 1-6 backwards through the segment; a step's inputs and do are loaded one step ahead
    StepIn nx;
    float dnx[kCols];
    auto load_do = [&](int t, float (&x)[kCols]) {
      const size_t g = ((size_t)b * d.T + t) * d.HV + hv;
#pragma unroll
      for (int j = 0; j < kCols; ++j) x[j] = col0 + j < d.V ? out.dout[g * d.V + col0 + j] : 0.f;
    };
    if (live) {
      load_step(in, d, b, hv, t1 - 1, lane, col0, nx);
      load_do(t1 - 1, dnx);
    }
    for (int t = t1 - 1; t >= t0; --t, ++step) {
      const int pb = step & 1;
      const size_t gv = ((size_t)b * d.T + t) * d.HV + hv;
      StepIn s = nx;
      float dov[kCols];
#pragma unroll
      for (int j = 0; j < kCols; ++j) dov[j] = dnx[j];
      if (live) {
        if (t > t0) {
          load_step(in, d, b, hv, t - 1, lane, col0, nx);
          load_do(t - 1, dnx);
        }
        finish_step(s, in.scale);
        float* st = scr + (size_t)(t - t0) * step_floats;
        float r[kCols], u[kCols];
#pragma unroll
        for (int j = 0; j < kCols; ++j) r[j] = r_at(st, j);
        // step 1: dS_acc += q (x) do;  dq = S_t do with S_t = S_dec + beta k (x) r;  step 2: da = dS_acc r
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
          const float a = s.beta * s.k[i];
          float xq = 0.f, xa = 0.f;
#pragma unroll
          for (int j = 0; j < kCols; ++j) {
            dS[i][j] = fmaf(s.q[i], dov[j], dS[i][j]);
            xq = fmaf(dov[j], fmaf(a, r[j], sd_at(st, i, j)), xq);
            xa = fmaf(r[j], dS[i][j], xa);
          }
          part[pb][wl][0][lane + 32 * i] = xq;
          part[pb][wl][1][lane + 32 * i] = xa;
        }
        // step 2: dr = a^T dS_acc = beta u with u = k^T dS_acc per column (a warp reduction);
        // step 3: dbeta = sum_k k da = sum_v r u
        float dbw = 0.f;
#pragma unroll
        for (int j = 0; j < kCols; ++j) {
          float x = 0.f;
#pragma unroll
          for (int i = 0; i < kRows; ++i) x = fmaf(s.k[i], dS[i][j], x);
          u[j] = warp_sum(x);
          dbw = fmaf(r[j], u[j], dbw);
        }
        // step 4: dv = dr,  dk_r = -S_dec dr;  step 5: dS_dec = dS_acc - k (x) dr (both paths),
        // dg = rowsum(S_dec o dS_dec),  dS_{t-1} = exp(g) o dS_dec
        float dvo = 0.f;
#pragma unroll
        for (int j = 0; j < kCols; ++j)
          if (lane == j) dvo = s.beta * u[j];
        if (lane < kCols && col0 + lane < d.V) out.dv[gv * d.V + col0 + lane] = dvo;
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
          float xk = 0.f, xg = 0.f;
#pragma unroll
          for (int j = 0; j < kCols; ++j) {
            const float dr = s.beta * u[j];
            const float sdv = sd_at(st, i, j);
            xk = fmaf(-sdv, dr, xk);
            const float tot = fmaf(-s.k[i], dr, dS[i][j]);
            xg = fmaf(sdv, tot, xg);
            dS[i][j] = s.eg[i] * tot;
          }
          part[pb][wl][2][lane + 32 * i] = xk;
          part[pb][wl][3][lane + 32 * i] = xg;
        }
        if (lane == 0) dbp[pb][wl] = dbw;
      }
      __syncthreads();
      // this CTA's row sums: its live warps added in warp order
      float* dst = out.part + (gv * d.nsplit + split) * rstride;
      for (int row = threadIdx.x; row < d.K; row += blockDim.x) {
        float q_ = 0.f, a_ = 0.f, k_ = 0.f, g_ = 0.f;
        for (int ww = 0; ww < nlive; ++ww) {
          q_ += part[pb][ww][0][row];
          a_ += part[pb][ww][1][row];
          k_ += part[pb][ww][2][row];
          g_ += part[pb][ww][3][row];
        }
        dst[row] = q_;
        dst[d.K + row] = a_;
        dst[2 * d.K + row] = k_;
        dst[3 * d.K + row] = g_;
      }
      if (threadIdx.x == 0) {
        float x = 0.f;
        for (int ww = 0; ww < nlive; ++ww) x += dbp[pb][ww];
        dst[4 * d.K] = x;
      }
    }
    __syncwarp();  // this segment's scratch has been read before the next replay overwrites it
  }
  if (live) {
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int j = 0; j < kCols; ++j) {
        const int r = lane + 32 * i, c = col0 + j;
        if (r < d.K && c < d.V) out.ds0[sbase + (size_t)r * d.V + c] = dS[i][j];
      }
  }
}

// Per (b, t, hv): the CTAs' row sums added in CTA order; dk = beta da + dk_r (step 6), dq per value head (w.r.t.
// the scaled q), dg and dbeta.  One block of 128 threads per (b, t, hv), thread = key row.
__global__ void __launch_bounds__(128) k_kda_rows(const float* __restrict__ part, const float* __restrict__ beta,
                                                  float* dq_e, float* dk_e, float* dg, float* dbeta, long long n,
                                                  int K, int nsplit) {
  const int rstride = 4 * K + 1;
  for (long long gv = blockIdx.x; gv < n; gv += gridDim.x) {
    const float* p = part + (size_t)gv * nsplit * rstride;
    const float bt = beta[gv];
    for (int row = threadIdx.x; row < K; row += blockDim.x) {
      float q_ = 0.f, a_ = 0.f, k_ = 0.f, g_ = 0.f;
      for (int s = 0; s < nsplit; ++s) {
        const float* ps = p + (size_t)s * rstride;
        q_ += ps[row];
        a_ += ps[K + row];
        k_ += ps[2 * K + row];
        g_ += ps[3 * K + row];
      }
      dq_e[(size_t)gv * K + row] = q_;
      dk_e[(size_t)gv * K + row] = fmaf(bt, a_, k_);
      dg[(size_t)gv * K + row] = g_;
    }
    if (threadIdx.x == 0) {
      float x = 0.f;
      for (int s = 0; s < nsplit; ++s) x += p[(size_t)s * rstride + 4 * K];
      dbeta[gv] = x;
    }
  }
}

// dq[b,t,h,:] = scale * sum_{j < G} dq_e[b,t,h*G+j,:],  dk[b,t,h,:] = sum_{j < G} dk_e[b,t,h*G+j,:]  (j ascending)
__global__ void k_kda_gva(const float* __restrict__ dq_e, const float* __restrict__ dk_e, float* dq, float* dk,
                          long long n, int G, int K, float scale) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / K, kk = i - row * K;  // row = (b*T + t)*H + h
    const size_t src = ((size_t)row * G) * K + kk;
    float sq = 0.f, sk = 0.f;
    for (int j = 0; j < G; ++j) {
      sq += dq_e[src + (size_t)j * K];
      sk += dk_e[src + (size_t)j * K];
    }
    dq[i] = sq * scale;
    dk[i] = sk;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ssd_status kda_dims(const ssd_kda_problem* p, KdaDims* d) {
  if (!p) return SSD_ERR_INVALID_ARG;
  if (p->batch < 1 || p->seqlen < 1 || p->nheads < 1 || p->value_heads < 1 || p->key_dim < 1 || p->value_dim < 1)
    return SSD_ERR_INVALID_ARG;
  if (p->value_heads % p->nheads) return SSD_ERR_SHAPE;
  if (p->key_dim > 32 * kRows || p->value_dim > kCols * kMaxWarps) return SSD_ERR_SHAPE;
  const long long units = p->batch * p->value_heads;
  if (units > 0x7fffffffll || p->seqlen > 0x7fffffffll || p->batch * p->seqlen * p->value_heads > (1ll << 40))
    return SSD_ERR_SHAPE;
  d->b = (int)p->batch;
  d->T = (int)p->seqlen;
  d->H = (int)p->nheads;
  d->HV = (int)p->value_heads;
  d->G = d->HV / d->H;
  d->K = (int)p->key_dim;
  d->V = (int)p->value_dim;
  d->nw = (d->V + kCols - 1) / kCols;
  d->nseg = (d->T + kSeg - 1) / kSeg;
  d->wpc = d->nw < kCtaWarps ? d->nw : kCtaWarps;
  d->nsplit = (d->nw + d->wpc - 1) / d->wpc;
  return SSD_OK;
}

struct KdaWs {
  float *ckpt, *part, *dq_e, *dk_e;
};

// Backward workspace: checkpoints (units x nseg x nw slices), the CTAs' per-step row sums, and the per-value-head
// dq, dk.
KdaWs kda_carve(const KdaDims& d, Carver& cv) {
  KdaWs w;
  const size_t units = (size_t)d.b * d.HV, rows = (size_t)d.b * d.T * d.HV;
  w.ckpt = cv.take<float>(units * d.nseg * d.nw * kSlice);
  w.part = cv.take<float>(rows * d.nsplit * (4 * (size_t)d.K + 1));
  w.dq_e = cv.take<float>(rows * d.K);
  w.dk_e = cv.take<float>(rows * d.K);
  return w;
}

ssd_status check_ptrs16(std::initializer_list<const void*> req, const void* opt) {
  for (const void* p : req) {
    if (!p) return SSD_ERR_INVALID_ARG;
    if (!aligned16(p)) return SSD_ERR_ALIGNMENT;
  }
  if (opt && !aligned16(opt)) return SSD_ERR_ALIGNMENT;
  return SSD_OK;
}

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

ssd_status ssd_kda_workspace_size(const ssd_kda_problem* prob, int backward, size_t* bytes) {
  if (!bytes) return SSD_ERR_INVALID_ARG;
  KdaDims d;
  ssd_status s = kda_dims(prob, &d);
  if (s != SSD_OK) return s;
  Carver cv(nullptr);
  if (backward) kda_carve(d, cv);
  *bytes = cv.off;
  return SSD_OK;
}

ssd_status ssd_kda_forward(const ssd_kda_problem* prob, const float* q, const float* k, const float* v,
                           const float* g, const float* beta, const float* s0, float scale, float* o, float* s_final,
                           void* ws, size_t ws_bytes, void* cuda_stream) {
  KdaDims d;
  ssd_status s = kda_dims(prob, &d);
  if (s != SSD_OK) return s;
  s = check_ptrs16({q, k, v, g, beta, o, s_final, ws}, s0);
  if (s != SSD_OK) return s;
  Carver cv(nullptr);
  if (ws_bytes < cv.off) return SSD_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return SSD_ERR_CUDA;
  const KdaIn in{q, k, v, g, beta, scale};
  const dim3 grid((unsigned)(d.b * d.HV), (unsigned)((d.nw + 1) / 2));
  SSD_LAUNCH("k_kda_forward", st, k_kda_forward<false><<<grid, 64, 0, st>>>(in, d, s0, o, s_final, nullptr));
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

ssd_status ssd_kda_backward(const ssd_kda_problem* prob, const float* dout, const float* ds_final, const float* q,
                            const float* k, const float* v, const float* g, const float* beta, const float* s0,
                            float scale, float* dq, float* dk, float* dv, float* dg, float* dbeta, float* ds0,
                            void* ws, size_t ws_bytes, void* cuda_stream) {
  KdaDims d;
  ssd_status s = kda_dims(prob, &d);
  if (s != SSD_OK) return s;
  s = check_ptrs16({dout, ds_final, q, k, v, g, beta, dq, dk, dv, dg, dbeta, ds0, ws}, s0);
  if (s != SSD_OK) return s;
  Carver need(nullptr);
  kda_carve(d, need);
  if (ws_bytes < need.off) return SSD_ERR_WORKSPACE;
  Carver cv(ws);
  const KdaWs w = kda_carve(d, cv);
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return SSD_ERR_CUDA;
  const KdaIn in{q, k, v, g, beta, scale};
  const dim3 grid((unsigned)(d.b * d.HV), (unsigned)((d.nw + 1) / 2));
  SSD_LAUNCH("k_kda_checkpoints", st, k_kda_forward<true><<<grid, 64, 0, st>>>(in, d, s0, nullptr, nullptr, w.ckpt));
  const KdaBwdOut out{dout, ds_final, w.part, dv, ds0, w.ckpt};
  if (cudaFuncSetAttribute(k_kda_backward, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBwdSmem) != cudaSuccess)
    return SSD_ERR_CUDA;
  SSD_LAUNCH("k_kda_backward", st,
             k_kda_backward<<<dim3((unsigned)(d.b * d.HV), (unsigned)d.nsplit), 32 * kCtaWarps, kBwdSmem, st>>>(in, d, out));
  const long long rows = (long long)d.b * d.T * d.HV;
  const unsigned rblocks = (unsigned)(rows < 65535 * 8 ? rows : 65535 * 8);
  SSD_LAUNCH("k_kda_rows", st,
             k_kda_rows<<<rblocks, 128, 0, st>>>(w.part, beta, w.dq_e, w.dk_e, dg, dbeta, rows, d.K, d.nsplit));
  const long long n = (long long)d.b * d.T * d.H * d.K;
  const unsigned blocks = (unsigned)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  SSD_LAUNCH("k_kda_gva", st, k_kda_gva<<<blocks, 256, 0, st>>>(w.dq_e, w.dk_e, dq, dk, n, d.G, d.K, scale));
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // extern "C"
