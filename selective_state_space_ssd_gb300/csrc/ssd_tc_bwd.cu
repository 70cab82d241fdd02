// Recompute backward of the Mamba-2 scan on tcgen05 tensor cores (bf16 io,
// chunk L = 64, head dim P = 64, state N = 128).  It follows the recompute
// backward of the burn-mamba page "combined_backward.rs": replay the forward
// intermediates from the saved leaf inputs, then walk the chunks in reverse
// carrying the state gradient dS from the (nonzero) ds_final seed, fusing the
// K5 (BLUE + ORANGE) and K4 backwards, with the K3, K2 and K1 backwards done
// chunk by chunk in the same pass.
//
// One CTA owns one (batch, head).
//   replay:  a separate launch (the pipelined forward kernel in its states
//            mode) writes every chunk-input state S_c (bf16) to the workspace.
//   reverse: for c = nc-1 .. 0, with dS = dS_{c+1} (fp32 in registers):
//     dS_blue^T = C^T dch          dch = exp(cum_t) dy     (BLUE: d state)
//     dC        = dch S_c + dCB B                         (BLUE + K2)
//     dW        = dy v^T,  CB = C B^T                      (ORANGE)
//     W = CB o decay_in, dCB = dW o decay_in, d_diff = dW o W (mask first)
//     dv        = W^T dy + exp(cum_end - cum_s) B dS^T     (ORANGE + K3)
//     dB        = dvd dS^T + dCB^T C                       (K3 + K2)
//     d cum     = rowsum - colsum of d_diff (ORANGE), C.dC_blue (BLUE),
//                 -exp(..) v.(B dS^T) (K3), exp(cum_end)<dS, S_c> at the
//                 chunk end (K4); K1 backward is a suffix sum.
//     dS_c      = exp(cum_end) dS_{c+1} + dS_blue                 (K4)
//   leaves: dx = dt' dv, ddt_raw = (sum_p dv x + A dda) sigmoid(dt_raw),
//           per-chunk dA parts; dB, dC are written per head (fp32) and summed
//           over the heads of each group afterwards in a fixed order.
#include "ssd_device.cuh"
#include "ssd_internal.h"
#include "tc_common.cuh"

namespace ssd {
namespace {
using namespace tc;

constexpr int kL = 64, kP = 64, kN = 128;
constexpr int kThreads = 256;
constexpr uint32_t kTileLP = kL * kP * 2;   // 8 KB
constexpr uint32_t kTileLN = kL * kN * 2;   // 16 KB
constexpr uint32_t kTileNP = kN * kP * 2;   // 16 KB
constexpr uint32_t kTmemCols = 512;

struct alignas(1024) BwdSmem {
  uint8_t x[kTileLP];       // [t][p]
  uint8_t dy[kTileLP];      // [t][p]
  uint8_t B[kTileLN];       // [n atom][t][64]
  uint8_t C[kTileLN];
  uint8_t v[kTileLP];       // dt' x               [s][p]
  uint8_t dvd[kTileLP];     // exp(cum_end-cum) v  [s][p]
  uint8_t dch[kTileLP];     // exp(cum) dy         [t][p]
  uint8_t W[kTileLP];       // [t][s]
  uint8_t dCB[kTileLP];     // [t][s]
  uint8_t S[kTileNP];       // S_c^T bf16 [n][p]
  uint8_t dS[2][kTileNP];   // dS^T bf16 [n][p], double-buffered
  uint8_t dx[kTileLP];      // output staging [t][p]
  float ddiff[kL][kL + 1];  // d_diff, padded
  float cum[kL], ecum[kL], dec[kL], dtp[kL], z[kL];
  float dcb[2][kL], dde[2][kL], dvx[2][kL];
  float drow[kL], dcol[kL], dda[kL];
  float wsum[2];
  float red[kThreads / 32];
  uint64_t bar_in, bar_s, bar_mma1, bar_mma2;
  uint32_t tmem_slot;
};

struct BwdParams {
  const float* dt_raw;
  const float* A;
  const float* s0;
  const float* ds_final;
  float* ddt_raw;
  float* ds0;
  float* dB_part;  // [b,T,H,N]
  float* dC_part;  // [b,T,H,N]
  float* dA_part;  // [b,H,nc]
  int* status;
  int T, H, hpg, nc;
};

__device__ __forceinline__ uint64_t kdesc(const void* tile, int rows, int kk) {
  return sdesc_sw128(smem_u32(tile) + (kk >> 6) * rows * 128 + (kk & 63) * 2, 0, 1024);
}
__device__ __forceinline__ uint64_t mdesc(const void* tile, int krows, int kk) {
  return sdesc_sw128(smem_u32(tile) + kk * 128, krows * 128, 1024);
}

// K1 for chunk c: cum, ecum = exp(cum), dec = exp(cum_end - cum), dtp = dt'
// (threads 0..63); returns nothing, leaves wsum = the two warp totals.
__device__ __forceinline__ void chunk_scalars(BwdSmem& sm, const BwdParams& prm, int row0, int h, int c, float A_h) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < kL) {
    const float z = prm.dt_raw[((size_t)row0 + c * kL + tid) * prm.H + h];
    const float d = softplus_f(z);
    float cs = d * A_h;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, cs, o);
      if (lane >= o) cs += u;
    }
    sm.z[tid] = z;
    sm.dtp[tid] = d;
    sm.cum[tid] = cs;
    if (lane == 31) sm.wsum[warp] = cs;
  }
  __syncthreads();
  if (tid < kL) {
    const float cs = sm.cum[tid] + (warp == 1 ? sm.wsum[0] : 0.f);
    const float cend = sm.wsum[0] + sm.wsum[1];
    sm.cum[tid] = cs;
    sm.ecum[tid] = expf(cs);
    sm.dec[tid] = expf(cend - cs);
  }
  __syncthreads();
}

__device__ __forceinline__ void store_row_bf16(uint8_t* tile, int row, int chunk0, const float* v, int nchunks) {
  for (int j = 0; j < nchunks; ++j) {
    uint4 w;
    w.x = pack_bf16(v[8 * j + 0], v[8 * j + 1]);
    w.y = pack_bf16(v[8 * j + 2], v[8 * j + 3]);
    w.z = pack_bf16(v[8 * j + 4], v[8 * j + 5]);
    w.w = pack_bf16(v[8 * j + 6], v[8 * j + 7]);
    *reinterpret_cast<uint4*>(tile + sw128_chunk(row, chunk0 + j)) = w;
  }
}

// Reads 8 bf16 values of row r, 16-byte chunk j of a 128-byte-row SW128 tile.
__device__ __forceinline__ void load_chunk(const uint8_t* tile, int r, int j, float* out) {
  const uint4 raw = *reinterpret_cast<const uint4*>(tile + sw128_chunk(r, j));
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = unpack_bf16(w[i]);
    out[2 * i] = f.x;
    out[2 * i + 1] = f.y;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    k_tc_bwd(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
             const __grid_constant__ CUtensorMap tm_dx, const __grid_constant__ CUtensorMap tm_B,
             const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_S, BwdParams prm) {
  extern __shared__ uint8_t smem_raw[];
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = warp & 3, hh = warp >> 2;  // TMEM lane quadrant, column half
  const int h = blockIdx.x, b = blockIdx.y;
  const int T = prm.T, H = prm.H, nc = prm.nc;
  const int g = h / prm.hpg;
  const float A_h = prm.A[h];
  const int row0 = b * T;
  const size_t unit = (size_t)b * H + h;
  const int srow0 = (int)(unit * nc) * kN;  // first row of this unit's states in the workspace view

  if (tid == 0) {
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_dy);
    prefetch_tmap(&tm_dx);
    prefetch_tmap(&tm_B);
    prefetch_tmap(&tm_C);
    prefetch_tmap(&tm_S);
    mbar_init(&sm.bar_in, 1);
    mbar_init(&sm.bar_s, 1);
    mbar_init(&sm.bar_mma1, 1);
    mbar_init(&sm.bar_mma2, 1);
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(&sm.tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  const uint32_t T1 = tmem;         // intra^T (replay) / dS_blue^T   M = 128, 64 cols
  const uint32_t T2 = tmem + 64;    // dC [t][n]                      M = 64, 128 cols
  const uint32_t T3 = tmem + 192;   // dW [t][s], then dB (with T4)    M = 64
  const uint32_t T4 = tmem + 256;   // CB [t][s]                       M = 64
  const uint32_t T5 = tmem + 320;   // dv_orange [s][p]                M = 64
  const uint32_t T6 = tmem + 384;   // d_decayed_v [s][p]              M = 64
  const uint32_t T7 = T3;           // dB [s][n]                       M = 64, 128 cols

  // thread (q, hh, lane) owns state row n = 32q + lane, columns p in [32hh, 32hh + 32)
  const int n_own = 32 * q + lane;
  const int p0 = 32 * hh;
  float R[32];
  const size_t sbase = unit * kP * kN;
  uint32_t ph_in = 0, ph_s = 0, ph1 = 0, ph2 = 0;
  bool ok = true;

  // ================================================================ reverse
  // dS = ds_final (fp32 registers) and its bf16 tile
#pragma unroll
  for (int i = 0; i < 32; ++i) R[i] = prm.ds_final[sbase + (size_t)(p0 + i) * kN + n_own];
  int dsb = 0;
  store_row_bf16(sm.dS[dsb], n_own, 4 * hh, R, 4);
  for (int c = (ok ? nc - 1 : -1); c >= 0; --c) {
    const int t0 = c * kL;
    if (tid == 0) {
      fence_proxy_async();
      mbar_expect_tx(&sm.bar_in, 2 * kTileLP + 2 * kTileLN);
      tma_load_2d(sm.x, &tm_x, h * kP, row0 + t0, &sm.bar_in);
      tma_load_2d(sm.dy, &tm_dy, h * kP, row0 + t0, &sm.bar_in);
      for (int a = 0; a < 2; ++a) {
        tma_load_3d(sm.B + a * (kTileLN / 2), &tm_B, a * 64, g, row0 + t0, &sm.bar_in);
        tma_load_3d(sm.C + a * (kTileLN / 2), &tm_C, a * 64, g, row0 + t0, &sm.bar_in);
      }
      mbar_expect_tx(&sm.bar_s, kTileNP);
      tma_load_2d(sm.S, &tm_S, 0, srow0 + c * kN, &sm.bar_s);
    }
    if (tid == 128) tma_store_wait_read0();  // previous dx tile read out
    chunk_scalars(sm, prm, row0, h, c, A_h);
    ok = mbar_wait(&sm.bar_in, ph_in, prm.status, 13);
    ph_in ^= 1;
    // v = dt' x, dvd = exp(cum_end - cum) v, dch = exp(cum) dy
    for (int ch = tid; ch < kL * 8; ch += kThreads) {
      const int t = ch >> 3, j = ch & 7;
      float f[8], gy[8];
      load_chunk(sm.x, t, j, f);
      load_chunk(sm.dy, t, j, gy);
      const float d = sm.dtp[t], e = sm.dec[t], ec = sm.ecum[t];
      uint4 wv, wd, wc;
      uint32_t* pv = &wv.x;
      uint32_t* pd = &wd.x;
      uint32_t* pc = &wc.x;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float v0 = d * f[2 * i], v1 = d * f[2 * i + 1];
        pv[i] = pack_bf16(v0, v1);
        pd[i] = pack_bf16(e * v0, e * v1);
        pc[i] = pack_bf16(ec * gy[2 * i], ec * gy[2 * i + 1]);
      }
      const uint32_t off = sw128_chunk(t, j);
      *reinterpret_cast<uint4*>(sm.v + off) = wv;
      *reinterpret_cast<uint4*>(sm.dvd + off) = wd;
      *reinterpret_cast<uint4*>(sm.dch + off) = wc;
    }
    ok = mbar_wait(&sm.bar_s, ph_s, prm.status, 14) && ok;
    ph_s ^= 1;
    fence_proxy_async();
    if (__syncthreads_or(!ok)) break;
    // ---- batch 1: CB, dW, dS_blue^T, dC_blue, d_decayed_v
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kN; kk += 16)  // CB[t][s] = sum_n C[t][n] B[s][n]
        mma_bf16(T4, kdesc(sm.C, kL, kk), kdesc(sm.B, kL, kk), idesc_bf16(64, 64, false, false), kk > 0);
#pragma unroll
      for (int kk = 0; kk < kP; kk += 16)  // dW[t][s] = sum_p dy[t][p] v[s][p]
        mma_bf16(T3, kdesc(sm.dy, kL, kk), kdesc(sm.v, kL, kk), idesc_bf16(64, 64, false, false), kk > 0);
#pragma unroll
      for (int kk = 0; kk < kL; kk += 16)  // dS_blue^T[n][p] = sum_t C[t][n] dch[t][p]
        mma_bf16(T1, mdesc(sm.C, kL, kk), mdesc(sm.dch, kL, kk), idesc_bf16(128, 64, true, true), kk > 0);
#pragma unroll
      for (int kk = 0; kk < kP; kk += 16)  // dC_blue[t][n] = sum_p dch[t][p] S[n][p]
        mma_bf16(T2, kdesc(sm.dch, kL, kk), kdesc(sm.S, kN, kk), idesc_bf16(64, 128, false, false), kk > 0);
#pragma unroll
      for (int kk = 0; kk < kN; kk += 16)  // ddv[s][p] = sum_n B[s][n] dS[n][p]
        mma_bf16(T6, kdesc(sm.B, kL, kk), mdesc(sm.dS[dsb], kN, kk), idesc_bf16(64, 64, false, true), kk > 0);
      mma_commit(&sm.bar_mma1);
    }
    ok = mbar_wait(&sm.bar_mma1, ph1, prm.status, 15);
    ph1 ^= 1;
    tc_fence_after();
    // ---- E1: W, dCB, d_diff from dW (T3) and CB (T4); BLUE d cum from dC_blue (T2);
    //          K3 decay gradient from ddv (T6); K4 term and the dS update from dS_blue^T (T1)
    {
      float dw[32], cb[32];
      tmem_ld32(taddr(T3, 32 * q, 32 * hh), dw);
      tmem_ld32(taddr(T4, 32 * q, 32 * hh), cb);
      if (lane < 16) {
        const int t = 16 * q + lane;
        const float ct = sm.cum[t];
        float w[32], dcbv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int s = 32 * hh + i;
          const float dec = (s <= t) ? expf(ct - sm.cum[s]) : 0.f;
          w[i] = cb[i] * dec;
          dcbv[i] = dw[i] * dec;
          sm.ddiff[t][s] = dcbv[i] * cb[i];
        }
        store_row_bf16(sm.W, t, 4 * hh, w, 4);
        store_row_bf16(sm.dCB, t, 4 * hh, dcbv, 4);
      }
    }
    {
      float dc[32];
      float acc = 0.f;
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        tmem_ld32(taddr(T2, 32 * q, 64 * hh + 32 * part), dc);
        if (lane < 16) {
          const int t = 16 * q + lane;
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int n = 64 * hh + 32 * part + 8 * jj;  // C[t][n..n+7]: atom n/64, chunk (n%64)/8
            float cv[8];
            load_chunk(sm.C + (n >> 6) * (kTileLN / 2), t, (n & 63) >> 3, cv);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc += cv[i] * dc[8 * jj + i];
          }
        }
      }
      if (lane < 16) sm.dcb[hh][16 * q + lane] = acc;
    }
    {
      float ddv[32];
      tmem_ld32(taddr(T6, 32 * q, 32 * hh), ddv);
      if (lane < 16) {
        const int s = 16 * q + lane;
        float acc = 0.f;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          float xv[8];
          load_chunk(sm.x, s, 4 * hh + jj, xv);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc += ddv[8 * jj + i] * xv[i];
        }
        sm.dde[hh][s] = acc * sm.dtp[s];  // sum_p ddv[s][p] v[s][p]
      }
    }
    {
      // K4: <dS_{c+1}, S_c> (S_c from its bf16 tile), then dS_c = a dS_{c+1} + dS_blue
      float sv[32], bl[32];
      load_chunk(sm.S, n_own, 4 * hh + 0, sv);
      load_chunk(sm.S, n_own, 4 * hh + 1, sv + 8);
      load_chunk(sm.S, n_own, 4 * hh + 2, sv + 16);
      load_chunk(sm.S, n_own, 4 * hh + 3, sv + 24);
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) part += R[i] * sv[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if (lane == 0) sm.red[warp] = part;
      tmem_ld32(taddr(T1, 32 * q, p0), bl);
      const float a = expf(sm.wsum[0] + sm.wsum[1]);
#pragma unroll
      for (int i = 0; i < 32; ++i) R[i] = a * R[i] + bl[i];
      store_row_bf16(sm.dS[dsb ^ 1], n_own, 4 * hh, R, 4);
    }
    tc_fence_before();
    fence_proxy_async();
    if (__syncthreads_or(!ok)) break;
    // ---- batch 2: dv_orange, dC += dCB B, dB = dvd dS^T + dCB^T C
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kL; kk += 16)  // dv_or[s][p] = sum_t W[t][s] dy[t][p]
        mma_bf16(T5, mdesc(sm.W, kL, kk), mdesc(sm.dy, kL, kk), idesc_bf16(64, 64, true, true), kk > 0);
#pragma unroll
      for (int kk = 0; kk < kL; kk += 16)  // dC[t][n] += sum_s dCB[t][s] B[s][n]
        mma_bf16(T2, kdesc(sm.dCB, kL, kk), mdesc(sm.B, kL, kk), idesc_bf16(64, 128, false, true), true);
#pragma unroll
      for (int kk = 0; kk < kP; kk += 16)  // dB[s][n] = sum_p dvd[s][p] dS[n][p]
        mma_bf16(T7, kdesc(sm.dvd, kL, kk), kdesc(sm.dS[dsb], kN, kk), idesc_bf16(64, 128, false, false), kk > 0);
#pragma unroll
      for (int kk = 0; kk < kL; kk += 16)  // dB[s][n] += sum_t dCB[t][s] C[t][n]
        mma_bf16(T7, mdesc(sm.dCB, kL, kk), mdesc(sm.C, kL, kk), idesc_bf16(64, 128, true, true), true);
      mma_commit(&sm.bar_mma2);
    }
    // ORANGE row / column sums of d_diff (fixed order)
    if (tid < kL) {
      float r = 0.f;
      for (int s = 0; s < kL; ++s) r += sm.ddiff[tid][s];
      sm.drow[tid] = r;
    } else if (tid < 2 * kL) {
      const int s = tid - kL;
      float cc = 0.f;
      for (int t = 0; t < kL; ++t) cc += sm.ddiff[t][s];
      sm.dcol[s] = cc;
    }
    ok = mbar_wait(&sm.bar_mma2, ph2, prm.status, 16);
    ph2 ^= 1;
    tc_fence_after();
    // ---- E2: dC, dB per head (fp32), dv -> dx and sum_p dv x
    {
      float acc[32];
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        tmem_ld32(taddr(T2, 32 * q, 64 * hh + 32 * part), acc);
        if (lane < 16) {
          const int t = 16 * q + lane;
          float4* dst = reinterpret_cast<float4*>(prm.dC_part + (((size_t)row0 + t0 + t) * H + h) * kN + 64 * hh +
                                                  32 * part);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
        }
        tmem_ld32(taddr(T7, 32 * q, 64 * hh + 32 * part), acc);
        if (lane < 16) {
          const int s = 16 * q + lane;
          float4* dst = reinterpret_cast<float4*>(prm.dB_part + (((size_t)row0 + t0 + s) * H + h) * kN + 64 * hh +
                                                  32 * part);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
        }
      }
    }
    {
      float dvo[32], ddv[32];
      tmem_ld32(taddr(T5, 32 * q, 32 * hh), dvo);
      tmem_ld32(taddr(T6, 32 * q, 32 * hh), ddv);
      if (lane < 16) {
        const int s = 16 * q + lane;
        const float e = sm.dec[s], d = sm.dtp[s];
        float dxv[32];
        float accx = 0.f;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          float xv[8];
          load_chunk(sm.x, s, 4 * hh + jj, xv);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float dv = dvo[8 * jj + i] + e * ddv[8 * jj + i];
            accx += dv * xv[i];
            dxv[8 * jj + i] = d * dv;
          }
        }
        sm.dvx[hh][s] = accx;
        store_row_bf16(sm.dx, s, 4 * hh, dxv, 4);
      }
    }
    tc_fence_before();
    fence_proxy_async();
    if (__syncthreads_or(!ok)) break;
    if (tid == 128) {
      tma_store_2d(&tm_dx, sm.dx, h * kP, row0 + t0);
      tma_store_commit();
    }
    // ---- d cum -> K1 backward (suffix sum) -> ddt_raw, dA part
    if (tid == 0) {
      float kd = 0.f;
      for (int w = 0; w < kThreads / 32; ++w) kd += sm.red[w];
      const float a = expf(sm.wsum[0] + sm.wsum[1]);
      float last = a * kd;  // K4
      float suf = 0.f;
      for (int l = kL - 1; l >= 0; --l) {
        const float k3 = (sm.dde[0][l] + sm.dde[1][l]) * sm.dec[l];
        last += k3;
        float dcum = sm.drow[l] - sm.dcol[l] + sm.dcb[0][l] + sm.dcb[1][l] - k3;
        sm.dda[l] = dcum;
      }
      sm.dda[kL - 1] += last;
      for (int l = kL - 1; l >= 0; --l) {
        suf += sm.dda[l];
        sm.dda[l] = suf;
      }
      float acc = 0.f;
      for (int l = 0; l < kL; ++l) acc += sm.dda[l] * sm.dtp[l];
      prm.dA_part[unit * nc + c] = acc;
    }
    __syncthreads();
    if (tid < kL) {
      const float ddtp = sm.dvx[0][tid] + sm.dvx[1][tid] + A_h * sm.dda[tid];
      prm.ddt_raw[((size_t)row0 + t0 + tid) * H + h] = ddtp * sigmoid_f(sm.z[tid]);
    }
    dsb ^= 1;
  }
  if (tid == 128) tma_store_wait0();
#pragma unroll
  for (int i = 0; i < 32; ++i) prm.ds0[sbase + (size_t)(p0 + i) * kN + n_own] = R[i];
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename TOut>
__global__ void k_tc_group_sum(const float* part, TOut* out, int b, int T, int H, int G, int N) {
  const size_t total = (size_t)b * T * G * N;
  const int hpg = H / G;
  for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int n = e % N;
    const size_t bt = e / N / G;
    const int gg = (e / N) % G;
    float acc = 0.f;
    for (int k = 0; k < hpg; ++k) acc += part[(bt * H + gg * hpg + k) * N + n];
    st(out, e, acc);
  }
}

__global__ void k_tc_dA_sum(const float* part, float* dA, int b, int H, int nc) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= H) return;
  float acc = 0.f;
  for (int bb = 0; bb < b; ++bb)
    for (int c = 0; c < nc; ++c) acc += part[((size_t)bb * H + h) * nc + c];
  dA[h] = acc;
}

struct TcBwdWs {
  __nv_bfloat16* states;  // [b,H,nc][N][P]
  float* dB_part;
  float* dC_part;
  float* dA_part;
};

TcBwdWs carve(const Dims& d, Carver& cv) {
  TcBwdWs w;
  w.states = cv.take<__nv_bfloat16>((size_t)d.b * d.H * d.nc * kN * kP);
  w.dB_part = cv.take<float>((size_t)d.b * d.T * d.H * kN);
  w.dC_part = cv.take<float>((size_t)d.b * d.T * d.H * kN);
  w.dA_part = cv.take<float>((size_t)d.b * d.H * d.nc);
  return w;
}

}  // namespace

bool tc_backward_supported(const Dims& d) { return tc_forward_supported(d); }

size_t tc_backward_ws(const Dims& d) {
  Carver cv(nullptr);
  carve(d, cv);
  return cv.off;
}

cudaError_t tc_backward(const Dims& d, const BwdArgs& a, void* ws, cudaStream_t st) {
  Carver cv(ws);
  TcBwdWs w = carve(d, cv);
  const uint64_t rows = (uint64_t)d.b * d.T;
  CUtensorMap tx, tdy, tdx, tb, tcm, ts;
  cudaError_t e = tc_replay_states(d, a.x, a.dt_raw, a.A, a.B, a.s0, w.states, static_cast<int*>(ws), st);
  if (e == cudaSuccess) e = make_tmap_2d_bf16(&tx, a.x, (uint64_t)d.H * kP, rows, 64, 64);
  if (e == cudaSuccess) e = make_tmap_2d_bf16(&tdy, a.dy, (uint64_t)d.H * kP, rows, 64, 64);
  if (e == cudaSuccess) e = make_tmap_2d_bf16(&tdx, a.dx, (uint64_t)d.H * kP, rows, 64, 64);
  if (e == cudaSuccess) e = make_tmap_3d_bf16(&tb, a.B, d.N, d.G, rows, 64, 1, 64);
  if (e == cudaSuccess) e = make_tmap_3d_bf16(&tcm, a.C, d.N, d.G, rows, 64, 1, 64);
  if (e == cudaSuccess)
    e = make_tmap_2d_bf16(&ts, w.states, kP, (uint64_t)d.b * d.H * d.nc * kN, 64, kN);
  if (e != cudaSuccess) return e;
  BwdParams prm{a.dt_raw, a.A, a.s0, a.ds_final, a.ddt_raw, a.ds0, w.dB_part, w.dC_part, w.dA_part,
                static_cast<int*>(ws), d.T, d.H, d.hpg, d.nc};
  const int smem = (int)sizeof(BwdSmem) + 1024;
  e = cudaFuncSetAttribute(k_tc_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  SSD_LAUNCH("k_tc_bwd", st, k_tc_bwd<<<dim3(d.H, d.b), kThreads, smem, st>>>(tx, tdy, tdx, tb, tcm, ts, prm));
  const size_t tot = (size_t)d.b * d.T * d.G * d.N;
  const int blocks = (int)((tot + 255) / 256 < 65535 ? (tot + 255) / 256 : 65535);
  SSD_LAUNCH("k_tc_group_sum", st,
             k_tc_group_sum<__nv_bfloat16><<<blocks, 256, 0, st>>>(w.dB_part, static_cast<__nv_bfloat16*>(a.dB), d.b,
                                                                   d.T, d.H, d.G, d.N));
  SSD_LAUNCH("k_tc_group_sum", st,
             k_tc_group_sum<__nv_bfloat16><<<blocks, 256, 0, st>>>(w.dC_part, static_cast<__nv_bfloat16*>(a.dC), d.b,
                                                                   d.T, d.H, d.G, d.N));
  SSD_LAUNCH("k_tc_dA_sum", st, k_tc_dA_sum<<<(d.H + 127) / 128, 128, 0, st>>>(w.dA_part, a.dA, d.b, d.H, d.nc));
  return cudaGetLastError();
}

}  // namespace ssd
