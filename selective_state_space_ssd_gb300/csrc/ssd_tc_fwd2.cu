// Warp-specialized, software-pipelined chunkwise forward of the Mamba-2 scan
// on tcgen05 tensor cores (bf16 io, chunk L = 64, head dim P = 64, state
// N = 128), and its "states" mode used as the replay of the recompute
// backward.
//
// One CTA owns one (batch, head) and walks its chunks in order (the K4 state
// passing of the burn-mamba page "combined_backward.rs" stays in fp32
// registers).  Per chunk c, with cum = in-chunk cumsum of da = dt' A (K1):
//   intra^T = B^T dvd,   dvd[s][p] = exp(cum_end - cum_s) dt'_s x[s][p]   (K3)
//   y_diag  = W' x,      W'[t][s]  = CB[t][s] exp(cum_t - cum_s) dt'_s [s<=t]
//   y_off   = C S_c^T                                                      (K5)
//   y       = exp(cum_t) y_off + y_diag,   S_{c+1} = exp(cum_end) S_c + intra
// The mask is applied before the exponential ("ORANGE backward": -inf is added
// before exp).  CB = C B^T comes from a small pre-pass (fp32, L2-resident).
//
// Warp roles (480 threads), all running concurrently on different chunks:
//   warps 0-7   epilogue: the fp32 state update from intra^T (each thread
//               owns half a state row), the bf16 S tile for the next y_off
//               MMA, and (forward) y = exp(cum) y_off + y_diag stored by TMA,
//               or (states mode) the S_c tile stored by TMA.
//   warps 8-11  tiles: the bf16 operand tiles dvd and W' of a chunk.
//   warp 12     K1: softplus, da, the in-chunk scan and the decay factors,
//               up to four chunks ahead of the tiles.
//   warp 13     TMA producer: x, B, C tiles into a two-stage ring.
//   warp 14     MMA issuer (one thread) and TMEM owner.
// Accumulators are double-buffered in TMEM so chunk c+1's MMAs overlap chunk
// c's epilogue.  Every wait is bounded; on timeout the kernel records a code
// in the workspace status word and stops issuing work.
#include "ssd_device.cuh"
#include "ssd_internal.h"
#include "tc_common.cuh"

namespace ssd {
namespace {
using namespace tc;

constexpr int kL = 64, kP = 64, kN = 128;
constexpr int kStages = 2;
constexpr int kScal = 4;  // chunks of K1 scalars in flight
constexpr int kThreads = 480;
constexpr int kWarpTile0 = 8, kWarpScal = 12, kWarpTma = 13, kWarpMma = 14;
constexpr uint32_t kTileLP = kL * kP * 2;  // 8 KB
constexpr uint32_t kTileLN = kL * kN * 2;  // 16 KB
constexpr uint32_t kTileNP = kN * kP * 2;  // 16 KB
constexpr uint32_t kTmemCols = 512;

struct alignas(1024) Fwd2Smem {
  uint8_t x[kStages][kTileLP];
  uint8_t B[kStages][kTileLN];
  uint8_t C[kStages][kTileLN];
  uint8_t dvd[2][kTileLP];
  uint8_t W[2][kTileLP];
  uint8_t S[2][kTileNP];
  uint8_t y[2][kTileLP];
  // K1 scalars, ring of kScal chunks: cum, exp(cum), exp(cum_end - cum), dt',
  // G_s = exp(cum_e(s) - cum_s) dt'_s and E_t[j] = exp(cum_t - cum_e(j)), where
  // e(j) is the last position of 16-block j; exp(cum_t - cum_s) for s in an
  // earlier block than t is E_t[blk(s)] * exp(cum_e - cum_s) (both <= 1).
  float cum[kScal][kL], ecum[kScal][kL], dec[kScal][kL], dtp[kScal][kL], G[kScal][kL], E[kScal][kL][4];
  float aend[kScal];
  uint64_t full[kStages], empty[kStages];
  uint64_t sc_ready[kScal], sc_free[kScal];
  uint64_t pre_done[2], intra_done[2], mma_done[2], s_ready[2], epi_done[2];
  uint32_t tmem_slot;
};

struct Fwd2Params {
  const float* dt_raw;
  const float* A;
  const float* s0;
  const float* CB;  // [b, nc, G, L, L] fp32
  float* s_final;   // forward only
  int* status;
  int T, H, G, hpg, nc;
  int srow_stride;  // states mode: rows of one (b,h) unit in the state view (= nc * N)
};

template <bool kStates>
__global__ void __launch_bounds__(kThreads, 1)
    k_tc_fwd2(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_out,
              const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_C, Fwd2Params prm) {
  extern __shared__ uint8_t smem_raw[];
  Fwd2Smem& sm = *reinterpret_cast<Fwd2Smem*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, b = blockIdx.y;
  const int T = prm.T, H = prm.H, nc = prm.nc;
  const int g = h / prm.hpg;
  const int row0 = b * T;
  int* status = prm.status;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 2);  // pre warps + MMA commit
    }
    for (int j = 0; j < kScal; ++j) {
      mbar_init(&sm.sc_ready[j], 1);
      mbar_init(&sm.sc_free[j], 2);  // tile warps + epilogue warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.pre_done[i], 1);
      mbar_init(&sm.intra_done[i], 1);
      mbar_init(&sm.mma_done[i], 1);
      mbar_init(&sm.s_ready[i], 1);
      mbar_init(&sm.epi_done[i], 1);
    }
    mbar_init_fence();
  }
  if (warp == kWarpMma) tmem_alloc(&sm.tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  // per slot i: intra^T (M=128, 64 cols), y_diag, y_off (M=64, 64 cols each)
  auto T_INTRA = [&](int i) { return tmem + 64u * i; };
  auto T_YD = [&](int i) { return tmem + 128u + 64u * i; };
  auto T_YO = [&](int i) { return tmem + 256u + 64u * i; };

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_x);
      prefetch_tmap(&tm_B);
      if (!kStates) prefetch_tmap(&tm_C);
      for (int c = 0; c < nc; ++c) {
        const int s = c % kStages, k = c / kStages;
        if (k > 0 && !mbar_wait(&sm.empty[s], (k - 1) & 1, status, 21)) break;
        const uint32_t bytes = kTileLP + kTileLN + (kStates ? 0 : kTileLN);
        mbar_expect_tx(&sm.full[s], bytes);
        tma_load_2d(sm.x[s], &tm_x, h * kP, row0 + c * kL, &sm.full[s]);
        for (int a = 0; a < 2; ++a) {
          tma_load_3d(sm.B[s] + a * (kTileLN / 2), &tm_B, a * 64, g, row0 + c * kL, &sm.full[s]);
          if (!kStates) tma_load_3d(sm.C[s] + a * (kTileLN / 2), &tm_C, a * 64, g, row0 + c * kL, &sm.full[s]);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      for (int c = 0; c < nc; ++c) {
        const int s = c % kStages, i = c & 1, k = c >> 1;
        bool ok = mbar_wait(&sm.pre_done[i], k & 1, status, 22);  // implies the stage landed
        if (ok && c >= 2) ok = mbar_wait(&sm.epi_done[i], (k - 1) & 1, status, 23);
        if (!ok) break;
        tc_fence_after();
        {
          constexpr uint32_t id = idesc_bf16(128, 64, true, true);
#pragma unroll
          for (int kk = 0; kk < kL; kk += 16)
            mma_bf16(T_INTRA(i), mdesc(sm.B[s], kL, kk), mdesc(sm.dvd[i], kL, kk), id, kk > 0);
        }
        if (!kStates) {
          constexpr uint32_t id = idesc_bf16(64, 64, false, true);
#pragma unroll
          for (int kk = 0; kk < kL; kk += 16)
            mma_bf16(T_YD(i), kdesc(sm.W[i], kL, kk), mdesc(sm.x[s], kL, kk), id, kk > 0);
        }
        mma_commit(&sm.intra_done[i]);
        if (!kStates) {
          if (!mbar_wait(&sm.s_ready[i], k & 1, status, 24)) break;
          tc_fence_after();
          constexpr uint32_t id = idesc_bf16(64, 64, false, true);
#pragma unroll
          for (int kk = 0; kk < kN; kk += 16)
            mma_bf16(T_YO(i), kdesc(sm.C[s], kL, kk), mdesc(sm.S[i], kN, kk), id, kk > 0);
        }
        mma_commit(&sm.mma_done[i]);
        mma_commit(&sm.empty[s]);
      }
    }
  } else if (warp == kWarpScal) {
    // ------------------------------------------------------------ K1 scalar warp
    // lane l handles positions 2l and 2l+1 of the chunk
    const float A_h = prm.A[h];
    auto load_z = [&](int c) {
      const size_t r0 = (size_t)row0 + c * kL + 2 * lane;
      return make_float2(prm.dt_raw[r0 * H + h], prm.dt_raw[(r0 + 1) * H + h]);
    };
    float2 z_next = load_z(0);
    for (int c = 0; c < nc; ++c) {
      const int j = c % kScal, k = c / kScal;
      if (c >= kScal && !mbar_wait(&sm.sc_free[j], (k - 1) & 1, status, 31)) break;
      const float2 z = z_next;
      if (c + 1 < nc) z_next = load_z(c + 1);
      const float d0 = softplus_f(z.x), d1 = softplus_f(z.y);
      const float a0 = d0 * A_h, a1 = a0 + d1 * A_h;  // local inclusive sums of the pair
      float inc = a1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      const float base = inc - a1;  // exclusive prefix of this pair
      const float c0 = base + a0, c1 = inc;
      const float cend = __shfl_sync(0xffffffffu, inc, 31);
      const int t0 = 2 * lane, t1 = t0 + 1;
      sm.cum[j][t0] = c0;
      sm.cum[j][t1] = c1;
      sm.dtp[j][t0] = d0;
      sm.dtp[j][t1] = d1;
      sm.ecum[j][t0] = expf(c0);
      sm.ecum[j][t1] = expf(c1);
      sm.dec[j][t0] = expf(cend - c0);
      sm.dec[j][t1] = expf(cend - c1);
      if (lane == 0) sm.aend[j] = expf(cend);
      // block ends: positions 15, 31, 47, 63 live in lanes 7, 15, 23, 31 (as c1)
      const float e0 = __shfl_sync(0xffffffffu, c1, 7), e1 = __shfl_sync(0xffffffffu, c1, 15);
      const float e2 = __shfl_sync(0xffffffffu, c1, 23), e3 = __shfl_sync(0xffffffffu, c1, 31);
      const int blk = t0 >> 4;  // t0 and t1 are in the same 16-block
      const float my_end = blk == 0 ? e0 : (blk == 1 ? e1 : (blk == 2 ? e2 : e3));
      const float ends[4] = {e0, e1, e2, e3};
      sm.G[j][t0] = expf(my_end - c0) * d0;
      sm.G[j][t1] = expf(my_end - c1) * d1;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        sm.E[j][t0][q] = (q < (t0 >> 4)) ? expf(c0 - ends[q]) : 0.f;
        sm.E[j][t1][q] = (q < (t1 >> 4)) ? expf(c1 - ends[q]) : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.sc_ready[j]);
    }
  } else if (warp >= kWarpTile0) {
    // ------------------------------------------------------------ tile warps 8-11
    const int pt = tid - 32 * kWarpTile0;  // 0..127
    const int wt = pt >> 1, whalf = pt & 1;  // W' row and 32-column half
    auto cb_ptr = [&](int c) {
      return reinterpret_cast<const float4*>(prm.CB + ((((size_t)b * nc + c) * prm.G + g) * kL + wt) * kL + 32 * whalf);
    };
    float4 cb_next[8];
    if (!kStates) {
#pragma unroll
      for (int q = 0; q < 8; ++q) cb_next[q] = __ldg(cb_ptr(0) + q);
    }
    for (int c = 0; c < nc; ++c) {
      const int s = c % kStages, i = c & 1, k = c >> 1, j = c % kScal;
      float4 cbv[8];
      if (!kStates) {
#pragma unroll
        for (int q = 0; q < 8; ++q) cbv[q] = cb_next[q];
        if (c + 1 < nc) {
#pragma unroll
          for (int q = 0; q < 8; ++q) cb_next[q] = __ldg(cb_ptr(c + 1) + q);
        }
      }
      bool ok = mbar_wait(&sm.sc_ready[j], (c / kScal) & 1, status, 32);
      ok = ok && mbar_wait(&sm.full[s], (c / kStages) & 1, status, 26);
      // tile slot i was last read by chunk c-2's intra and y_diag MMAs
      if (ok && c >= 2) ok = mbar_wait(&sm.intra_done[i], (k - 1) & 1, status, 33);
      if (named_bar_or(2, 128, !ok)) break;
      // dvd[s][p] = exp(cum_end - cum_s) dt'_s x[s][p]  (same swizzled positions as x)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int ch = pt + 128 * r;
        const int t = ch >> 3, jj = ch & 7;
        const uint32_t off = sw128_chunk(t, jj);
        const uint4 raw = *reinterpret_cast<const uint4*>(sm.x[s] + off);
        const float f = sm.dec[j][t] * sm.dtp[j][t];
        const uint32_t in[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 v = unpack_bf16(in[e]);
          o[e] = pack_bf16(f * v.x, f * v.y);
        }
        *reinterpret_cast<uint4*>(sm.dvd[i] + off) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      if (!kStates) {
        // W'[t][s] = CB[t][s] exp(cum_t - cum_s) dt'_s for s <= t, else 0.  The 32
        // columns of this thread are two 16-blocks; the case (earlier block,
        // diagonal block, later block) is uniform over a block.
        const int t = wt, tb = t >> 4;
        const float ct = sm.cum[j][t];
        float w[32];
        float cb[32];
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) {
          cb[4 * qq + 0] = cbv[qq].x;
          cb[4 * qq + 1] = cbv[qq].y;
          cb[4 * qq + 2] = cbv[qq].z;
          cb[4 * qq + 3] = cbv[qq].w;
        }
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const int sb = 2 * whalf + bb, s0 = 16 * sb;
          if (sb < tb) {
            const float f = sm.E[j][t][sb];  // exp(cum_t - cum at the end of block sb)
#pragma unroll
            for (int e = 0; e < 16; ++e) w[16 * bb + e] = cb[16 * bb + e] * (f * sm.G[j][s0 + e]);
          } else if (sb == tb) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int ss = s0 + e;
              const float dec = expf(fminf(ct - sm.cum[j][ss], 0.f)) * sm.dtp[j][ss];
              w[16 * bb + e] = (ss <= t) ? cb[16 * bb + e] * dec : 0.f;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) w[16 * bb + e] = 0.f;
          }
        }
        store_row_bf16(sm.W[i], t, 4 * whalf, w, 4);
      }
      fence_proxy_async();
      named_bar(2, 128);
      if (pt == 0) {
        mbar_arrive(&sm.pre_done[i]);
        mbar_arrive(&sm.empty[s]);
        mbar_arrive(&sm.sc_free[j]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps 0-7
    // thread ct owns state row n = 32*(warp%4) + lane, columns p in [32*half, 32*half + 32)
    const int ct = tid;
    const int q = warp & 3, half = warp >> 2;
    const int n = 32 * q + lane, p0 = 32 * half;
    const size_t sbase = (((size_t)b * H + h) * kP) * kN;
    float S[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) S[e] = prm.s0 ? prm.s0[sbase + (size_t)(p0 + e) * kN + n] : 0.f;
    store_row_bf16(sm.S[0], n, 4 * half, S, 4);
    fence_proxy_async();
    named_bar(1, 256);
    if (ct == 0) {
      prefetch_tmap(&tm_out);
      mbar_arrive(&sm.s_ready[0]);
      if (kStates) {
        tma_store_2d(&tm_out, sm.S[0], 0, (int)(((size_t)b * H + h) * prm.srow_stride));
        tma_store_commit();
      }
    }
    for (int c = 0; c < nc; ++c) {
      const int i = c & 1, k = c >> 1, i1 = (c + 1) & 1, j = c % kScal;
      bool ok = mbar_wait(&sm.intra_done[i], k & 1, status, 27);
      ok = ok && mbar_wait(&sm.sc_ready[j], (c / kScal) & 1, status, 28);
      if (named_bar_or(1, 256, !ok)) break;
      tc_fence_after();
      // ---- K4: S_{c+1} = exp(cum_end) S_c + intra   (row n, columns p0..p0+31)
      {
        const float a = sm.aend[j];
        float iv[32];
        tmem_ld32(taddr(T_INTRA(i), 32 * q, p0), iv);
#pragma unroll
        for (int e = 0; e < 32; ++e) S[e] = a * S[e] + iv[e];
      }
      if (c + 1 < nc) {
        // S tile i1 was last read by y_off(c-1) (waited in epilogue(c-1)) or, in
        // states mode, by the TMA store of S_{c-1}
        if (kStates) {
          if (ct == 0) tma_store_wait_read0();
          named_bar(1, 256);
        }
        store_row_bf16(sm.S[i1], n, 4 * half, S, 4);
        fence_proxy_async();
        named_bar(1, 256);
        if (ct == 0) {
          if (!kStates) mbar_arrive(&sm.s_ready[i1]);
          if (kStates) {
            tma_store_2d(&tm_out, sm.S[i1], 0, (int)(((size_t)b * H + h) * prm.srow_stride + (size_t)(c + 1) * kN));
            tma_store_commit();
          }
        }
      }
      if (!kStates) {
        // ---- y = exp(cum_t) y_off + y_diag  (M = 64 layout: row t in lane t%16 of quadrant t/16)
        ok = mbar_wait(&sm.mma_done[i], k & 1, status, 30);
        if (ct == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");  // y tile i (chunk c-2) read out
        if (named_bar_or(1, 256, !ok)) break;
        tc_fence_after();
        float dg[32], of[32];
        tmem_ld32(taddr(T_YD(i), 32 * q, p0), dg);
        tmem_ld32(taddr(T_YO(i), 32 * q, p0), of);
        if (lane < 16) {
          const int t = 16 * q + lane;
          const float e = sm.ecum[j][t];
          float yv[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) yv[u] = e * of[u] + dg[u];
          store_row_bf16(sm.y[i], t, 4 * half, yv, 4);
        }
        fence_proxy_async();
      }
      tc_fence_before();
      named_bar(1, 256);
      if (ct == 0) {
        mbar_arrive(&sm.epi_done[i]);
        mbar_arrive(&sm.sc_free[j]);
        if (!kStates) {
          tma_store_2d(&tm_out, sm.y[i], h * kP, row0 + c * kL);
          tma_store_commit();
        }
      }
    }
    if (ct == 0) tma_store_wait0();
    if (!kStates) {
#pragma unroll
      for (int e = 0; e < 32; ++e) prm.s_final[sbase + (size_t)(p0 + e) * kN + n] = S[e];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// CB[b][c][g][t][s] = sum_n C[b, c*L+t, g, n] B[b, c*L+s, g, n]  (fp32)
__global__ void __launch_bounds__(256) k_cb(const __nv_bfloat16* B, const __nv_bfloat16* C, float* CB, int T, int G,
                                            int nc) {
  __shared__ float sC[kL][kN + 1];
  __shared__ float sB[kL][kN + 1];
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  for (int e = threadIdx.x; e < kL * kN; e += blockDim.x) {
    const int t = e / kN, n = e % kN;
    const size_t gi = (((size_t)b * T + c * kL + t) * G + g) * kN + n;
    sC[t][n] = __bfloat162float(C[gi]);
    sB[t][n] = __bfloat162float(B[gi]);
  }
  __syncthreads();
  const int t = threadIdx.x >> 2, s0 = threadIdx.x & 3;
  float acc[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.f;
  for (int n = 0; n < kN; ++n) {
    const float cv = sC[t][n];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] += cv * sB[s0 + 4 * j][n];
  }
  float* out = CB + ((((size_t)b * nc + c) * G + g) * kL + t) * kL;
#pragma unroll
  for (int j = 0; j < 16; ++j) out[s0 + 4 * j] = acc[j];
}

}  // namespace

// The tensor-core kernels serve Mamba-2 with bf16 io, chunk 64, head dim 64
// and state 128 (the 130M and 2.7B layer shapes); everything else runs on the
// CUDA-core kernels.
bool tc_forward_supported(const Dims& d) {
  return d.variant == kMamba2 && d.bf16 && d.L == kL && d.P == kP && d.N == kN;
}
// The chunk-parallel backward indexes its (chunk, head) items with 32-bit integers.
bool tc_backward_supported(const Dims& d) {
  return tc_forward_supported(d) && (long long)d.b * d.nc * d.H < (1ll << 31);
}

size_t tc_fwd2_ws(const Dims& d) {
  Carver cv(nullptr);
  cv.take<float>((size_t)d.b * d.nc * d.G * kL * kL);
  return cv.off;
}

cudaError_t tc_cb_prepass(const Dims& d, const void* B, const void* C, float* CB, cudaStream_t st) {
  SSD_LAUNCH("k_cb", st,
             k_cb<<<dim3(d.nc, d.G, d.b), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(B),
                                                        static_cast<const __nv_bfloat16*>(C), CB, d.T, d.G, d.nc));
  return cudaGetLastError();
}

cudaError_t tc_forward2(const Dims& d, const FwdArgs& a, void* ws, cudaStream_t st) {
  Carver cv(ws);
  float* CB = cv.take<float>((size_t)d.b * d.nc * d.G * kL * kL);
  cudaError_t e = tc_cb_prepass(d, a.B, a.C, CB, st);
  if (e != cudaSuccess) return e;
  CUtensorMap tx, ty, tb, tcm;
  const uint64_t rows = (uint64_t)d.b * d.T;
  e = make_tmap_2d_bf16(&tx, a.x, (uint64_t)d.H * d.P, rows, 64, 64);
  if (e == cudaSuccess) e = make_tmap_2d_bf16(&ty, a.y, (uint64_t)d.H * d.P, rows, 64, 64);
  if (e == cudaSuccess) e = make_tmap_3d_bf16(&tb, a.B, d.N, d.G, rows, 64, 1, 64);
  if (e == cudaSuccess) e = make_tmap_3d_bf16(&tcm, a.C, d.N, d.G, rows, 64, 1, 64);
  if (e != cudaSuccess) return e;
  Fwd2Params prm{a.dt_raw, a.A, a.s0, CB, a.s_final, static_cast<int*>(ws), d.T, d.H, d.G, d.hpg, d.nc, 0};
  const int smem = (int)sizeof(Fwd2Smem) + 1024;
  e = cudaFuncSetAttribute(k_tc_fwd2<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  SSD_LAUNCH("k_tc_fwd2", st, k_tc_fwd2<false><<<dim3(d.H, d.b), kThreads, smem, st>>>(tx, ty, tb, tcm, prm));
  return cudaGetLastError();
}

cudaError_t tc_replay_states(const Dims& d, const void* x, const float* dt_raw, const float* A, const void* B,
                             const float* s0, __nv_bfloat16* states, int* status, cudaStream_t st) {
  CUtensorMap tx, ts, tb;
  const uint64_t rows = (uint64_t)d.b * d.T;
  cudaError_t e = make_tmap_2d_bf16(&tx, x, (uint64_t)d.H * d.P, rows, 64, 64);
  if (e == cudaSuccess) e = make_tmap_2d_bf16(&ts, states, kP, (uint64_t)d.b * d.H * d.nc * kN, 64, kN);
  if (e == cudaSuccess) e = make_tmap_3d_bf16(&tb, B, d.N, d.G, rows, 64, 1, 64);
  if (e != cudaSuccess) return e;
  Fwd2Params prm{dt_raw, A, s0, nullptr, nullptr, status, d.T, d.H, d.G, d.hpg, d.nc, d.nc * kN};
  const int smem = (int)sizeof(Fwd2Smem) + 1024;
  e = cudaFuncSetAttribute(k_tc_fwd2<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  SSD_LAUNCH("k_tc_replay", st, k_tc_fwd2<true><<<dim3(d.H, d.b), kThreads, smem, st>>>(tx, ts, tb, tb, prm));
  return cudaGetLastError();
}

}  // namespace ssd
