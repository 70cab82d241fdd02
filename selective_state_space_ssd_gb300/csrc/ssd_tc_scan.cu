// The two sequential state scans of the Mamba-2 chunkwise algorithm on
// tcgen05 tensor cores (bf16 io, chunk L = 64, head dim P = 64, state N = 128).
//
// Forward (the state passing of the "Mamba-2 part III" page, section "The
// state passing step"; the K3 + K4 pair of the burn-mamba page
// "combined_backward.rs"):
//     S_0 = s0,   S_{c+1} = exp(cum_end) S_c + B_c^T dvd_c,
//     dvd[s][p] = exp(cum_end - cum_s) dt'_s x[s][p];
// it writes every chunk-input state S_c (bf16, [n][p] tiles) and S_nc = s_final.
// Reverse (the same recurrence transposed, the K4 backward):
//     dS_nc = ds_final,   dS_c = exp(cum_end) dS_{c+1} + C_c^T dch_c,
//     dch[t][p] = exp(cum_t) dy[t][p];
// it writes dS_{c+1} for every chunk c (bf16 tiles) and dS_0 = ds0.
//
// One CTA owns one (batch, head); three CTAs share an SM.  The fp32 state
// lives in 64 TMEM columns (thread n of the state warps owns row n): per chunk
// the state warps read it, send its bf16 copy out through TMA, scale it by
// exp(cum_end) in place, and the MMA then accumulates the chunk's K^T U into
// the same columns, so the recurrence costs one MMA group and one TMEM round
// trip per chunk.
//
// Warp roles (288 threads): warps 0-3 state, warps 4-5 scale the U tile in
// place (x -> dvd or dy -> dch), warp 6 K1 scalars (softplus, in-chunk cumsum,
// exponentials), warp 7 TMA producer, warp 8 MMA issuer and TMEM owner.
// Every wait is bounded; on a timeout the kernel records a code in the
// workspace status word and stops.
#include "ssd_device.cuh"
#include "ssd_internal.h"
#include "tc_common.cuh"

namespace ssd {
namespace {
using namespace tc;

constexpr int kL = 64, kP = 64, kN = 128;
constexpr int kThreads = 288;
constexpr int kWarpScale0 = 4, kWarpScal = 6, kWarpTma = 7, kWarpMma = 8;
constexpr uint32_t kTileLP = kL * kP * 2;  // 8 KB
constexpr uint32_t kTileLN = kL * kN * 2;  // 16 KB
constexpr uint32_t kTileNP = kN * kP * 2;  // 16 KB
constexpr uint32_t kTmemCols = 64;

struct alignas(1024) ScanSmem {
  uint8_t u[2][kTileLP];  // x or dy [t][p], scaled in place to dvd or dch
  uint8_t k[2][kTileLN];  // B or C [t][n], two 64-column atoms
  uint8_t out[kTileNP];   // bf16 state tile [n][p] on its way out
  float scale[2][kL];     // per-row factor of U: exp(cum_end - cum) dt' or exp(cum)
  float aend[2];          // exp(cum_end)
  uint64_t full[2], empty[2], sc_ready[2], sc_free[2], pre_done[2];
  uint64_t d_ready, mma_done, drain;
  uint32_t tmem_slot;
};

struct ScanParams {
  const float* dt_raw;
  const float* A;
  const float* init;  // s0 or ds_final [b,H,P,N]; s0 may be null (zeros)
  float* fin;         // s_final or ds0 [b,H,P,N]; null: not written
  int* status;
  int T, H, hpg, nc;
};

template <bool kRev>
__global__ void __launch_bounds__(kThreads, 3)
    k_scan(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_out, ScanParams prm) {
  extern __shared__ uint8_t smem_raw[];
  ScanSmem& sm = *reinterpret_cast<ScanSmem*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, b = blockIdx.y;
  const int T = prm.T, H = prm.H, nc = prm.nc;
  const int g = h / prm.hpg;
  const int row0 = b * T;
  const size_t unit = (size_t)b * H + h;
  int* status = prm.status;
  auto chunk_of = [&](int r) { return kRev ? nc - 1 - r : r; };

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);  // MMA commit (it waited for the scale warps)
      mbar_init(&sm.sc_ready[s], 1);
      mbar_init(&sm.sc_free[s], 2);  // scale warps + state warps
      mbar_init(&sm.pre_done[s], 1);
    }
    mbar_init(&sm.d_ready, 1);
    mbar_init(&sm.mma_done, 1);
    mbar_init(&sm.drain, 1);
    mbar_init_fence();
  }
  if (warp == kWarpMma) tmem_alloc(&sm.tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tm_u);
      prefetch_tmap(&tm_k);
      for (int r = 0; r < nc; ++r) {
        const int s = r & 1, c = chunk_of(r);
        if (r >= 2 && !mbar_wait(&sm.empty[s], ((r >> 1) - 1) & 1, status, 81)) break;
        mbar_expect_tx(&sm.full[s], kTileLP + kTileLN);
        tma_load_2d(sm.u[s], &tm_u, h * kP, row0 + c * kL, &sm.full[s]);
        for (int a = 0; a < 2; ++a)
          tma_load_3d(sm.k[s] + a * (kTileLN / 2), &tm_k, a * 64, g, row0 + c * kL, &sm.full[s]);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int r = 0; r < nc && ok; ++r) {
        const int s = r & 1;
        ok = mbar_wait(&sm.pre_done[s], (r >> 1) & 1, status, 82);
        ok = ok && mbar_wait(&sm.d_ready, r & 1, status, 83);
        if (!ok) break;
        tc_fence_after();
        // D[n][p] += sum_t K[t][n] U[t][p]: A = K^T (MN-major), B = U (MN-major)
#pragma unroll
        for (int kk = 0; kk < kL; kk += 16)
          mma_bf16(tmem, mdesc(sm.k[s], kL, kk), mdesc(sm.u[s], kL, kk), idesc_bf16(128, 64, true, true), true);
        mma_commit(&sm.mma_done);
        mma_commit(&sm.empty[s]);
      }
      // nothing may still be writing TMEM when it is freed
      mma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, status, 84);
    }
  } else if (warp == kWarpScal) {
    // ------------------------------------------------------------ K1 scalars
    const float A_h = prm.A[h];
    const int t0 = 2 * lane, t1 = t0 + 1;
    for (int r = 0; r < nc; ++r) {
      const int s = r & 1, c = chunk_of(r);
      if (r >= 2 && !mbar_wait(&sm.sc_free[s], ((r >> 1) - 1) & 1, status, 85)) break;
      const size_t rr = (size_t)row0 + c * kL + t0;
      const float z0 = prm.dt_raw[rr * H + h], z1 = prm.dt_raw[(rr + 1) * H + h];
      const float d0 = softplus_f(z0), d1 = softplus_f(z1);
      const float a0 = d0 * A_h, a1 = a0 + d1 * A_h;
      float inc = a1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      const float c0 = inc - a1 + a0, c1 = inc;
      const float cend = __shfl_sync(0xffffffffu, inc, 31);
      if (kRev) {
        sm.scale[s][t0] = expf(c0);
        sm.scale[s][t1] = expf(c1);
      } else {
        sm.scale[s][t0] = expf(cend - c0) * d0;
        sm.scale[s][t1] = expf(cend - c1) * d1;
      }
      if (lane == 0) sm.aend[s] = expf(cend);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.sc_ready[s]);
    }
  } else if (warp >= kWarpScale0) {
    // ------------------------------------------------------------ scale warps: U *= scale (per row)
    const int pt = tid - 32 * kWarpScale0;  // 0..63
    for (int r = 0; r < nc; ++r) {
      const int s = r & 1;
      bool ok = mbar_wait(&sm.sc_ready[s], (r >> 1) & 1, status, 86);
      ok = ok && mbar_wait(&sm.full[s], (r >> 1) & 1, status, 87);
      if (named_bar_or(2, 64, !ok)) break;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = pt + 64 * i, t = q >> 3, j = q & 7;
        uint4* p = reinterpret_cast<uint4*>(sm.u[s] + sw128_chunk(t, j));
        const uint4 w = *p;
        const float f = sm.scale[s][t];
        const float2 v0 = unpack_bf16(w.x), v1 = unpack_bf16(w.y), v2 = unpack_bf16(w.z), v3 = unpack_bf16(w.w);
        *p = make_uint4(pack_bf16(f * v0.x, f * v0.y), pack_bf16(f * v1.x, f * v1.y), pack_bf16(f * v2.x, f * v2.y),
                        pack_bf16(f * v3.x, f * v3.y));
      }
      fence_proxy_async();
      named_bar(2, 64);
      if (pt == 0) {
        mbar_arrive(&sm.pre_done[s]);
        mbar_arrive(&sm.sc_free[s]);
      }
    }
  } else {
    // ------------------------------------------------------------ state warps 0-3 (thread n owns row n)
    const int n = tid;
    const uint32_t trow = taddr(tmem, 32 * warp, 0);
    const size_t fbase = unit * kP * kN;
    bool alive = true;  // the same in every state thread (set after a vote)
    for (int r = 0; r < nc; ++r) {
      const int s = r & 1, c = chunk_of(r);
      bool ok = r == 0 || mbar_wait(&sm.mma_done, (r - 1) & 1, status, 88);
      ok = ok && mbar_wait(&sm.sc_ready[s], (r >> 1) & 1, status, 89);
      if (n == 0 && r > 0) tma_store_wait_read0();  // the previous out tile has been read
      if (named_bar_or(1, 128, !ok)) {
        alive = false;
        break;
      }
      tc_fence_after();
      const float a = sm.aend[s];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float v[32];
        if (r == 0) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            v[e] = prm.init ? prm.init[fbase + (size_t)(32 * hf + e) * kN + n] : 0.f;
        } else {
          tmem_ld32(trow + 32 * hf, v);
        }
        store_row_bf16(sm.out, n, 4 * hf, v, 4);  // the state at the chunk boundary
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] *= a;
        tmem_st32(trow + 32 * hf, v);
      }
      tmem_wait_st();
      fence_proxy_async();
      tc_fence_before();
      named_bar(1, 128);
      if (n == 0) {
        tma_store_2d(&tm_out, sm.out, 0, (int)((unit * nc + c) * kN));
        tma_store_commit();
        mbar_arrive(&sm.d_ready);
        mbar_arrive(&sm.sc_free[s]);
      }
    }
    if (alive && prm.fin && !named_bar_or(1, 128, !mbar_wait(&sm.mma_done, (nc - 1) & 1, status, 90))) {
      tc_fence_after();
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float v[32];
        tmem_ld32(trow + 32 * hf, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) prm.fin[fbase + (size_t)(32 * hf + e) * kN + n] = v[e];
      }
    }
    if (n == 0) tma_store_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t tc_scan_states_bytes(const Dims& d) { return (size_t)d.b * d.H * d.nc * kN * kP * sizeof(__nv_bfloat16); }

cudaError_t tc_scan(const Dims& d, bool reverse, const void* u, const void* k, const float* dt_raw, const float* A,
                    const float* init, float* fin, __nv_bfloat16* states, int* status, cudaStream_t st) {
  CUtensorMap tu, tk, to;
  const uint64_t rows = (uint64_t)d.b * d.T;
  cudaError_t e = make_tmap_2d_bf16(&tu, u, (uint64_t)d.H * kP, rows, 64, 64);
  if (e == cudaSuccess) e = make_tmap_3d_bf16(&tk, k, d.N, d.G, rows, 64, 1, 64);
  if (e == cudaSuccess) e = make_tmap_2d_bf16(&to, states, kP, (uint64_t)d.b * d.H * d.nc * kN, 64, kN);
  if (e != cudaSuccess) return e;
  ScanParams prm{dt_raw, A, init, fin, status, d.T, d.H, d.hpg, d.nc};
  const int smem = (int)sizeof(ScanSmem) + 1024;
  if (reverse) {
    e = cudaFuncSetAttribute(k_scan<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    SSD_LAUNCH("k_tc_dstates", st, k_scan<true><<<dim3(d.H, d.b), kThreads, smem, st>>>(tu, tk, to, prm));
  } else {
    e = cudaFuncSetAttribute(k_scan<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    SSD_LAUNCH("k_tc_states", st, k_scan<false><<<dim3(d.H, d.b), kThreads, smem, st>>>(tu, tk, to, prm));
  }
  return cudaGetLastError();
}

}  // namespace ssd
