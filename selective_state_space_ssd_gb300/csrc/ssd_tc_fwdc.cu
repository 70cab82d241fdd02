// Chunk-parallel forward output of the Mamba-2 scan on tcgen05 tensor cores
// (bf16 io, chunk L = 64, head dim P = 64, state N = 128).
//
// The forward runs as K2 (C B^T per chunk, k_cb), the K3 + K4 state scan
// (ssd_tc_scan.cu: every chunk-input state S_c and s_final), and this kernel,
// the K5 output of the burn-mamba page "combined_backward.rs" (BLUE + ORANGE),
// for which every (chunk, head) is independent once S_c is known:
//
//   y[t][p] = (W' x)[t][p] + exp(cum_t) (C S_c^T)[t][p],
//   W'[t][s] = CB[t][s] exp(cum_t - cum_s) dt'_s  for s <= t, 0 above
//
// (mask before exp: the exponent of a masked entry is never formed).  The
// work items and the persistent grid are those of tc_items.cuh.  Four heads
// are in flight: their x and S_c tiles, W' tiles, TMEM accumulators and K1
// scalars sit in rings of four.
//
// Warp roles (352 threads):
//   warps 0-3   epilogue: y = y_diag + exp(cum) y_off -> bf16 tile -> TMA store
//   warps 4-7   W' tiles (CB of the chunk run in registers)
//   warp 8      K1 scalars: softplus, in-chunk cumsum, decay factors
//   warp 9      TMA producer (C per chunk run; x and S_c per head)
//   warp 10     MMA issuer and TMEM owner
// Every wait is bounded; on a timeout the kernel records a code in the
// workspace status word and stops.
#include "ssd_device.cuh"
#include "ssd_internal.h"
#include "tc_common.cuh"
#include "tc_items.cuh"

namespace ssd {
namespace {
using namespace tc;

constexpr int kL = 64, kP = 64, kN = 128;
constexpr int kThreads = 352;
constexpr int kWarpW0 = 4, kWarpScal = 8, kWarpTma = 9, kWarpMma = 10;
constexpr int kRing = 4;                   // heads in flight
constexpr uint32_t kTileLP = kL * kP * 2;  // 8 KB
constexpr uint32_t kTileNP = kN * kP * 2;  // 16 KB
constexpr uint32_t kTmemCols = 512;        // per head: y_diag (64 columns) and y_off (64 columns)

struct alignas(1024) FwdcSmem {
  struct Slot {
    uint8_t x[kTileLP];  // [s][p]
    uint8_t S[kTileNP];  // S_c bf16 [n][p]
  } sl[kRing];
  uint8_t C[2][kTileLP];   // C [t][n], two 64-column atoms
  uint8_t W[kRing][kTileLP];  // W' [t][s]
  uint8_t y[2][kTileLP];   // y staging [t][p]
  // K1 scalars of the heads in flight.  Gd_s = exp(cum_e(s) - cum_s) dt'_s and E_t[j] =
  // exp(cum_t - cum_e(j)), where e(j) is the last position of 16-block j: for s in an earlier block
  // than t, exp(cum_t - cum_s) dt'_s = E_t[blk(s)] Gd_s (both exponentials <= 1).
  float cum[kRing][kL], ecum[kRing][kL], dtp[kRing][kL], Gd[kRing][kL];
  float E[kRing][kL][4];
  uint64_t slot_full[kRing], slot_empty[kRing], sc_ready[kRing], sc_free[kRing], w_ready[kRing], mma_done[kRing],
      epi_done[kRing];
  uint64_t chunk_full, chunk_empty, drain;
  uint32_t tmem_slot;
};

struct FwdcParams {
  const float* dt_raw;
  const float* A;
  const float* CB;  // [b, nc, G, L, L] fp32
  int* status;
  int T, H, G, hpg, nc;
  int total;  // items b * nc * G * hpg (< 2^31)
};

__global__ void __launch_bounds__(kThreads, 1)
    k_tc_fwdc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_C,
              const __grid_constant__ CUtensorMap tm_S, const __grid_constant__ CUtensorMap tm_y, FwdcParams prm) {
  extern __shared__ uint8_t smem_raw[];
  FwdcSmem& sm = *reinterpret_cast<FwdcSmem*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = prm.T, H = prm.H, nc = prm.nc;
  const int total = prm.total;
  const int q0 = (int)((long long)blockIdx.x * total / gridDim.x);
  const int q1 = (int)((long long)(blockIdx.x + 1) * total / gridDim.x);
  const int nh = q1 - q0;
  int* status = prm.status;
  const ItemGeom geo{prm.hpg, prm.G, nc};

  if (tid == 0) {
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&sm.slot_full[r], 1);
      mbar_init(&sm.slot_empty[r], 1);  // MMA commit
      mbar_init(&sm.sc_ready[r], 1);
      mbar_init(&sm.sc_free[r], 2);  // W warps + epilogue warps
      mbar_init(&sm.w_ready[r], 1);
      mbar_init(&sm.mma_done[r], 1);
      mbar_init(&sm.epi_done[r], 1);
    }
    mbar_init(&sm.chunk_full, 1);
    mbar_init(&sm.chunk_empty, 1);
    mbar_init(&sm.drain, 1);
    mbar_init_fence();
  }
  if (warp == kWarpMma) tmem_alloc(&sm.tmem_slot, kTmemCols);
  // W' is zero above the diagonal blocks for every head: written once here
  for (int i = tid; i < (int)(kRing * kTileLP / 16); i += kThreads)
    reinterpret_cast<uint4*>(sm.W[0])[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  auto TYD = [&](int r) { return tmem + 128u * r; };        // y_diag = W' x (M = 64)
  auto TYO = [&](int r) { return tmem + 128u * r + 64u; };  // y_off = C S_c^T (M = 64)

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tm_x);
      prefetch_tmap(&tm_C);
      prefetch_tmap(&tm_S);
      int seg = -1;
      ItemCursor it, ip;  // this head, and the one kRing ahead for the L2 prefetch
      it.seek(geo, q0);
      ip.seek(geo, q0 + kRing);
      for (int q = 0; q < nh; ++q, it.next(geo), ip.next(geo)) {
        const int r = q % kRing, row = it.b * T + it.c * kL;
        if (it.first(q0)) {
          ++seg;
          if (seg >= 1 && !mbar_wait(&sm.chunk_empty, (seg - 1) & 1, status, 201)) break;
          mbar_expect_tx(&sm.chunk_full, 2 * kTileLP);
          for (int a = 0; a < 2; ++a) tma_load_3d(sm.C[a], &tm_C, a * 64, it.g, row, &sm.chunk_full);
        }
        if (q + kRing < nh) {
          tma_prefetch_2d(&tm_x, ip.h(geo) * kP, ip.b * T + ip.c * kL);
          tma_prefetch_2d(&tm_S, 0, (int)((((size_t)ip.b * H + ip.h(geo)) * nc + ip.c) * kN));
        }
        if (q >= kRing && !mbar_wait(&sm.slot_empty[r], ((q / kRing) - 1) & 1, status, 202)) break;
        mbar_expect_tx(&sm.slot_full[r], kTileLP + kTileNP);
        tma_load_2d(sm.sl[r].x, &tm_x, it.h(geo) * kP, row, &sm.slot_full[r]);
        tma_load_2d(sm.sl[r].S, &tm_S, 0, (int)((((size_t)it.b * H + it.h(geo)) * nc + it.c) * kN),
                    &sm.slot_full[r]);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int seg = -1;
      ItemCursor it;
      it.seek(geo, q0);
      for (int q = 0; q < nh; ++q, it.next(geo)) {
        const int r = q % kRing, ph = (q / kRing) & 1;
        bool ok = mbar_wait(&sm.slot_full[r], ph, status, 203);
        if (ok && it.first(q0)) ok = mbar_wait(&sm.chunk_full, (seg + 1) & 1, status, 204);
        if (ok && q >= kRing) ok = mbar_wait(&sm.epi_done[r], ph ^ 1, status, 205);  // TMEM buffer r read out
        if (!ok) break;
        if (it.first(q0)) ++seg;
        tc_fence_after();
#pragma unroll 1
        for (int kk = 0; kk < kN; kk += 16)  // y_off[t][p] = sum_n C[t][n] S[n][p]
          mma_bf16(TYO(r), kdesc(sm.C[0], kL, kk), mdesc(sm.sl[r].S, kN, kk), idesc_bf16(64, 64, false, true), kk > 0);
        if (!mbar_wait(&sm.w_ready[r], ph, status, 206)) break;
        tc_fence_after();
#pragma unroll 1
        for (int kk = 0; kk < kL; kk += 16)  // y_diag[t][p] = sum_s W'[t][s] x[s][p]
          mma_bf16(TYD(r), kdesc(sm.W[r], kL, kk), mdesc(sm.sl[r].x, kL, kk), idesc_bf16(64, 64, false, true), kk > 0);
        mma_commit(&sm.mma_done[r]);
        mma_commit(&sm.slot_empty[r]);
        if (it.last(geo, q1)) mma_commit(&sm.chunk_empty);
      }
      mma_commit(&sm.drain);  // nothing may still be writing TMEM when it is freed
      mbar_wait(&sm.drain, 0, status, 207);
    }
  } else if (warp == kWarpScal) {
    // ------------------------------------------------------------ K1 scalars, up to kRing heads ahead
    const int t0 = 2 * lane, t1 = t0 + 1;
    ItemCursor it;
    it.seek(geo, q0);
    for (int q = 0; q < nh; ++q, it.next(geo)) {
      const int r = q % kRing;
      if (q >= kRing && !mbar_wait(&sm.sc_free[r], ((q / kRing) - 1) & 1, status, 208)) break;
      const int h = it.h(geo);
      const float A_h = prm.A[h];
      const size_t rr = (size_t)it.b * T + it.c * kL + t0;
      const float d0 = softplus_f(__ldcs(prm.dt_raw + rr * H + h)), d1 = softplus_f(__ldcs(prm.dt_raw + (rr + 1) * H + h));
      const float a0 = d0 * A_h, a1 = a0 + d1 * A_h;
      float inc = a1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      const float c0 = inc - a1 + a0, c1 = inc;
      sm.cum[r][t0] = c0;
      sm.cum[r][t1] = c1;
      sm.dtp[r][t0] = d0;
      sm.dtp[r][t1] = d1;
      sm.ecum[r][t0] = expf(c0);
      sm.ecum[r][t1] = expf(c1);
      const float e0 = __shfl_sync(0xffffffffu, c1, 7), e1 = __shfl_sync(0xffffffffu, c1, 15);
      const float e2 = __shfl_sync(0xffffffffu, c1, 23), e3 = __shfl_sync(0xffffffffu, c1, 31);
      const int blk = t0 >> 4;
      const float my_end = blk == 0 ? e0 : (blk == 1 ? e1 : (blk == 2 ? e2 : e3));
      sm.Gd[r][t0] = expf(my_end - c0) * d0;  // decay to the end of the 16-block, times dt'
      sm.Gd[r][t1] = expf(my_end - c1) * d1;
      const float ends[4] = {e0, e1, e2, e3};
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        sm.E[r][t0][jj] = (jj < blk) ? expf(c0 - ends[jj]) : 0.f;
        sm.E[r][t1][jj] = (jj < blk) ? expf(c1 - ends[jj]) : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.sc_ready[r]);
    }
  } else if (warp >= kWarpW0) {
    // ------------------------------------------------------------ W' tiles
    // Row t = 16 (warp - 4) + (lane & 15); lane l < 16 takes columns 16 jj .. 16 jj + 7 of each block jj and
    // lane l + 16 the other 8, so the branch on the block (before / on / after the row's block) is uniform
    // across the warp.  Blocks after the row's block stay zero.
    const int qw = warp - kWarpW0;
    const int hl = lane >> 4, t = 16 * qw + (lane & 15);
    float cbv[32];  // CB[t][16 jj + 8 hl .. + 7] for jj <= qw, loaded once per chunk run
    ItemCursor it;
    it.seek(geo, q0);
    for (int q = 0; q < nh; ++q, it.next(geo)) {
      const int r = q % kRing, ph = (q / kRing) & 1;
      if (it.first(q0)) {
        const float* cbrow = prm.CB + ((size_t)it.k * kL + t) * kL + 8 * hl;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          if (jj <= qw) {
            const float4 u = __ldg(reinterpret_cast<const float4*>(cbrow + 16 * jj));
            const float4 v = __ldg(reinterpret_cast<const float4*>(cbrow + 16 * jj + 4));
            cbv[8 * jj + 0] = u.x;
            cbv[8 * jj + 1] = u.y;
            cbv[8 * jj + 2] = u.z;
            cbv[8 * jj + 3] = u.w;
            cbv[8 * jj + 4] = v.x;
            cbv[8 * jj + 5] = v.y;
            cbv[8 * jj + 6] = v.z;
            cbv[8 * jj + 7] = v.w;
          }
        }
      }
      bool ok = mbar_wait(&sm.sc_ready[r], ph, status, 209);
      if (ok && q >= kRing) ok = mbar_wait(&sm.mma_done[r], ph ^ 1, status, 210);  // W[r] read by head q - kRing
      if (named_bar_or(2, 128, !ok)) break;
      const float ct = sm.cum[r][t];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        if (jj > qw) break;
        const int s0 = 16 * jj + 8 * hl;
        float w[8];
        if (jj < qw) {
          const float f = sm.E[r][t][jj];
#pragma unroll
          for (int e = 0; e < 8; ++e) w[e] = cbv[8 * jj + e] * (f * sm.Gd[r][s0 + e]);
        } else {  // the diagonal block, masked before the exponential
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int s = s0 + e;
            w[e] = (s <= t) ? cbv[8 * jj + e] * expf(fminf(ct - sm.cum[r][s], 0.f)) * sm.dtp[r][s] : 0.f;
          }
        }
        store_row_bf16(sm.W[r], t, hl + 2 * jj, w, 1);
      }
      fence_proxy_async();
      named_bar(2, 128);
      if (tid == 32 * kWarpW0) {
        mbar_arrive(&sm.w_ready[r]);
        mbar_arrive(&sm.sc_free[r]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warps 0-3
    // y_diag and y_off are M = 64 accumulators: row t = 16 warp + (lane & 15) sits in lanes 0-15 of the
    // warp's quadrant; lanes 0-15 take columns 0-31 and lanes 16-31 columns 32-63.
    const int hl = lane >> 4, t = 16 * warp + (lane & 15);
    ItemCursor it;
    it.seek(geo, q0);
    for (int q = 0; q < nh; ++q, it.next(geo)) {
      const int r = q % kRing, ph = (q / kRing) & 1, i = q & 1;
      bool ok = mbar_wait(&sm.mma_done[r], ph, status, 211);
      ok = ok && mbar_wait(&sm.sc_ready[r], ph, status, 212);
      if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");  // y[i] (head q-2) read out
      if (named_bar_or(1, 128, !ok)) break;
      tc_fence_after();
      uint32_t vd[32], vo[32];
      tmem_ld_pair32(taddr(TYD(r), 32 * warp, 0), vd);
      tmem_ld_pair32(taddr(TYO(r), 32 * warp, 0), vo);
      tmem_wait_ld();
      const float ec = sm.ecum[r][t];
      float yv[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) yv[e] = __uint_as_float(vd[e]) + ec * __uint_as_float(vo[e]);
      store_row_bf16(sm.y[i], t, 4 * hl, yv, 4);
      tc_fence_before();
      fence_proxy_async();
      named_bar(1, 128);
      if (tid == 0) {
        tma_store_2d(&tm_y, sm.y[i], it.h(geo) * kP, it.b * T + it.c * kL);
        tma_store_commit();
        mbar_arrive(&sm.epi_done[r]);
        mbar_arrive(&sm.sc_free[r]);
      }
    }
    if (tid == 0) tma_store_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

struct FwdcWs {
  __nv_bfloat16* states;  // S_c [b,H,nc][N][P]
  float* CB;              // [b,nc,G,L,L]
};

FwdcWs carve(const Dims& d, Carver& cv) {
  FwdcWs w;
  w.states = cv.take<__nv_bfloat16>((size_t)d.b * d.H * d.nc * kN * kP);
  w.CB = cv.take<float>((size_t)d.b * d.nc * d.G * kL * kL);
  return w;
}

}  // namespace

size_t tc_forward_ws(const Dims& d) {
  Carver cv(nullptr);
  carve(d, cv);
  return cv.off;
}

cudaError_t tc_forward(const Dims& d, const FwdArgs& a, void* ws, cudaStream_t st) {
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  Carver cv(ws);
  FwdcWs w = carve(d, cv);
  int* status = static_cast<int*>(ws);
  cudaError_t e = tc_cb_prepass(d, a.B, a.C, w.CB, st);
  if (e == cudaSuccess) e = tc_scan(d, false, a.x, a.B, a.dt_raw, a.A, a.s0, a.s_final, w.states, status, st);
  if (e != cudaSuccess) return e;
  const uint64_t rows = (uint64_t)d.b * d.T;
  CUtensorMap tx, tcm, ts, ty;
  e = make_tmap_2d_bf16(&tx, a.x, (uint64_t)d.H * kP, rows, 64, 64);
  if (e == cudaSuccess) e = make_tmap_3d_bf16(&tcm, a.C, d.N, d.G, rows, 64, 1, 64);
  if (e == cudaSuccess) e = make_tmap_2d_bf16(&ts, w.states, kP, (uint64_t)d.b * d.H * d.nc * kN, 64, kN);
  if (e == cudaSuccess) e = make_tmap_2d_bf16(&ty, a.y, (uint64_t)d.H * kP, rows, 64, 64);
  if (e != cudaSuccess) return e;
  const long long total = (long long)d.b * d.nc * d.H;
  const int grid = (int)(total < sms ? total : sms);
  FwdcParams prm{a.dt_raw, a.A, w.CB, status, d.T, d.H, d.G, d.hpg, d.nc, (int)total};
  const int smem = (int)sizeof(FwdcSmem) + 1024;
  e = cudaFuncSetAttribute(k_tc_fwdc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  SSD_LAUNCH("k_tc_fwd_chunk", st, k_tc_fwdc<<<grid, kThreads, smem, st>>>(tx, tcm, ts, ty, prm));
  return cudaGetLastError();
}

}  // namespace ssd
