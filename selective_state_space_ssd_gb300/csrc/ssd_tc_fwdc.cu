// Chunk-parallel forward output of the Mamba-2 scan on tcgen05 tensor cores
// (bf16 io, chunk L = 64, head dim P = 64, state N = 128).
//
// The forward runs as one launch of the K3 + K4 state scan with the K2 tiles
// C B^T per chunk beside it (ssd_tc_scan.cu: every chunk-input state S_c,
// s_final and CB), and this kernel,
// the K5 output of the burn-mamba page "combined_backward.rs" (BLUE + ORANGE),
// for which every (chunk, head) is independent once S_c is known:
//
//   y[t][p] = (W' x)[t][p] + exp(cum_t) (C S_c^T)[t][p],
//   W'[t][s] = CB[t][s] exp(cum_t - cum_s) dt'_s  for s <= t, 0 above
//
// (mask before exp: the exponent of a masked entry is never formed).
//
// Heads go in pairs of one chunk.  A tcgen05.mma costs about the same whatever
// its shape, so both heads share each product:
//   y_diag: [W'_a; W'_b] [x_a | x_b]^T   (M = 128, N = 128, K = 64)
//   y_off:  [C; C] [S_a | S_b]^T          (M = 128, N = 128, K = 128)
// head a's results are the upper-left 64 x 64 block (lanes 0-63), head b's the
// lower-right (lanes 64-127); the two off-diagonal blocks are discarded.  A
// chunk run of odd length ends in a single head (its partner's half is junk and
// is not stored).  The work items and the persistent grid are those of
// tc_items.cuh; two pairs are in flight.
//
// Warp roles (608 threads):
//   warps 0-15  the pool, one named barrier per pair k, after which every warp runs
//                    W' tiles of pair k: twenty 16 x 16 blocks (two heads x the ten blocks
//                    at or left of the diagonal): the eight diagonal blocks on warps 0-7, the
//                    twelve others on warps 8-15, CB of the chunk run in registers, and then
//                    the epilogue of pair k-2: y = y_diag + exp(cum) y_off -> bf16 tiles,
//                    warp w on TMEM lane quadrant w % 4 and 16 columns;
//               the barrier hands W' of pair k-1 to its MMAs (which run during iteration k)
//               and the y tiles of pair k-3 to their TMA stores; one pool thread waits on
//               the mbarriers for the whole pool
//   warp 16     K1 scalars: softplus, in-chunk cumsum, decay factors (up to four pairs ahead)
//   warp 17     TMA producer (C per chunk run, twice; x and S_c per head)
//   warp 18     MMA issuer and TMEM owner
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
constexpr int kPoolWarps = 16, kPoolThreads = 32 * kPoolWarps;
constexpr int kWarpScal = kPoolWarps, kWarpTma = kPoolWarps + 1, kWarpMma = kPoolWarps + 2;
constexpr int kEpiCols = 64 / (kPoolWarps / 4);             // epilogue columns per pool warp
constexpr int kThreads = 32 * (kPoolWarps + 3);
constexpr int kBarPool = 1;  // named barrier of the pool
// The pool thread that waits on the mbarriers and issues the y stores: lane 0 of the last pool warp, which has one
// W' block (the first warps have two) and shares its scheduler with no other role
constexpr int kLead = 32 * (kPoolWarps - 1);
constexpr int kSc = 4;       // K1 scalar ring (pairs): read by W of pair k and the epilogue of pair k a phase later
constexpr uint32_t kTileLP = kL * kP * 2;  // 8 KB
constexpr uint32_t kTileNP = kN * kP * 2;  // 16 KB
constexpr uint32_t kTmemCols = 512;        // per pair slot: y_diag and y_off, 128 columns each

struct alignas(1024) FwdcSmem {
  uint8_t x[2][2][kTileLP];  // [pair slot][head]: x [s][p]; a slot's two tiles are one MN-major operand
  uint8_t S[2][2][kTileNP];  // S_c bf16 [n][p], likewise
  uint8_t W[2][2][kTileLP];  // W' [t][s]; a slot's two tiles are one K-major operand of 128 rows
  uint8_t CC[4][kTileLP];    // C atom 0, C atom 0, C atom 1, C atom 1 ([t][64 n]): [C; C] of 128 rows
  uint8_t y[2][2][kTileLP];  // y staging [t][p]
  // K1 scalars of the pairs in flight, [ring slot][head].  Gd_s = exp(cum_e(s) - cum_s) dt'_s and E_t[j] =
  // exp(cum_t - cum_e(j)), where e(j) is the last position of 16-block j: for s in an earlier block
  // than t, exp(cum_t - cum_s) dt'_s = E_t[blk(s)] Gd_s (both exponentials <= 1).
  float cum[kSc][2][kL], ecum[kSc][2][kL], dtp[kSc][2][kL], Gd[kSc][2][kL];
  float E[kSc][2][kL][4];
  float dtraw[4][2][kL], araw[4][2];  // dt_raw and A of the pairs the scalar warp has in flight (cp.async)
  uint64_t slot_full[2], slot_empty[2], w_ready[2], mma_done[2], epi_done[2], sc_ready[kSc], sc_free[kSc];
  uint64_t chunk_full, chunk_empty, drain;
  uint32_t tmem_slot;
};

struct FwdcParams {
  const float* dt_raw;
  const float* A;
  const float* CB;  // [b, nc, G, L, L]: fp32, bf16 for MIMO (load_cb8)
  int* status;
  int T, H, G, hpg, nc;
  int total;     // items b * nc * G * hpg (< 2^31)
  int mimo, rs;  // MIMO: dt_raw holds da [b, T >> rs, H] (dt' = 1), A is unused, ranks of a step see each other
};

// 16 or 32 TMEM columns of this warp's lanes, without the wait.
__device__ __forceinline__ void tmem_ld_cols(uint32_t a, uint32_t (&r)[16]) { tmem_ld16_nowait(a, r); }
__device__ __forceinline__ void tmem_ld_cols(uint32_t a, uint32_t (&r)[32]) { tmem_ld32_nowait(a, r); }

// Walks a CTA's items in units of one or two heads of the same chunk.
struct PairCursor {
  ItemCursor a;
  int n;  // heads in this unit (1 or 2)
  __device__ __forceinline__ void seek(const ItemGeom& m, int f0, int q1) {
    a.seek(m, f0);
    count(m, q1);
  }
  __device__ __forceinline__ void count(const ItemGeom& m, int q1) {
    n = (a.f + 1 < q1 && a.jh + 1 < m.hpg) ? 2 : 1;
  }
  __device__ __forceinline__ void next(const ItemGeom& m, int q1) {
    for (int i = 0; i < n; ++i) a.next(m);
    count(m, q1);
  }
  __device__ __forceinline__ bool last(const ItemGeom& m, int q1) const {  // last unit of the CTA's run on the chunk
    return a.f + n == q1 || a.jh + n == m.hpg;
  }
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
  int* status = prm.status;
  const ItemGeom geo{prm.hpg, prm.G, nc};

  if (tid == 0) {
    for (int r = 0; r < 2; ++r) {
      mbar_init(&sm.slot_full[r], 1);
      mbar_init(&sm.slot_empty[r], 1);  // MMA commit
      mbar_init(&sm.w_ready[r], 1);
      mbar_init(&sm.mma_done[r], 1);
      mbar_init(&sm.epi_done[r], kPoolWarps);  // every pool warp once its TMEM reads of the pair are done
    }
    for (int r = 0; r < kSc; ++r) {
      mbar_init(&sm.sc_ready[r], 1);
      mbar_init(&sm.sc_free[r], kPoolWarps);  // every pool warp after the pair's epilogue
    }
    mbar_init(&sm.chunk_full, 1);
    mbar_init(&sm.chunk_empty, 1);
    mbar_init(&sm.drain, 1);
    mbar_init_fence();
  }
  if (warp == kWarpMma) tmem_alloc(&sm.tmem_slot, kTmemCols);
  // W' is zero above the diagonal blocks for every head: written once here
  for (int i = tid; i < (int)(4 * kTileLP / 16); i += kThreads) reinterpret_cast<uint4*>(sm.W[0][0])[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the chunk states and C B^T tiles of the scan launch before this kernel
  const uint32_t tmem = sm.tmem_slot;
  auto TYD = [&](int r) { return tmem + 256u * r; };          // y_diag of the pair (M = 128, 128 columns)
  auto TYO = [&](int r) { return tmem + 256u * r + 128u; };   // y_off of the pair

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tm_x);
      prefetch_tmap(&tm_C);
      prefetch_tmap(&tm_S);
      int seg = -1;
      PairCursor u;
      u.seek(geo, q0, q1);
      for (int k = 0; u.a.f < q1; ++k, u.next(geo, q1)) {
        const int r = k & 1, t0 = u.a.c * kL;
        if (u.a.first(q0)) {
          ++seg;
          if (seg >= 1 && !mbar_wait(&sm.chunk_empty, (seg - 1) & 1, status, 201)) break;
          mbar_expect_tx(&sm.chunk_full, 4 * kTileLP);
          for (int a = 0; a < 4; ++a) tma_load_4d(sm.CC[a], &tm_C, (a >> 1) * 64, u.a.g, t0, u.a.b, &sm.chunk_full);
        }
        if (k >= 2 && !mbar_wait(&sm.slot_empty[r], ((k >> 1) - 1) & 1, status, 202)) break;
        mbar_expect_tx(&sm.slot_full[r], u.n * (kTileLP + kTileNP));
        for (int i = 0; i < u.n; ++i) {
          const int h = u.a.h(geo) + i;
          tma_load_3d(sm.x[r][i], &tm_x, h * kP, t0, u.a.b, &sm.slot_full[r]);
          tma_load_2d(sm.S[r][i], &tm_S, 0, (int)((((size_t)u.a.b * H + h) * nc + u.a.c) * kN), &sm.slot_full[r]);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int seg = -1;
      PairCursor u;
      u.seek(geo, q0, q1);
      for (int k = 0; u.a.f < q1; ++k, u.next(geo, q1)) {
        const int r = k & 1, ph = (k >> 1) & 1;
        bool ok = mbar_wait(&sm.slot_full[r], ph, status, 203);
        if (ok && u.a.first(q0)) ok = mbar_wait(&sm.chunk_full, (seg + 1) & 1, status, 204);
        if (ok && k >= 2) ok = mbar_wait(&sm.epi_done[r], ph ^ 1, status, 205);  // TMEM slot r read out
        if (!ok) break;
        if (u.a.first(q0)) ++seg;
        tc_fence_after();
        // y_off[t][p] = sum_n C[t][n] S[n][p], both heads (unrolled, precomputed descriptors)
        const uint64_t cd = kdesc(sm.CC[0], 2 * kL, 0), sd = mdesc(sm.S[r][0], kN, 0);
#pragma unroll
        for (int kk = 0; kk < kN; kk += 16)
          mma_bf16(TYO(r), cd + kdesc_step(2 * kL, kk), sd + mdesc_step(kk), idesc_bf16(128, 128, false, true), kk > 0);
        if (!mbar_wait(&sm.w_ready[r], ph, status, 206)) break;
        tc_fence_after();
        // y_diag[t][p] = sum_s W'[t][s] x[s][p], both heads: after W' is ready, on the pair's critical path, so
        // issued unrolled from precomputed descriptors
        const uint64_t wd = kdesc(sm.W[r][0], 2 * kL, 0), xd = mdesc(sm.x[r][0], kL, 0);
#pragma unroll
        for (int kk = 0; kk < kL; kk += 16)
          mma_bf16(TYD(r), wd + kdesc_step(2 * kL, kk), xd + mdesc_step(kk), idesc_bf16(128, 128, false, true), kk > 0);
        mma_commit(&sm.mma_done[r]);
        mma_commit(&sm.slot_empty[r]);
        if (u.last(geo, q1)) mma_commit(&sm.chunk_empty);
      }
      mma_commit(&sm.drain);  // nothing may still be writing TMEM when it is freed
      mbar_wait(&sm.drain, 0, status, 207);
    }
  } else if (warp == kWarpScal) {
    // ------------------------------------------------------------ K1 scalars, up to kSc pairs ahead.  The
    //   strided dt_raw reads (and A) of pair k + 3 go out as cp.async copies into a ring while pair k is
    //   formed: global-memory latency under the kernel's own HBM load (~2 us) would otherwise set the pace
    //   of the whole CTA.  Steps past the end of the sequence (a partial last chunk) get dt_raw = -inf,
    //   i.e. dt' = 0: their W' columns vanish, and their y rows are not stored.
    //   MIMO reads da at the first rank of each step and 0 at the others.
    const int t0 = 2 * lane, t1 = t0 + 1;
    const int msk = (1 << prm.rs) - 1;
    auto fetch = [&](const PairCursor& c, int slot) {
      if (c.a.f < q1) {
        const int h0 = c.a.h(geo);
        const int tt = c.a.c * kL + t0;
        if (prm.mimo) {
          const size_t sr = (size_t)c.a.b * (T >> prm.rs);
          for (int i = 0; i < c.n; ++i) {
            if (tt < T && (tt & msk) == 0) cp_async4(&sm.dtraw[slot][i][t0], prm.dt_raw + (sr + (tt >> prm.rs)) * H + h0 + i);
            else sm.dtraw[slot][i][t0] = 0.f;
            if (tt + 1 < T && ((tt + 1) & msk) == 0)
              cp_async4(&sm.dtraw[slot][i][t1], prm.dt_raw + (sr + ((tt + 1) >> prm.rs)) * H + h0 + i);
            else sm.dtraw[slot][i][t1] = 0.f;
          }
          if (lane < c.n) sm.araw[slot][lane] = 1.f;
        } else {
          const size_t rr = (size_t)c.a.b * T + tt;
          for (int i = 0; i < c.n; ++i) {
            if (tt < T) cp_async4(&sm.dtraw[slot][i][t0], prm.dt_raw + rr * H + h0 + i);
            else sm.dtraw[slot][i][t0] = -INFINITY;
            if (tt + 1 < T) cp_async4(&sm.dtraw[slot][i][t1], prm.dt_raw + (rr + 1) * H + h0 + i);
            else sm.dtraw[slot][i][t1] = -INFINITY;
          }
          if (lane < c.n) cp_async4(&sm.araw[slot][lane], prm.A + h0 + lane);
        }
      }
      cp_async_commit();  // one group per pair, empty past the last, so that the count stays uniform
    };
    PairCursor u, uf;  // pairs k (formed) and k + 3 (fetched)
    u.seek(geo, q0, q1);
    uf = u;
    for (int d = 0; d < 3; ++d) {
      fetch(uf, d);
      if (uf.a.f < q1) uf.next(geo, q1);
    }
    for (int k = 0; u.a.f < q1; ++k, u.next(geo, q1)) {
      const int r = k % kSc, sl = k & 3;
      fetch(uf, (k + 3) & 3);  // the slot pair k - 1 used
      if (uf.a.f < q1) uf.next(geo, q1);
      cp_async_wait<3>();  // pair k's copies have landed
      __syncwarp();
      if (k >= kSc && !mbar_wait(&sm.sc_free[r], (k / kSc - 1) & 1, status, 208)) break;
#pragma unroll 1
      for (int i = 0; i < u.n; ++i) {
        const float A_h = sm.araw[sl][i];
        const float z0 = sm.dtraw[sl][i][t0], z1 = sm.dtraw[sl][i][t1];
        const float d0 = prm.mimo ? 1.f : softplus_fast(z0), d1 = prm.mimo ? 1.f : softplus_fast(z1);
        const float a0 = prm.mimo ? z0 : d0 * A_h, a1 = a0 + (prm.mimo ? z1 : d1 * A_h);
        float inc = a1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float v = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += v;
        }
        const float c0 = inc - a1 + a0, c1 = inc;
        sm.cum[r][i][t0] = c0;
        sm.cum[r][i][t1] = c1;
        sm.dtp[r][i][t0] = d0;
        sm.dtp[r][i][t1] = d1;
        sm.ecum[r][i][t0] = __expf(c0);
        sm.ecum[r][i][t1] = __expf(c1);
        const float e0 = __shfl_sync(0xffffffffu, c1, 7), e1 = __shfl_sync(0xffffffffu, c1, 15);
        const float e2 = __shfl_sync(0xffffffffu, c1, 23), e3 = __shfl_sync(0xffffffffu, c1, 31);
        const int blk = t0 >> 4;
        const float my_end = blk == 0 ? e0 : (blk == 1 ? e1 : (blk == 2 ? e2 : e3));
        sm.Gd[r][i][t0] = __expf(my_end - c0) * d0;  // decay to the end of the 16-block, times dt'
        sm.Gd[r][i][t1] = __expf(my_end - c1) * d1;
        const float ends[4] = {e0, e1, e2, e3};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          sm.E[r][i][t0][jj] = (jj < blk) ? __expf(c0 - ends[jj]) : 0.f;
          sm.E[r][i][t1][jj] = (jj < blk) ? __expf(c1 - ends[jj]) : 0.f;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.sc_ready[r]);
    }
    cp_async_wait<0>();
  } else if (warp < kPoolWarps) {
    // ------------------------------------------------------------ the pool (warps 0 .. kPoolWarps-1).
    //   Iteration k, after one barrier:
    //     W' of pair k: 20 blocks of 16 x 16 (two heads x the ten blocks at or left of the diagonal),
    //       split by kind between the warps (below)
    //     epilogue of pair k - 2: y = y_diag + exp(cum) y_off; warp w reads TMEM lanes 32 (w % 4) ..
    //       (head w % 4 / 2) and kEpiCols columns from kEpiCols (w / 4) of that head
    //   The barrier releases W' of pair k - 1 to its y_diag MMAs and the y tiles of pair k - 3 to their
    //   TMA stores; the MMAs of pair k - 1 run during iteration k, one iteration before their epilogue.
    const int qd = warp & 3, hf = warp >> 2;
    // W' blocks of a pair: the eight diagonal blocks (masked exponentials) on warps 0-7, one each; the twelve
    // blocks left of the diagonal (two products from the scalar tables) two each on warps 8-11 and one on
    // warps 12-15 (which compute theirs twice, so that every off-diagonal warp runs one straight-line path)
    const bool wdiag = warp < 8;
    int ti[2], tq[2], tj[2];
    if (wdiag) {
      ti[0] = ti[1] = warp >> 2;
      tq[0] = tq[1] = tj[0] = tj[1] = warp & 3;
    } else {
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int o = warp < 12 ? 2 * (warp - 8) + m : warp - 4;  // 0 .. 11: head o / 6, block o % 6
        const int bo = o % 6;
        ti[m] = o / 6;
        tq[m] = bo < 1 ? 1 : bo < 3 ? 2 : 3;
        tj[m] = bo < 1 ? 0 : bo < 3 ? bo - 1 : bo - 3;
      }
    }
    float cbv[16];  // CB of this warp's blocks (the same for both heads), loaded once per chunk run
    PairCursor uw, ue, us;  // pairs k (W), k - 2 (epilogue), k - 3 (y stores)
    uw.seek(geo, q0, q1);
    ue = uw;
    us = uw;
    int np = 0;  // pairs of this CTA
    for (PairCursor c = uw; c.a.f < q1; c.next(geo, q1)) ++np;
    for (int k = 0; k <= np + 2; ++k) {
      const bool has_w = k < np, has_r = k >= 1 && k - 1 < np, has_e = k >= 2 && k - 2 < np,
                 has_s = k >= 3 && k - 3 < np;
      const int r = k & 1, sc = k % kSc;
      if (has_w && uw.a.first(q0)) {
#pragma unroll
        for (int m = 0; m < 2; ++m)
          load_cb8(prm.CB, ((size_t)uw.a.k * kL + 16 * tq[m] + (lane & 15)) * kL + 16 * tj[m] + 8 * (lane >> 4),
                   prm.mimo, cbv + 8 * m);
      }
      bool ok = true;
      if (tid == kLead) {  // one thread waits; the named barrier passes the inputs to the pool
        if (has_w) ok = mbar_wait(&sm.sc_ready[sc], (k / kSc) & 1, status, 209);
        // pair k - 2's MMAs are done: W[r] may be rewritten and its y read out of TMEM
        if (ok && k >= 2 && k - 2 < np) ok = mbar_wait(&sm.mma_done[r], ((k >> 1) - 1) & 1, status, 210);
        if (k >= 4) tma_store_wait_read0();  // the y tiles of pair k - 4 (pair k - 2's staging slot) are read
      }
      tc_fence_before();
      fence_proxy_async();  // W' of pair k - 1 for its MMAs; the y tiles of pair k - 3 for their stores
      if (named_bar_or(kBarPool, kPoolThreads, !ok)) break;
      if (tid == kLead) {
        if (has_r) mbar_arrive(&sm.w_ready[(k - 1) & 1]);
        if (has_s) {
          const int rs = (k - 3) & 1;
          for (int i = 0; i < us.n; ++i)
            tma_store_3d(&tm_y, sm.y[rs][i], (us.a.h(geo) + i) * kP, us.a.c * kL, us.a.b);
          tma_store_commit();
        }
      }
      if (has_w) {
        const int hl = lane >> 4;
        if (wdiag) {  // the diagonal block, masked before the exponential
          const int i = ti[0], t = 16 * tq[0] + (lane & 15), s0 = 16 * tj[0] + 8 * hl;
          const float ct = sm.cum[sc][i][t];
          float w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int s2 = s0 + e;
            // (MIMO: the ranks of one step see each other, cum being flat across them)
            w[e] = ((s2 >> prm.rs) <= (t >> prm.rs)) ? cbv[e] * __expf(fminf(ct - sm.cum[sc][i][s2], 0.f)) * sm.dtp[sc][i][s2]
                                                     : 0.f;
          }
          store_row_bf16(sm.W[r][i], t, hl + 2 * tj[0], w, 1);
        } else {  // two blocks left of the diagonal: exp(cum_t - cum_s) dt'_s = E_t[jj] Gd_s
          const int ta = 16 * tq[0] + (lane & 15), tb = 16 * tq[1] + (lane & 15);
          const int sa = 16 * tj[0] + 8 * hl, sb = 16 * tj[1] + 8 * hl;
          const float fa = sm.E[sc][ti[0]][ta][tj[0]], fb = sm.E[sc][ti[1]][tb][tj[1]];
          float wa[8], wb[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            wa[e] = cbv[e] * (fa * sm.Gd[sc][ti[0]][sa + e]);
            wb[e] = cbv[8 + e] * (fb * sm.Gd[sc][ti[1]][sb + e]);
          }
          store_row_bf16(sm.W[r][ti[0]], ta, hl + 2 * tj[0], wa, 1);
          store_row_bf16(sm.W[r][ti[1]], tb, hl + 2 * tj[1], wb, 1);
        }
      }
      if (has_e) {
        const int re = (k - 2) & 1, se = (k - 2) % kSc;
        tc_fence_after();
        const int hi = qd >> 1, t = 32 * (qd & 1) + lane;
        if (hi < ue.n) {
          const float ec = sm.ecum[se][hi][t];
          uint32_t vd[kEpiCols], vo[kEpiCols];
          tmem_ld_cols(taddr(TYD(re), 32 * qd, 64 * hi + kEpiCols * hf), vd);
          tmem_ld_cols(taddr(TYO(re), 32 * qd, 64 * hi + kEpiCols * hf), vo);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.epi_done[re]);  // the next MMAs into this TMEM slot may start
          float yv[kEpiCols];
#pragma unroll
          for (int e = 0; e < kEpiCols; ++e) yv[e] = __uint_as_float(vd[e]) + ec * __uint_as_float(vo[e]);
          store_row_bf16(sm.y[re][hi], t, (kEpiCols / 8) * hf, yv, kEpiCols / 8);
        } else if (lane == 0) {
          mbar_arrive(&sm.epi_done[re]);  // a single-head pair: this warp's lanes hold no live rows
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.sc_free[se]);  // the pair's last scalar reader
      }
      if (has_s) us.next(geo, q1);
      if (has_e) ue.next(geo, q1);
      if (has_w) uw.next(geo, q1);
    }
    if (tid == kLead) tma_store_wait0();
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

size_t tc_forward_ws(const Dims& problem) {
  Carver cv(nullptr);
  carve(tc_dims(problem), cv);
  return cv.off;
}

cudaError_t tc_forward(const Dims& problem, const FwdArgs& a, void* ws, cudaStream_t st) {
  const Dims d = tc_dims(problem);
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  Carver cv(ws);
  FwdcWs w = carve(d, cv);
  int* status = static_cast<int*>(ws);
  __nv_bfloat16* states = a.states_out ? a.states_out : w.states;  // a stash for the backward, or scratch
  const ScanSide fwd{a.x, a.s0, a.s_final, states, a.ckpt_out, nullptr, a.ckpt_every};
  cudaError_t e = tc_scans(d, &fwd, nullptr, a.B, a.C, a.dt_raw, a.A, w.CB, status, st);
  if (e != cudaSuccess) return e;
  CUtensorMap tx, tcm, ts, ty;
  e = make_tmap_seq_bf16(&tx, a.x, d, (uint64_t)d.H * kP);
  if (e == cudaSuccess) e = make_tmap_bc_bf16(&tcm, a.C, d);
  if (e == cudaSuccess) e = make_tmap_2d_bf16(&ts, states, kP, (uint64_t)d.b * d.H * d.nc * kN, 64, kN);
  if (e == cudaSuccess) e = make_tmap_seq_bf16(&ty, a.y, d, (uint64_t)d.H * kP);
  if (e != cudaSuccess) return e;
  const long long total = (long long)d.b * d.nc * d.H;
  const int grid = (int)(total < sms ? total : sms);
  FwdcParams prm{a.dt_raw, a.A, w.CB, status, d.T, d.H, d.G, d.hpg, d.nc, (int)total, d.variant == kMimo, d.rs};
  const int smem = (int)sizeof(FwdcSmem) + 1024;
  e = cudaFuncSetAttribute(k_tc_fwdc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  SSD_LAUNCH("k_tc_fwd_chunk", st, e = launch_after(k_tc_fwdc, grid, kThreads, smem, st, tx, tcm, ts, ty, prm));
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace ssd
