// Chunk-parallel backward of the Mamba-2 scan on tcgen05 tensor cores (bf16
// io, chunk L = 64, head dim P = 64, state N = 128).
//
// The recompute backward of the burn-mamba page "combined_backward.rs" in
// three stages, the first two in one launch (ssd_tc_scan.cu, which also
// writes the K2 tiles CB = C B^T), since neither needs the other:
//   1. the forward state scan replays S_c (the state entering chunk c) from
//      the saved inputs;
//   2. the reverse scan gives dS_{c+1} (the gradient of the state leaving
//      chunk c) for every chunk, and ds0;
//   3. this kernel: with S_c and dS_{c+1} known, every (chunk, head) is
//      independent, and computes the K5 (BLUE + ORANGE), K4, K3 and K2
//      backwards of the page:
//
//   1a:  dW~ = dy x^T
//   E:   W = CB o decay,  dCB = dW~ o dt'_s o decay,  ORANGE row sums of dCB o CB (mask before exp)
//   2:   dv_or = W^T dy;  at a chunk run's end dB^T += C^T dCBsum, dC^T += B^T dCBsum^T
//   1b:  [B; C] [dS_{c+1} | S_c]^T (ddv and Y);  dB^T += dS_{c+1} dvd^T,  dC^T += S_c dch^T
//   O:   dv = dv_or + exp(cum_end - cum_s) ddv,  dx = dt' dv,  sum_p dv x, sum_p ddv x
//   BK:  BLUE d cum_t = exp(cum_t) sum_p dy Y;  K4: exp(cum_end) <dS_{c+1}, S_c>
//   AS:  d cum assembly, suffix sums -> ddt_raw, dA part
// with dch = exp(cum) dy, dvd = exp(cum_end - cum) dt' x and decay[t][s] =
// exp(cum_t - cum_s) for s <= t.
//
// The (chunk, group, head) list is cut into one contiguous range per CTA (a
// persistent grid of one CTA per SM), so that every SM gets the same number
// of heads.  Heads of one chunk share B, C and CB, and their dB^T and dC^T
// add up in two TMEM accumulators; a CTA writes one fp32 partial per chunk
// it touched, and a small kernel adds the (at most a few) partials of each
// chunk in a fixed order.
//
// Warps (608 threads):
//   warps 0-15  the pool: all CUDA-core work, in three phases per iteration i
//               (warp w works on TMEM lane quadrant w % 4):
//                 S1  O of head i-1 (quadrants 0-1: rows s of dv_or and ddv) beside
//                     BLUE of head i-1 (quadrants 2-3: rows t of Y);
//                     at a chunk run's end every warp reads the dB^T, dC^T accumulators out
//                 S2  P of head i+1: the dch and dvd tiles
//                 S3  E of head i on ten warps (one 16 x 16 block of dW~ each) beside
//                     the d cum assembly AS of head i-1 on one more and K4 of head i on four
//               The phases run in lockstep (named barriers), so the pool executes one
//               phase's code at a time: a small instruction footprint and short per-head
//               latency chains.
//   warp 16     SC: K1 scalars up to four heads ahead.
//   warp 17     MMA issuer and TMEM owner, in a fixed order: 1a of head n, 2 of head n-1,
//               1b of head n (blocking waits, no polling).
//   warp 18     TMA producer (x, dy, S_c, dS_{c+1} per head; B, C per chunk run).
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
constexpr int kWarpScal = 16, kWarpMma = 17, kWarpTma = 18;
// The pool thread that waits on the mbarriers and issues the dx stores: lane 0 of warp 15, an E warp (row and
// column block 3) on the one scheduler that hosts no other role
constexpr int kLead = 32 * 15;
constexpr int kThreads = 32 * 19;
constexpr int kBarPool = 1;  // named barrier of the pool
constexpr int kEWarps = 10;  // pool warps w with w / 4 <= w % 4: one (row block w % 4, column block w / 4) each
constexpr int kWarpAs = 4;   // pool warp that runs AS in phase S3 (idle in E)
constexpr uint32_t kTileLP = kL * kP * 2;  // 8 KB
constexpr uint32_t kTileNP = kN * kP * 2;  // 16 KB
constexpr uint32_t kTmemCols = 512;

struct alignas(1024) BwdcSmem {
  // per-head TMA tiles in two rings: x, dy (three slots) and dS, S (two slots)
  struct XY {
    uint8_t x[kTileLP];   // [s][p]
    uint8_t dy[kTileLP];  // [t][p]
  } xy[3];
  struct SD {
    uint8_t dS[kTileNP];  // dS_{c+1} bf16 [n][p]
    uint8_t S[kTileNP];   // S_c bf16 [n][p], right after dS: [dS | S] is one MN-major operand
  } sd[2];
  uint8_t BC[4][kTileLP];   // B atom 0, C atom 0, B atom 1, C atom 1 ([t][64 n] each): [B; C] is one
                            // K-major operand of 128 rows
  uint8_t dch[2][kTileLP];  // exp(cum) dy [t][p]
  uint8_t dvd[2][kTileLP];  // exp(cum_end - cum) dt' x [s][p]
  uint8_t W[2][kTileLP];    // [t][s]; (the 8 KB after W[j] feed the unused upper rows of dv_or)
  uint8_t dcbs[kTileLP];    // sum over the chunk run of dCB [t][s], bf16 (the fp32 sum lives in E's registers)
  uint8_t dxs[kTileLP];     // dx staging [s][p]
  // K1 scalars, ring of four heads
  float cum[4][kL], ecum[4][kL], dec[4][kL], dtp[4][kL], z[4][kL];
  float aend[4], Ah[4];
  // per-head partial sums for the d cum assembly (two heads): ORANGE row sums per column block, BLUE
  // and the dv.x / ddv.x sums per 16-column group, K4 per K4 warp
  float drow[2][4][kL], blue[2][4][kL], dvx[2][4][kL], dde[2][4][kL], k4p[2][4];
  uint64_t xy_full[3], xy_empty[3], sd_full[2], sd_empty[2];
  uint64_t pre_done[2], s1a_done[2], s1b_done[2], e_done[2], s2_done[2], tmem_free[2];
  uint64_t sc_ready[4], sc_free[4];
  uint64_t chunk_full, chunk_empty, acc_full, acc_free, drain;
  uint32_t tmem_slot;
};

struct BwdcParams {
  const float* dt_raw;
  const float* A;
  const float* CB;  // [b, nc, G, L, L]: fp32, bf16 for MIMO (load_cb8)
  float* ddt_raw;
  float* dA_part;  // [b, H, nc]
  float* dB_part;  // [chunks][nseg][L][N]
  float* dC_part;
  int* status;
  int T, H, G, hpg, nc;
  int nseg;      // partial slots per chunk
  int total;     // number of (chunk, group, head) items: b * nc * G * hpg (< 2^31)
  int mimo, rs;  // MIMO: dt_raw holds da [b, T >> rs, H] (dt' = 1) and ddt_raw receives its gradient; A unused
  // one head per group (hpg == 1): a chunk's accumulators are its final dB, dC, written as bf16 [b, T, G, N]
  // straight from TMEM instead of through the fp32 partials
  __nv_bfloat16* dB;
  __nv_bfloat16* dC;
};

__device__ __forceinline__ void load_row8(const uint8_t* tile, int r, int j, float* out) {
  const uint4 raw = *reinterpret_cast<const uint4*>(tile + sw128_chunk(r, j));
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = unpack_bf16(w[e]);
    out[2 * e] = f.x;
    out[2 * e + 1] = f.y;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    k_tc_bwdc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
              const __grid_constant__ CUtensorMap tm_dx, const __grid_constant__ CUtensorMap tm_B,
              const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_S,
              const __grid_constant__ CUtensorMap tm_dS, BwdcParams prm) {
  extern __shared__ uint8_t smem_raw[];
  BwdcSmem& sm = *reinterpret_cast<BwdcSmem*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = prm.T, H = prm.H, nc = prm.nc;
  const int total = prm.total;
  const int q0 = (int)((long long)blockIdx.x * total / gridDim.x);
  const int q1 = (int)((long long)(blockIdx.x + 1) * total / gridDim.x);
  const int nh = q1 - q0;
  int* status = prm.status;
  const ItemGeom geo{prm.hpg, prm.G, nc};

  if (tid == 0) {
    for (int j = 0; j < 2; ++j) {
      mbar_init(&sm.sd_full[j], 1);
      mbar_init(&sm.sd_empty[j], 1);  // the pool, after BK
      mbar_init(&sm.pre_done[j], 1);
      mbar_init(&sm.s1a_done[j], 1);
      mbar_init(&sm.s1b_done[j], 1);
      mbar_init(&sm.e_done[j], kEWarps);
      mbar_init(&sm.s2_done[j], 1);
      mbar_init(&sm.tmem_free[j], 1);
    }
    for (int x = 0; x < 3; ++x) {
      mbar_init(&sm.xy_full[x], 1);
      mbar_init(&sm.xy_empty[x], 1);  // the pool, after O and BK
    }
    for (int k = 0; k < 4; ++k) {
      mbar_init(&sm.sc_ready[k], 1);
      mbar_init(&sm.sc_free[k], 1);  // AS, the scalars' last reader
    }
    mbar_init(&sm.chunk_full, 1);
    mbar_init(&sm.chunk_empty, 1);
    mbar_init(&sm.acc_full, 1);
    mbar_init(&sm.acc_free, 1);
    mbar_init(&sm.drain, 1);
    mbar_init_fence();
  }
  if (warp == kWarpMma) tmem_alloc(&sm.tmem_slot, kTmemCols);
  // W and the dCB sum are zero above the diagonal blocks, and so are the row-sum parts of the column
  // blocks right of a row's block, for every head: written once here, never touched by the per-head work
  for (int i = tid; i < (int)(3 * kTileLP / 16); i += kThreads)
    reinterpret_cast<uint4*>(sm.W[0])[i] = make_uint4(0, 0, 0, 0);  // W[0], W[1], dcbs are contiguous
  for (int i = tid; i < 2 * 4 * kL; i += kThreads) (&sm.drow[0][0][0])[i] = 0.f;
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();     // the chunk states, dS and C B^T tiles of the scan launch before this kernel
  pdl_trigger();  // the sums kernel may be scheduled as this kernel's CTAs finish
  const uint32_t tmem = sm.tmem_slot;
  const uint32_t ACC_B = tmem, ACC_C = tmem + 64u;                  // dB^T, dC^T (M = 128, lane n)
  auto TW = [&](int j) { return tmem + 128u + 192u * j; };         // dW~ (M = 64), then dv_or (M = 128, lane s)
  auto YD = [&](int j) { return tmem + 128u + 192u * j + 64u; };   // [B; C] [dS | S]^T (M = 128, 128 columns):
                                                                   // ddv in lanes 0-63 / cols 0-63, Y in lanes
                                                                   // 64-127 / cols 64-127

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tm_x);
      prefetch_tmap(&tm_dy);
      prefetch_tmap(&tm_S);
      prefetch_tmap(&tm_dS);
      prefetch_tmap(&tm_B);
      prefetch_tmap(&tm_C);
      int seg = -1;
      ItemCursor hr, hp;  // this head, and the one two ahead for the L2 prefetch
      hr.seek(geo, q0);
      hp.seek(geo, q0 + 2);
      for (int q = 0; q < nh; ++q, hr.next(geo), hp.next(geo)) {
        const int j = q & 1;
        const int t0 = hr.c * kL;
        if (q + 2 < nh) {  // warm L2 with the tiles of head q + 2 while the rings are still busy
          const int psrow = (int)((((size_t)hp.b * H + hp.h(geo)) * nc + hp.c) * kN);
          tma_prefetch_3d(&tm_x, hp.h(geo) * kP, hp.c * kL, hp.b);
          tma_prefetch_3d(&tm_dy, hp.h(geo) * kP, hp.c * kL, hp.b);
          tma_prefetch_2d(&tm_S, 0, psrow);
          tma_prefetch_2d(&tm_dS, 0, psrow);
        }
        const int x3 = q % 3, xr = q / 3;
        if (q >= 3 && !mbar_wait(&sm.xy_empty[x3], (xr - 1) & 1, status, 102)) break;
        mbar_expect_tx(&sm.xy_full[x3], 2 * kTileLP);
        tma_load_3d(sm.xy[x3].x, &tm_x, hr.h(geo) * kP, t0, hr.b, &sm.xy_full[x3]);
        tma_load_3d(sm.xy[x3].dy, &tm_dy, hr.h(geo) * kP, t0, hr.b, &sm.xy_full[x3]);
        if (q >= 2 && !mbar_wait(&sm.sd_empty[j], ((q >> 1) - 1) & 1, status, 99)) break;
        const int srow = (int)((((size_t)hr.b * H + hr.h(geo)) * nc + hr.c) * kN);
        mbar_expect_tx(&sm.sd_full[j], 2 * kTileNP);
        tma_load_2d(sm.sd[j].dS, &tm_dS, 0, srow, &sm.sd_full[j]);
        tma_load_2d(sm.sd[j].S, &tm_S, 0, srow, &sm.sd_full[j]);
        // B, C of a new chunk run after the head's own tiles: the wait for the previous run's last MMAs
        // needs E of the head before, which the pool runs after P of this head (P waits for x / dy)
        if (hr.first(q0)) {
          ++seg;
          if (seg >= 1 && !mbar_wait(&sm.chunk_empty, (seg - 1) & 1, status, 101)) break;
          mbar_expect_tx(&sm.chunk_full, 4 * kTileLP);
          for (int a = 0; a < 2; ++a) {
            tma_load_4d(sm.BC[2 * a], &tm_B, a * 64, hr.g, t0, hr.b, &sm.chunk_full);
            tma_load_4d(sm.BC[2 * a + 1], &tm_C, a * 64, hr.g, t0, hr.b, &sm.chunk_full);
          }
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer.  Slot n issues, in order:
    //   1a(n)  dW~ = dy x^T                      (x / dy of head n; TMEM slot n & 1 read out by the pool)
    //   2(n-1) dv_or = W^T dy (after E), and at a chunk run's end the run's summed dCB terms
    //   1b(n)  [B; C] [dS | S]^T (ddv and Y), dB^T += dS dvd^T and dC^T += S dch^T (after P)
    // 2(n-1) comes before 1b(n), so the pool's O and BK of head n-1 wait for 8 MMAs, not 24.
    if (lane == 0) {
      int seg1 = -1;
      ItemCursor c1, c2;  // heads n and n - 1
      c1.seek(geo, q0);
      c2.seek(geo, q0);
      const uint32_t bc_b = smem_u32(sm.BC[0]), bc_c = smem_u32(sm.BC[1]);
      for (int n = 0; n <= nh; ++n) {
        const int j = n & 1, ph = (n >> 1) & 1;
        if (n < nh) {  // 1a(n)
          bool ok = mbar_wait(&sm.xy_full[n % 3], (n / 3) & 1, status, 131);
          if (ok && n >= 2) ok = mbar_wait(&sm.tmem_free[j], ph ^ 1, status, 132);
          if (!ok) break;
          tc_fence_after();
          const BwdcSmem::XY& gx = sm.xy[n % 3];
#pragma unroll 1
          for (int kk = 0; kk < kP; kk += 16)  // dW~[t][s] = sum_p dy[t][p] x[s][p]
            mma_bf16(TW(j), kdesc(gx.dy, kL, kk), kdesc(gx.x, kL, kk), idesc_bf16(64, 64, false, false), kk > 0);
          mma_commit(&sm.s1a_done[j]);
        }
        if (n >= 1) {  // 2(n-1)
          const int m = n - 1, jm = m & 1;
          if (!mbar_wait(&sm.e_done[jm], (m >> 1) & 1, status, 133)) break;
          tc_fence_after();
          // dv_or[s][p] = sum_t W[t][s] dy[t][p]  (rows s in lanes 0-63).  These four MMAs sit between E and the
          // next O phase, so they are issued unrolled from precomputed descriptors; the other loops stay rolled
          // (issued faster, their MMAs run beside the pool's shared-memory work and slow it more than they gain)
          const uint64_t wa = mdesc(sm.W[jm], kL, 0), wb = mdesc(sm.xy[m % 3].dy, kL, 0);
#pragma unroll
          for (int kk = 0; kk < kL; kk += 16)
            mma_bf16(TW(jm), wa + mdesc_step(kk), wb + mdesc_step(kk), idesc_bf16(128, 64, true, true), kk > 0);
          if (c2.last(geo, q1)) {
            // dB^T[n][s] += sum_t C[t][n] dCBsum[t][s],  dC^T[n][t] += sum_s B[s][n] dCBsum[t][s]
#pragma unroll 1
            for (int kk = 0; kk < kL; kk += 16) {
              mma_bf16(ACC_B, sdesc_sw128(bc_c + kk * 128, 2 * kTileLP, 1024), mdesc(sm.dcbs, kL, kk),
                       idesc_bf16(128, 64, true, true), true);
              mma_bf16(ACC_C, sdesc_sw128(bc_b + kk * 128, 2 * kTileLP, 1024), kdesc(sm.dcbs, kL, kk),
                       idesc_bf16(128, 64, true, false), true);
            }
            mma_commit(&sm.acc_full);
            mma_commit(&sm.chunk_empty);
          }
          mma_commit(&sm.s2_done[jm]);
          c2.next(geo);
        }
        if (n < nh) {  // 1b(n)
          const bool first = c1.first(q0);
          bool ok = mbar_wait(&sm.sd_full[j], ph, status, 134);
          ok = ok && mbar_wait(&sm.pre_done[j], ph, status, 135);
          if (ok && first) {
            ok = mbar_wait(&sm.chunk_full, (seg1 + 1) & 1, status, 136);
            if (ok && seg1 >= 0) ok = mbar_wait(&sm.acc_free, seg1 & 1, status, 137);
          }
          if (!ok) break;
          if (first) ++seg1;
          tc_fence_after();
          const BwdcSmem::SD& gs = sm.sd[j];
#pragma unroll 1
          for (int kk = 0; kk < kN; kk += 16)  // [B; C][s or t][n] x [dS | S][n][p]: ddv and Y
            mma_bf16(YD(j), kdesc(sm.BC[0], 2 * kL, kk), mdesc(gs.dS, kN, kk), idesc_bf16(128, 128, false, true),
                     kk > 0);
#pragma unroll 1
          for (int kk = 0; kk < kP; kk += 16) {  // dB^T[n][s] += sum_p dS[n][p] dvd[s][p];  dC^T[n][t] += S dch^T
            mma_bf16(ACC_B, kdesc(gs.dS, kN, kk), kdesc(sm.dvd[j], kL, kk), idesc_bf16(128, 64, false, false),
                     !(first && kk == 0));
            mma_bf16(ACC_C, kdesc(gs.S, kN, kk), kdesc(sm.dch[j], kL, kk), idesc_bf16(128, 64, false, false),
                     !(first && kk == 0));
          }
          mma_commit(&sm.s1b_done[j]);
          c1.next(geo);
        }
      }
      mma_commit(&sm.drain);  // nothing may still be writing TMEM when it is freed
      mbar_wait(&sm.drain, 0, status, 104);
    }
  } else if (warp == kWarpScal) {
    // ------------------------------------------------------------ SC: K1 scalars, up to four heads ahead
    const int t0 = 2 * lane, t1 = t0 + 1;
    ItemCursor hr;
    hr.seek(geo, q0);
    for (int q = 0; q < nh; ++q, hr.next(geo)) {
      const int k = q & 3;
      if (q >= 4 && !mbar_wait(&sm.sc_free[k], ((q >> 2) - 1) & 1, status, 105)) break;
      const int h = hr.h(geo);
      const float A_h = prm.mimo ? 1.f : prm.A[h];
      const int tt = hr.c * kL + t0;
      // streaming loads: these strided reads must not push CB (read by E) out of L1.  Steps past the end of
      // the sequence (a partial last chunk) take dt_raw = -inf: dt' = 0 and da = 0, so they hold the state
      // and (with their zero-filled x, dy, B, C rows) add nothing to any gradient.  MIMO reads da at the
      // first rank of each step, 0 at the others and past the end, with dt' = 1.
      float z0, z1;
      if (prm.mimo) {
        const int msk = (1 << prm.rs) - 1;
        const size_t sr = (size_t)hr.b * (T >> prm.rs);
        z0 = tt < T && (tt & msk) == 0 ? __ldcs(prm.dt_raw + (sr + (tt >> prm.rs)) * H + h) : 0.f;
        z1 = tt + 1 < T && ((tt + 1) & msk) == 0 ? __ldcs(prm.dt_raw + (sr + ((tt + 1) >> prm.rs)) * H + h) : 0.f;
      } else {
        const size_t rr = (size_t)hr.b * T + tt;
        z0 = tt < T ? __ldcs(prm.dt_raw + rr * H + h) : -INFINITY;
        z1 = tt + 1 < T ? __ldcs(prm.dt_raw + (rr + 1) * H + h) : -INFINITY;
      }
      const float d0 = prm.mimo ? 1.f : softplus_fast(z0), d1 = prm.mimo ? 1.f : softplus_fast(z1);
      const float a0 = prm.mimo ? z0 : d0 * A_h, a1 = a0 + (prm.mimo ? z1 : d1 * A_h);
      float inc = a1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      const float c0 = inc - a1 + a0, c1 = inc;
      const float cend = __shfl_sync(0xffffffffu, inc, 31);
      sm.cum[k][t0] = c0;
      sm.cum[k][t1] = c1;
      sm.dtp[k][t0] = d0;
      sm.dtp[k][t1] = d1;
      sm.z[k][t0] = z0;
      sm.z[k][t1] = z1;
      sm.ecum[k][t0] = __expf(c0);
      sm.ecum[k][t1] = __expf(c1);
      sm.dec[k][t0] = __expf(cend - c0);
      sm.dec[k][t1] = __expf(cend - c1);
      if (lane == 0) {
        sm.aend[k] = __expf(cend);
        sm.Ah[k] = A_h;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.sc_ready[k]);
    }
  } else if (warp < kPoolWarps) {
    // ------------------------------------------------------------ the pool
    const int qd = warp & 3, gi = warp >> 2;  // TMEM lane quadrant, index within the quadrant
    const bool e_warp = gi <= qd;             // E block (row block qd, column block gi)
    float cbv[8];   // E: CB[t][16 gi + 8 (lane >> 4) .. + 7], loaded once per chunk run
    float dacc[8];  // E: the run's dCB sum over the same elements
    int seg_e = -1, seg_o = -1;
    ItemCursor ce, co;  // heads i (E) and i - 1 (O, BK, AS)
    ce.seek(geo, q0);
    co.seek(geo, q0);
    // iteration i: O / BK / AS of head i - 1, P of head i + 1, E of head i (i = -1 only runs P of head 0)
    for (int i = -1; i <= nh; ++i) {
      const bool has_prev = i >= 1, has_next = i + 1 < nh, has_cur = i >= 0 && i < nh;
      // ---------------------------------------------------------- S1: O / BK of head i - 1
      {
        const int ip = i - 1, jp = ip & 1, kp = ip & 3;
        const bool run_end = has_prev && co.last(geo, q1);
        // one thread waits for the phase's inputs; the named barrier passes them to the pool
        bool ok = true;
        if (tid == kLead && has_prev) ok = mbar_wait(&sm.s2_done[jp], (ip >> 1) & 1, status, 121);
        if (tid == kLead && ok && run_end) ok = mbar_wait(&sm.acc_full, (seg_o + 1) & 1, status, 122);
        if (named_bar_or(kBarPool, kPoolThreads, !ok)) break;
        tc_fence_after();
        if (has_prev) {
          if (qd < 2) {
            // O: rows s = 32 qd + lane of dv_or (TW) and ddv (YD), columns 16 gi .. 16 gi + 15
            const int s = 32 * qd + lane, c0 = 16 * gi;
            uint32_t ro[16], rd[16];
            tmem_ld16_nowait(taddr(TW(jp), 32 * qd, c0), ro);
            tmem_ld16_nowait(taddr(YD(jp), 32 * qd, c0), rd);
            float xv[16];
            load_row8(sm.xy[ip % 3].x, s, 2 * gi, xv);
            load_row8(sm.xy[ip % 3].x, s, 2 * gi + 1, xv + 8);
            const float e = sm.dec[kp][s], d = sm.dtp[kp][s];
            tmem_wait_ld();
            float sx = 0.f, sd = 0.f, dxv[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              const float ddv = __uint_as_float(rd[u]);
              const float dv = __uint_as_float(ro[u]) + e * ddv;
              sx += dv * xv[u];
              sd += ddv * xv[u];
              dxv[u] = d * dv;
            }
            store_row_bf16(sm.dxs, s, 2 * gi, dxv, 2);
            sm.dvx[jp][gi][s] = sx;
            sm.dde[jp][gi][s] = sd * d;  // sum_p ddv[s][p] v[s][p], this column group
          } else {
            // BK: BLUE on rows t = 32 (qd - 2) + lane of Y (YD lanes 64-127, columns 64 + 16 gi ..); K4 runs in S3
            const int t = 32 * (qd - 2) + lane;
            uint32_t ry[16];
            tmem_ld16_nowait(taddr(YD(jp), 32 * qd, 64 + 16 * gi), ry);
            float gv[16];
            load_row8(sm.xy[ip % 3].dy, t, 2 * gi, gv);
            load_row8(sm.xy[ip % 3].dy, t, 2 * gi + 1, gv + 8);
            tmem_wait_ld();
            float acc = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) acc += gv[u] * __uint_as_float(ry[u]);
            sm.blue[jp][gi][t] = acc;
          }
          if (run_end) {
            // the chunk run ends: dB^T and dC^T (lane n, column s or t) to this CTA's partial slot of the chunk;
            // warp (qd, gi) reads lanes 32 qd .. and columns 32 gi .. of [dB^T | dC^T]
            ++seg_o;
            tc_fence_before();
            named_bar(kBarPool, kPoolThreads);  // O / BK read their TMEM columns before these loads
            tc_fence_after();
            const int n = 32 * qd + lane, col0 = 32 * (gi & 1);
            uint32_t v[32];
            tmem_ld32_nowait(taddr(gi < 2 ? ACC_B : ACC_C, 32 * qd, col0), v);
            tmem_wait_ld();
            if (prm.dB) {
              __nv_bfloat16* out = gi < 2 ? prm.dB : prm.dC;
              const int tb = co.c * kL + col0;
#pragma unroll
              for (int e2 = 0; e2 < 32; ++e2)
                if (tb + e2 < T)
                  out[(((size_t)co.b * T + tb + e2) * prm.G + co.g) * kN + n] = __float2bfloat16_rn(__uint_as_float(v[e2]));
            } else {
              const long long slot = (long long)co.k * prm.nseg +
                                     ((long long)blockIdx.x - cta_of((long long)co.k * prm.hpg, total, gridDim.x));
              float* dst = (gi < 2 ? prm.dB_part : prm.dC_part) + (size_t)slot * kL * kN;
#pragma unroll
              for (int e2 = 0; e2 < 32; ++e2) __stcs(dst + (size_t)(col0 + e2) * kN + n, __uint_as_float(v[e2]));
            }
          }
        }
      }
      // ---------------------------------------------------------- S2: P of head i + 1
      {
        const int in = i + 1, jn = in & 1, kn = in & 3;
        bool ok = true;
        if (tid == kLead && has_next) {
          ok = mbar_wait(&sm.sc_ready[kn], (in >> 2) & 1, status, 110);
          ok = ok && mbar_wait(&sm.xy_full[in % 3], (in / 3) & 1, status, 111);
          if (ok && in >= 2) ok = mbar_wait(&sm.s1b_done[jn], ((in >> 1) - 1) & 1, status, 112);  // 1b(i-1) read dch, dvd
        }
        tc_fence_before();
        fence_proxy_async();
        if (named_bar_or(kBarPool, kPoolThreads, !ok)) break;
        if (tid == kLead && has_prev) {
          tma_store_3d(&tm_dx, sm.dxs, co.h(geo) * kP, co.c * kL, co.b);
          tma_store_commit();
          mbar_arrive(&sm.tmem_free[(i - 1) & 1]);
          mbar_arrive(&sm.xy_empty[(i - 1) % 3]);
          mbar_arrive(&sm.sd_empty[(i - 1) & 1]);
          if (co.last(geo, q1)) mbar_arrive(&sm.acc_free);
        }
        if (has_next) {
          const int t = tid >> 3, jj = tid & 7;  // one 16-byte chunk of x and of dy per thread
          const uint32_t off = sw128_chunk(t, jj);
          const BwdcSmem::XY& sg = sm.xy[in % 3];
          const uint4 rx = *reinterpret_cast<const uint4*>(sg.x + off);
          const uint4 ry = *reinterpret_cast<const uint4*>(sg.dy + off);
          const float fx = sm.dec[kn][t] * sm.dtp[kn][t], fy = sm.ecum[kn][t];
          const uint32_t ix[4] = {rx.x, rx.y, rx.z, rx.w}, iy[4] = {ry.x, ry.y, ry.z, ry.w};
          uint32_t ox[4], oy[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 vx = unpack_bf16(ix[e]), vy = unpack_bf16(iy[e]);
            ox[e] = pack_bf16(fx * vx.x, fx * vx.y);
            oy[e] = pack_bf16(fy * vy.x, fy * vy.y);
          }
          *reinterpret_cast<uint4*>(sm.dvd[jn] + off) = make_uint4(ox[0], ox[1], ox[2], ox[3]);
          *reinterpret_cast<uint4*>(sm.dch[jn] + off) = make_uint4(oy[0], oy[1], oy[2], oy[3]);
        }
      }
      // ---------------------------------------------------------- S3: E of head i, AS of head i - 1
      {
        const int j = i & 1, k = i & 3;
        const bool first = has_cur && ce.first(q0), last = has_cur && ce.last(geo, q1);
        if (has_cur && e_warp && first) {
          ++seg_e;
          load_cb8(prm.CB, ((size_t)ce.k * kL + 16 * qd + (lane & 15)) * kL + 16 * gi + 8 * (lane >> 4), prm.mimo, cbv);
        }
        const int k4w = (warp == 8 || warp == 9 || warp == 12 || warp == 13) ? 2 * ((warp >> 2) - 2) + (warp & 1) : -1;
        bool ok = true;
        if (tid == kLead && has_cur) {
          ok = mbar_wait(&sm.sd_full[j], (i >> 1) & 1, status, 127);  // K4
          ok = ok && mbar_wait(&sm.s1a_done[j], (i >> 1) & 1, status, 117);
          // the bf16 dCB sum of the previous run must have been read by its MMAs
          // (the waiting thread is in an E warp, so seg_e counts its runs)
          if (ok && last && seg_e >= 1) ok = mbar_wait(&sm.chunk_empty, (seg_e - 1) & 1, status, 126);
        }
        fence_proxy_async();
        if (named_bar_or(kBarPool, kPoolThreads, !ok)) break;
        if (tid == kLead && has_next) mbar_arrive(&sm.pre_done[(i + 1) & 1]);
        if (has_cur && e_warp) {
          tc_fence_after();
          // W, the run's dCB sum and the ORANGE row sums of block (qd, gi): rows t = 16 qd + (lane & 15),
          // lane l < 16 columns 16 gi .. + 7, lane l + 16 the other 8 (blocks right of the row's block are
          // zero; see the set-up)
          const int hl = lane >> 4, t = 16 * qd + (lane & 15), s0 = 16 * gi + 8 * hl;
          uint32_t r8[8];  // dW~[t][s0 .. s0 + 7]
          tmem_ld_pair8(taddr(TW(j), 32 * qd, 16 * gi), r8);
          const float ct = sm.cum[k][t];
          tmem_wait_ld();
          float w[8], rowsum = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int s = s0 + e;
            // exp(cum_t - cum_s), masked before the exponential (cum_t - cum_s <= 0 for s <= t)
            // (MIMO: the ranks of one step see each other, cum being flat across them)
            const float ex = ((s >> prm.rs) <= (t >> prm.rs)) ? __expf(fminf(ct - sm.cum[k][s], 0.f)) : 0.f;
            w[e] = cbv[e] * ex;
            const float dg = __uint_as_float(r8[e]) * sm.dtp[k][s];
            const float dcb = dg * ex;
            dacc[e] = first ? dcb : dacc[e] + dcb;
            // ORANGE row sum of dW o dt' o W, with W rounded to bf16 as the dv_or MMA reads it: the column
            // sums come from dv_or (AS), and the two must see the same W or their large terms stop
            // cancelling in dA
            rowsum += dg * __bfloat162float(__float2bfloat16_rn(w[e]));
          }
          store_row_bf16(sm.W[j], t, hl + 2 * gi, w, 1);
          if (last) store_row_bf16(sm.dcbs, t, hl + 2 * gi, dacc, 1);
          rowsum += __shfl_xor_sync(0xffffffffu, rowsum, 16);
          if (lane < 16) sm.drow[j][gi][t] = rowsum;
          tc_fence_before();
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.e_done[j]);
        } else if (has_cur && k4w >= 0) {
          // K4 of head i: <dS_{c+1}, S_c>, thread u takes state row n = u of both tiles
          const int n = 32 * k4w + lane;
          float part = 0.f;
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            float sv[8], dv[8];
            load_row8(sm.sd[j].S, n, c, sv);
            load_row8(sm.sd[j].dS, n, c, dv);
#pragma unroll
            for (int e2 = 0; e2 < 8; ++e2) part += dv[e2] * sv[e2];
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
          if (lane == 0) sm.k4p[j][k4w] = part;
        } else if (warp == kWarpAs && has_prev) {
          // AS of head i - 1: d cum per position, then the K1 backward (suffix sums) to ddt_raw and dA
          const int ip = i - 1, jp = ip & 1, kp = ip & 3;
          const int t0 = 2 * lane, t1 = t0 + 1;
          const float A_h = sm.Ah[kp];
          const float dec0 = sm.dec[kp][t0], dec1 = sm.dec[kp][t1];
          const float vx0 = sm.dvx[jp][0][t0] + sm.dvx[jp][1][t0] + sm.dvx[jp][2][t0] + sm.dvx[jp][3][t0];
          const float vx1 = sm.dvx[jp][0][t1] + sm.dvx[jp][1][t1] + sm.dvx[jp][2][t1] + sm.dvx[jp][3][t1];
          const float de0 = sm.dde[jp][0][t0] + sm.dde[jp][1][t0] + sm.dde[jp][2][t0] + sm.dde[jp][3][t0];
          const float de1 = sm.dde[jp][0][t1] + sm.dde[jp][1][t1] + sm.dde[jp][2][t1] + sm.dde[jp][3][t1];
          const float bl0 = (sm.blue[jp][0][t0] + sm.blue[jp][1][t0] + sm.blue[jp][2][t0] + sm.blue[jp][3][t0]) * sm.ecum[kp][t0];
          const float bl1 = (sm.blue[jp][0][t1] + sm.blue[jp][1][t1] + sm.blue[jp][2][t1] + sm.blue[jp][3][t1]) * sm.ecum[kp][t1];
          // Every term in which cum_s enters through exp(-cum_s) v_s (ORANGE's column sums and K3's
          // exp(cum_end - cum_s)) adds up to -<dv_s, v_s>, with dv the whole gradient of v = dt' x
          float dc0 = sm.drow[jp][0][t0] + sm.drow[jp][1][t0] + sm.drow[jp][2][t0] + sm.drow[jp][3][t0] + bl0 -
                      sm.dtp[kp][t0] * vx0;
          float dc1 = sm.drow[jp][0][t1] + sm.drow[jp][1][t1] + sm.drow[jp][2][t1] + sm.drow[jp][3][t1] + bl1 -
                      sm.dtp[kp][t1] * vx1;
          // chunk-end terms at t = 63: K3's exp(cum_end - cum_s) and K4's exp(cum_end) <dS_{c+1}, S_c>
          float k3sum = de0 * dec0 + de1 * dec1;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) k3sum += __shfl_xor_sync(0xffffffffu, k3sum, o);
          const float k4 = (sm.k4p[jp][0] + sm.k4p[jp][1]) + (sm.k4p[jp][2] + sm.k4p[jp][3]);
          if (lane == 31) dc1 += k3sum + sm.aend[kp] * k4;
          // suffix sums (K1 backward): dda[t] = sum_{u >= t} d cum[u]
          const float pair = dc0 + dc1;
          float suf = pair;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_down_sync(0xffffffffu, suf, o);
            if (lane + o < 32) suf += u;
          }
          const float dda0 = suf, dda1 = suf - dc0;
          const int h = co.h(geo);
          const int tt = co.c * kL + t0;
          if (prm.mimo) {  // d da of a step: the suffix sum from its first rank
            const int msk = (1 << prm.rs) - 1;
            const size_t sr = (size_t)co.b * (T >> prm.rs);
            if (tt < T && (tt & msk) == 0) __stcs(prm.ddt_raw + (sr + (tt >> prm.rs)) * H + h, dda0);
            if (tt + 1 < T && ((tt + 1) & msk) == 0) __stcs(prm.ddt_raw + (sr + ((tt + 1) >> prm.rs)) * H + h, dda1);
          } else {
            const size_t rr = (size_t)co.b * T + tt;
            if (tt < T) __stcs(prm.ddt_raw + rr * H + h, (vx0 + A_h * dda0) * sigmoid_fast(sm.z[kp][t0]));
            if (tt + 1 < T) __stcs(prm.ddt_raw + (rr + 1) * H + h, (vx1 + A_h * dda1) * sigmoid_fast(sm.z[kp][t1]));
          }
          float dAp = dda0 * sm.dtp[kp][t0] + dda1 * sm.dtp[kp][t1];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) dAp += __shfl_xor_sync(0xffffffffu, dAp, o);
          if (lane == 0) prm.dA_part[((size_t)co.b * H + h) * nc + co.c] = dAp;
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.sc_free[kp]);
        }
        // the dx store of this iteration has been read before the next S1 writes the staging tile
        if (tid == kLead && has_prev) tma_store_wait_read0();
      }
      if (has_prev) co.next(geo);
      if (has_cur) ce.next(geo);
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

// The fixed-order sums after the chunk kernel, in one launch:
//   blocks [0, 4 nchunks): a quarter of chunk k's dB, dC (2048 elements, 8 per
//     thread as two float4), the chunk's partial slots added in slot order;
//   the blocks after them: dA[h] = sum over (batch, chunk) of the per-head
//     parts, one warp per head (lane-strided sums, then a fixed shuffle tree).
__global__ void __launch_bounds__(256) k_bwdc_sums(const float* __restrict__ dB_part, const float* __restrict__ dC_part,
                                                   __nv_bfloat16* dB, __nv_bfloat16* dC, const float* __restrict__ dA_part,
                                                   float* dA, long long nchunks, int nseg, long long total, long long grid,
                                                   int hpg, int T, int G, int nc, int b, int H) {
  const long long nb = 4 * nchunks;
  const int lane = threadIdx.x & 31;
  pdl_wait();  // the partials of the chunk kernel before this one
  if ((long long)blockIdx.x >= nb) {
    const int h = (int)(((long long)blockIdx.x - nb) * 8) + (threadIdx.x >> 5);
    if (h >= H) return;
    const int n = b * nc;
    float acc = 0.f;
    for (int i = lane; i < n; i += 32) {
      const int bb = i / nc, c = i - bb * nc;
      acc += dA_part[((size_t)bb * H + h) * nc + c];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) dA[h] = acc;
    return;
  }
  const long long k = blockIdx.x >> 2;
  const int ns = (int)(cta_of((k + 1) * hpg - 1, total, grid) - cta_of(k * hpg, total, grid)) + 1;
  const int g = (int)(k % G);
  const long long bc = k / G;
  const int c = (int)(bc % nc), bb = (int)(bc / nc);
  const float4* pb = reinterpret_cast<const float4*>(dB_part + (size_t)k * nseg * kL * kN);
  const float4* pc = reinterpret_cast<const float4*>(dC_part + (size_t)k * nseg * kL * kN);
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int e4 = (int)(blockIdx.x & 3) * 512 + u * 256 + threadIdx.x;  // float4 index in the chunk's [L][N]
    float4 sb = pb[e4], sc = pc[e4];
    for (int s = 1; s < ns; ++s) {
      const float4 vb = pb[(size_t)s * (kL * kN / 4) + e4], vc = pc[(size_t)s * (kL * kN / 4) + e4];
      sb.x += vb.x, sb.y += vb.y, sb.z += vb.z, sb.w += vb.w;
      sc.x += vc.x, sc.y += vc.y, sc.z += vc.z, sc.w += vc.w;
    }
    const int t = (4 * e4) / kN, n = (4 * e4) % kN;
    if (c * kL + t >= T) continue;  // past the end of the sequence (a partial last chunk)
    const size_t o = (((size_t)bb * T + c * kL + t) * G + g) * kN + n;
    *reinterpret_cast<uint2*>(dB + o) = make_uint2(pack_bf16(sb.x, sb.y), pack_bf16(sb.z, sb.w));
    *reinterpret_cast<uint2*>(dC + o) = make_uint2(pack_bf16(sc.x, sc.y), pack_bf16(sc.z, sc.w));
  }
}

struct BwdcLayout {
  long long total, nchunks;
  int grid, nseg;
};

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

BwdcLayout layout(const Dims& d, int sms) {
  BwdcLayout l;
  l.nchunks = (long long)d.b * d.nc * d.G;
  l.total = l.nchunks * d.hpg;
  l.grid = (int)(l.total < sms ? l.total : sms);
  if (l.grid < 1) l.grid = 1;
  // most CTAs one chunk's heads can span: ceil(hpg / min items per CTA) + 1
  const long long per = l.total / l.grid;
  l.nseg = (int)((d.hpg + per - 1) / per + 1);
  return l;
}

struct BwdcWs {
  __nv_bfloat16* states;   // S_c   [b,H,nc][N][P]
  __nv_bfloat16* dstates;  // dS_{c+1}
  float* CB;               // [b,nc,G,L,L]
  float* dB_part;
  float* dC_part;
  float* dA_part;
};

BwdcWs carve(const Dims& d, const BwdcLayout& l, Carver& cv) {
  BwdcWs w;
  w.states = cv.take<__nv_bfloat16>((size_t)d.b * d.H * d.nc * kN * kP);
  w.dstates = cv.take<__nv_bfloat16>((size_t)d.b * d.H * d.nc * kN * kP);
  w.CB = cv.take<float>((size_t)l.nchunks * kL * kL);
  w.dB_part = cv.take<float>((size_t)l.nchunks * l.nseg * kL * kN);
  w.dC_part = cv.take<float>((size_t)l.nchunks * l.nseg * kL * kN);
  w.dA_part = cv.take<float>((size_t)d.b * d.H * d.nc);
  return w;
}

// The workspace is sized for the largest grid (the device's SM count may not
// be known when it is sized): slots for a grid of 1024 CTAs cover any smaller grid.
constexpr int kMaxGrid = 1024;

}  // namespace

size_t tc_backward_ws(const Dims& problem) {
  const Dims d = tc_dims(problem);
  Carver cv(nullptr);
  carve(d, layout(d, kMaxGrid), cv);
  return cv.off;
}

cudaError_t tc_backward(const Dims& problem, const BwdArgs& a, void* ws, cudaStream_t st) {
  const Dims d = tc_dims(problem);
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  const BwdcLayout l = layout(d, sms < kMaxGrid ? sms : kMaxGrid);
  const BwdcLayout lmax = layout(d, kMaxGrid);
  Carver cv(ws);
  BwdcWs w = carve(d, lmax, cv);
  int* status = static_cast<int*>(ws);
  // the chunk states: replayed from the leaf inputs, or the forward's stash (the same kernel on the same
  // inputs wrote it, so the two give the same bits)
  const __nv_bfloat16* states = a.states_in ? a.states_in : w.states;
  // the replay (unless stashed) and the reverse scan are independent: one launch runs both, plus CB; from
  // checkpoints the replay runs as short independent segments, started from the checkpointed fp32 states
  // (the whole-sequence replay computes the same states with the same operations, so the same bits)
  const ScanSide fwd{a.x, a.s0, nullptr, w.states, nullptr, a.ckpt_in, a.ckpt_every};
  const ScanSide rev{a.dy, a.ds_final, a.ds0, w.dstates};
  cudaError_t e = tc_scans(d, a.states_in ? nullptr : &fwd, &rev, a.B, a.C, a.dt_raw, a.A, w.CB, status, st);
  if (e != cudaSuccess) return e;
  const uint64_t srows = (uint64_t)d.b * d.H * d.nc * kN;
  CUtensorMap tx, tdy, tdx, tb, tcm, ts, tds;
  e = make_tmap_seq_bf16(&tx, a.x, d, (uint64_t)d.H * kP);
  if (e == cudaSuccess) e = make_tmap_seq_bf16(&tdy, a.dy, d, (uint64_t)d.H * kP);
  if (e == cudaSuccess) e = make_tmap_seq_bf16(&tdx, a.dx, d, (uint64_t)d.H * kP);
  if (e == cudaSuccess) e = make_tmap_bc_bf16(&tb, a.B, d);
  if (e == cudaSuccess) e = make_tmap_bc_bf16(&tcm, a.C, d);
  if (e == cudaSuccess) e = make_tmap_2d_bf16(&ts, states, kP, srows, 64, kN);
  if (e == cudaSuccess) e = make_tmap_2d_bf16(&tds, w.dstates, kP, srows, 64, kN);
  if (e != cudaSuccess) return e;
  // partial slots use the layout of the launched grid (nseg of the largest grid bounds it)
  const bool direct = d.hpg == 1;
  BwdcParams prm{a.dt_raw, a.A,   w.CB, a.ddt_raw, w.dA_part, w.dB_part, w.dC_part, status,
                 d.T,      d.H,   d.G,  d.hpg,     d.nc,      lmax.nseg, (int)l.total, d.variant == kMimo, d.rs,
                 direct ? static_cast<__nv_bfloat16*>(a.dB) : nullptr,
                 direct ? static_cast<__nv_bfloat16*>(a.dC) : nullptr};
  const int smem = (int)sizeof(BwdcSmem) + 1024;
  e = cudaFuncSetAttribute(k_tc_bwdc, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  SSD_LAUNCH("k_tc_bwd_chunk", st,
             e = launch_after(k_tc_bwdc, l.grid, kThreads, smem, st, tx, tdy, tdx, tb, tcm, ts, tds, prm));
  if (e != cudaSuccess) return e;
  // dB, dC blocks unless the chunk kernel wrote them; dA blocks unless there is no A (MIMO)
  const long long nchunks_sum = direct ? 0 : l.nchunks;
  const long long sum_blocks = 4 * nchunks_sum + (a.dA ? (d.H + 7) / 8 : 0);
  if (sum_blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  if (sum_blocks > 0)
    SSD_LAUNCH("k_tc_bwd_sums", st,
               e = launch_after(k_bwdc_sums, (unsigned)sum_blocks, 256, 0, st, (const float*)w.dB_part,
                                (const float*)w.dC_part, static_cast<__nv_bfloat16*>(a.dB),
                                static_cast<__nv_bfloat16*>(a.dC), (const float*)w.dA_part, a.dA, nchunks_sum,
                                lmax.nseg, l.total, (long long)l.grid, d.hpg, d.T, d.G, d.nc, d.b, d.H));
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace ssd
