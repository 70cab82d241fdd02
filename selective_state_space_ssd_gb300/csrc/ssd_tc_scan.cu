// The two sequential state scans of the Mamba-2 chunkwise algorithm on
// tcgen05 tensor cores (bf16 io, chunk L = 64, head dim P = 64, state N = 128).
//
// Forward (the K3 chunk state and K4 state passing of the burn-mamba page
// "combined_backward.rs", section "RECOMPUTE FORWARD INTERMEDIATES"):
//     S_0 = s0,   S_{c+1} = exp(cum_end) S_c + B_c^T dvd_c,
//     dvd[s][p] = exp(cum_end - cum_s) dt'_s x[s][p];
// it writes every chunk-input state S_c (bf16, [n][p] tiles) and S_nc = s_final.
// Reverse (the same recurrence transposed: the page's "K4 backward step", which
// carries d_s_{i+1} back as decay_i d_s_{i+1} plus the BLUE term):
//     dS_nc = ds_final,   dS_c = exp(cum_end) dS_{c+1} + C_c^T dch_c,
//     dch[t][p] = exp(cum_t) dy[t][p];
// it writes dS_{c+1} for every chunk c (bf16 tiles) and dS_0 = ds0.
//
// One CTA owns one (batch, head); three CTAs share an SM.  The fp32 state S
// lives in 64 TMEM columns (thread n of the state warps owns row n) and the
// chunk's contribution P = K^T U in 64 more: the MMA writes P for chunk c while
// the state warps still finish chunk c - 1, and the state warps then form
// S <- exp(cum_end) S + P a quarter of the row at a time; the bf16 copy of the
// new state (the next chunk's input state) goes out through shared memory, one
// TMA store of 32 rows per state warp.
// The recurrence's critical path per chunk is one P read-out and a few FMAs;
// the MMA is off it.
//
// Warp roles (288 threads): warps 0-3 state, warps 4-5 scale the U tile in
// place (x -> dvd or dy -> dch), warp 6 K1 scalars (softplus, in-chunk cumsum,
// exponentials), warp 7 TMA producer, warp 8 MMA issuer and TMEM owner.
// Every wait is bounded; on a timeout the kernel records a code in the
// workspace status word and stops.
//
// One launch carries every independent piece of sequential-scan work a call
// has, in grid order: the forward chains, the reverse chains, then the K2 tiles
// CB = C B^T (one (chunk, group) per CTA, fp32; the chunk kernels read them).
// The backward's forward replay and reverse scan do not depend on each other,
// so they share the launch: a chain is a latency chain of 64 steps, and the
// SMs' third CTA slots (left partly idle by 320 chains on 152 SMs) take the
// other direction's chains.  The CB tiles come last and fill the slots the
// chains leave free, instead of costing a launch of their own.
#include <string.h>

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
constexpr uint32_t kTmemCols = 128;  // S in columns 0-63, P in 64-127
constexpr int kScal = 4;             // K1 scalars run up to four chunks ahead
constexpr int kStK = 2;              // B / C tiles (mostly L2 hits: every head of a group reads them)

// kStU: depth of the x / dy ring, the HBM stream whose latency the ring hides (three stages when three
// CTAs still fit an SM, else two).
template <int kStU>
struct alignas(1024) ScanSmem {
  uint8_t u[kStU][kTileLP];  // x or dy [t][p], scaled in place to dvd or dch
  uint8_t k[kStK][kTileLN];  // B or C [t][n], two 64-column atoms
  uint8_t out[kTileNP];      // bf16 state tile [n][p] on its way out; state warp w owns rows 32 w .. 32 w + 31
  float scale[kScal][kL];    // per-row factor of U: exp(cum_end - cum) dt' or exp(cum); ring of kScal chunks
  float aend[kScal];         // exp(cum_end)
  uint64_t full_u[kStU], empty_u[kStU], pre_done[kStU], full_k[kStK], empty_k[kStK];
  uint64_t sc_ready[kScal], sc_free[kScal];
  uint64_t p_ready, p_free, drain;
  uint32_t tmem_slot;
};

struct ScanParams {
  const float* dt_raw;
  const float* A;
  const float* init;  // s0 or ds_final [b,H,P,N]; s0 may be null (zeros)
  float* fin;         // s_final or ds0 [b,H,P,N]; null: not written
  int* status;
  int T, H, hpg, nc;
  int mimo, rs;  // MIMO: dt_raw holds da [b, T >> rs, H] (the fused positions' dt' is 1), A is unused
  // checkpoints (forward only), fp32 [b, H, nk][P][N], entry k = the state entering chunk k * every:
  float* ckpt_out;       // written by the whole-sequence chains (entry 0 = s0), or null
  const float* ckpt_in;  // not null: the chains are segments of `every` chunks, each started from its entry
  int every, nk;
};

// One direction's chains: the tensor maps of U (x or dy), K (B or C) and the state tiles out, and the scalars.
struct ScanJob {
  CUtensorMap u, k, out;
  ScanParams prm;
};

// One (batch, head) chain, run by the whole CTA: the whole sequence, or (forward, from checkpoints) the
// segment `seg` of `every` chunks, which writes the input states of its chunks and nothing else.
template <bool kRev, int kStU>
__device__ __forceinline__ void scan_chain(const ScanJob& job, int h, int b, int seg, uint8_t* smem) {
  ScanSmem<kStU>& sm = *reinterpret_cast<ScanSmem<kStU>*>(smem);
  const CUtensorMap& tm_u = job.u;
  const CUtensorMap& tm_k = job.k;
  const CUtensorMap& tm_out = job.out;
  const ScanParams& prm = job.prm;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = prm.T, H = prm.H, nc = prm.nc;
  const int g = h / prm.hpg;
  const size_t row0 = (size_t)b * T;
  const size_t unit = (size_t)b * H + h;
  int* status = prm.status;
  const bool segmented = !kRev && prm.ckpt_in;
  const int cbeg = segmented ? seg * prm.every : 0;
  const int clen = segmented ? min(prm.every, nc - cbeg) : nc;
  // state updates: one per chunk of the whole sequence (the last gives fin), one per chunk but the last of a
  // segment (its last chunk's input state is the last one it writes)
  const int nsteps = segmented ? clen - 1 : nc;
  auto chunk_of = [&](int r) { return kRev ? nc - 1 - r : cbeg + r; };

  if (tid == 0) {
    for (int s = 0; s < kStU; ++s) {
      mbar_init(&sm.full_u[s], 1);
      mbar_init(&sm.empty_u[s], 1);  // MMA commit (it waited for the scale warps)
      mbar_init(&sm.pre_done[s], 1);
    }
    for (int s = 0; s < kStK; ++s) {
      mbar_init(&sm.full_k[s], 1);
      mbar_init(&sm.empty_k[s], 1);  // MMA commit
    }
    for (int s = 0; s < kScal; ++s) {
      mbar_init(&sm.sc_ready[s], 1);
      mbar_init(&sm.sc_free[s], 5);  // scale warps + the four state warps
    }
    mbar_init(&sm.p_ready, 1);
    mbar_init(&sm.p_free, 4);  // the four state warps have read P
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
      int su = 0, pu = 0;  // x / dy ring slot and its phase
      for (int r = 0; r < nsteps; ++r) {
        const int sk = r & 1, c = chunk_of(r);
        if (r >= kStU && !mbar_wait(&sm.empty_u[su], pu ^ 1, status, 81)) break;
        mbar_expect_tx(&sm.full_u[su], kTileLP);
        tma_load_3d(sm.u[su], &tm_u, h * kP, c * kL, b, &sm.full_u[su]);
        if (r >= kStK && !mbar_wait(&sm.empty_k[sk], ((r >> 1) - 1) & 1, status, 80)) break;
        mbar_expect_tx(&sm.full_k[sk], kTileLN);
        for (int a = 0; a < 2; ++a)
          tma_load_4d(sm.k[sk] + a * (kTileLN / 2), &tm_k, a * 64, g, c * kL, b, &sm.full_k[sk]);
        if (++su == kStU) su = 0, pu ^= 1;
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t tP = tmem + 64u;
      bool ok = true;
      int su = 0, pu = 0;
      for (int r = 0; r < nsteps && ok; ++r) {
        const int sk = r & 1;
        ok = mbar_wait(&sm.pre_done[su], pu, status, 82);
        ok = ok && mbar_wait(&sm.full_k[sk], (r >> 1) & 1, status, 79);
        ok = ok && (r == 0 || mbar_wait(&sm.p_free, (r - 1) & 1, status, 83));
        if (!ok) break;
        tc_fence_after();
        // P[n][p] = sum_t K[t][n] U[t][p]: A = K^T (MN-major), B = U (MN-major)
#pragma unroll
        for (int kk = 0; kk < kL; kk += 16)
          mma_bf16(tP, mdesc(sm.k[sk], kL, kk), mdesc(sm.u[su], kL, kk), idesc_bf16(128, 64, true, true), kk > 0);
        mma_commit(&sm.p_ready);
        mma_commit(&sm.empty_u[su]);
        mma_commit(&sm.empty_k[sk]);
        if (++su == kStU) su = 0, pu ^= 1;
      }
      // nothing may still be writing TMEM when it is freed
      mma_commit(&sm.drain);
      mbar_wait(&sm.drain, 0, status, 84);
    }
  } else if (warp == kWarpScal) {
    // ------------------------------------------------------------ K1 scalars.  The dt_raw reads (64
    //   strided floats per chunk) are issued two chunks ahead of their use.  Steps past the end of the
    //   sequence (the tail of a partial last chunk) read dt_raw = -inf: dt' = 0 and da = 0 there, so they
    //   leave the state as it is, and their U rows are zeros (TMA fill) as well.
    //   MIMO reads da at the first rank of each step and 0 at the others (dt' = 1 everywhere).
    const float A_h = prm.mimo ? 1.f : prm.A[h];
    const int t0 = 2 * lane, t1 = t0 + 1;
    const int msk = (1 << prm.rs) - 1;
    const size_t srow0 = (size_t)b * (T >> prm.rs);
    auto fetch = [&](int r, float& z0, float& z1) {
      if (r < nsteps) {
        const int tt = chunk_of(r) * kL + t0;
        if (prm.mimo) {
          z0 = tt < T && (tt & msk) == 0 ? prm.dt_raw[(srow0 + (tt >> prm.rs)) * H + h] : 0.f;
          z1 = tt + 1 < T && ((tt + 1) & msk) == 0 ? prm.dt_raw[(srow0 + ((tt + 1) >> prm.rs)) * H + h] : 0.f;
        } else {
          const size_t rr = (size_t)row0 + tt;
          z0 = tt < T ? prm.dt_raw[rr * H + h] : -INFINITY;
          z1 = tt + 1 < T ? prm.dt_raw[(rr + 1) * H + h] : -INFINITY;
        }
      }
    };
    auto step = [&](int r, float z0, float z1) -> bool {
      const int s = r % kScal;
      if (r >= kScal && !mbar_wait(&sm.sc_free[s], (r / kScal - 1) & 1, status, 85)) return false;
      const float d0 = prm.mimo ? 1.f : softplus_fast(z0), d1 = prm.mimo ? 1.f : softplus_fast(z1);
      const float a0 = prm.mimo ? z0 : d0 * A_h, a1 = a0 + (prm.mimo ? z1 : d1 * A_h);
      float inc = a1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      const float c0 = inc - a1 + a0, c1 = inc;
      const float cend = __shfl_sync(0xffffffffu, inc, 31);
      if (kRev) {
        sm.scale[s][t0] = __expf(c0);
        sm.scale[s][t1] = __expf(c1);
      } else {
        sm.scale[s][t0] = __expf(cend - c0) * d0;
        sm.scale[s][t1] = __expf(cend - c1) * d1;
      }
      if (lane == 0) sm.aend[s] = __expf(cend);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.sc_ready[s]);
      return true;
    };
    float za0 = 0.f, za1 = 0.f, zb0 = 0.f, zb1 = 0.f;
    fetch(0, za0, za1);
    fetch(1, zb0, zb1);
    for (int r = 0; r < nsteps; r += 2) {
      if (!step(r, za0, za1)) break;
      fetch(r + 2, za0, za1);
      if (r + 1 < nsteps) {
        if (!step(r + 1, zb0, zb1)) break;
        fetch(r + 3, zb0, zb1);
      }
    }
  } else if (warp >= kWarpScale0) {
    // ------------------------------------------------------------ scale warps: U *= scale (per row), as bf16x2
    //   products with the row's factor rounded to bf16 (a relative error below 2^-9 on each row of dvd / dch,
    //   which only ever enter bf16 MMAs): one instruction per two elements instead of unpacking to fp32, which
    //   had made this transform the longest stage of every chain step
    const int pt = tid - 32 * kWarpScale0;  // 0..63
    int s = 0, ps = 0;  // x / dy ring slot and its phase
    for (int r = 0; r < nsteps; ++r) {
      const int k = r % kScal;
      bool ok = mbar_wait(&sm.sc_ready[k], (r / kScal) & 1, status, 86);
      ok = ok && mbar_wait(&sm.full_u[s], ps, status, 87);
      if (named_bar_or(2, 64, !ok)) break;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = pt + 64 * i, t = q >> 3, j = q & 7;
        uint4* p = reinterpret_cast<uint4*>(sm.u[s] + sw128_chunk(t, j));
        const uint4 w = *p;
        const uint32_t f2 = pack_bf16(sm.scale[k][t], sm.scale[k][t]);  // the row's factor, rounded to bf16
        *p = make_uint4(mul_bf16x2(w.x, f2), mul_bf16x2(w.y, f2), mul_bf16x2(w.z, f2), mul_bf16x2(w.w, f2));
      }
      fence_proxy_async();
      named_bar(2, 64);
      if (pt == 0) {
        mbar_arrive(&sm.pre_done[s]);
        mbar_arrive(&sm.sc_free[k]);
      }
      if (++s == kStU) s = 0, ps ^= 1;
    }
  } else {
    // ------------------------------------------------------------ state warps 0-3 (thread n owns row n)
    const int n = tid;
    const uint32_t srow = taddr(tmem, 32 * warp, 0), prow = taddr(tmem, 32 * warp, 64);
    const size_t fbase = unit * kP * kN;
    const float* init = segmented ? prm.ckpt_in + ((size_t)unit * prm.nk + seg) * kP * kN : prm.init;
    const size_t ibase = segmented ? 0 : fbase;
    // checkpoint k of this chain (whole-sequence forward chains only)
    auto ckpt = [&](int k) -> float* {
      return !kRev && prm.ckpt_out ? prm.ckpt_out + ((size_t)unit * prm.nk + k) * kP * kN : nullptr;
    };
    uint8_t* slice = sm.out + 4096 * warp;  // this warp's 32 rows of the out tile
    // this warp's rows of the out tile to the input state of chunk c (rows of 64 bf16, [b,H,nc][N][P])
    auto send = [&](int c) {
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&tm_out, slice, 0, (int)((unit * nc + c) * kN) + 32 * warp);
        tma_store_commit();
      }
    };
    float* ck0 = ckpt(0);
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {  // S = init: into TMEM, and out as the first chunk's input state
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = init ? init[ibase + (size_t)(16 * q + e) * kN + n] : 0.f;
      tmem_st16(srow + 16 * q, v);
      store_row_bf16(sm.out, n, 2 * q, v, 2);
      if (ck0) {
#pragma unroll
        for (int e = 0; e < 16; ++e) ck0[(size_t)(16 * q + e) * kN + n] = v[e];
      }
    }
    send(chunk_of(0));
    tmem_wait_st();
    for (int r = 0; r < nsteps; ++r) {
      const int k = r % kScal;
      bool ok = mbar_wait(&sm.sc_ready[k], (r / kScal) & 1, status, 89);
      ok = ok && mbar_wait(&sm.p_ready, r & 1, status, 88);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const float a = sm.aend[k];
      const bool more = r + 1 < clen;
      float* ckn = !kRev && prm.ckpt_out && more && (r + 1) % prm.every == 0 ? ckpt((r + 1) / prm.every) : nullptr;
      if (more) {  // the previous store has read the slice
        if (lane == 0) tma_store_wait_read0();
        __syncwarp();
      }
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t sv[16], pv[16];
        tmem_ld16_nowait(srow + 16 * q, sv);
        tmem_ld16_nowait(prow + 16 * q, pv);
        tmem_wait_ld();
        if (q == 3) {  // P and exp(cum_end) fully read by this warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&sm.p_free);
            mbar_arrive(&sm.sc_free[k]);
          }
        }
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = fmaf(a, __uint_as_float(sv[e]), __uint_as_float(pv[e]));
        tmem_st16(srow + 16 * q, v);
        if (ckn) {
#pragma unroll
          for (int e = 0; e < 16; ++e) ckn[(size_t)(16 * q + e) * kN + n] = v[e];
        }
        if (more) {
          store_row_bf16(sm.out, n, 2 * q, v, 2);
        } else if (prm.fin) {
#pragma unroll
          for (int e = 0; e < 16; ++e) prm.fin[fbase + (size_t)(16 * q + e) * kN + n] = v[e];
        }
      }
      if (more) send(chunk_of(r + 1));
      tmem_wait_st();
    }
    if (lane == 0) tma_store_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// CB[b][c][g][t][s] = sum_n C[b, c*L+t, g, n] B[b, c*L+s, g, n] (fp32) for one (chunk, group): the C and
// B tiles come in by TMA (two 64-column atoms each, K-major), one thread issues the eight K = 16 steps of one
// M = 64, N = 64 MMA, and warps 0-3 write the accumulator rows out; the other warps only join the barriers.
struct CbJob {
  CUtensorMap c, b;
  float* CB;  // [b, nc, G, L, L]: fp32, or bf16 when bf16 is set (MIMO: one tile per head, twice the bytes of y)
  int* status;
  int G, nc;
  int bf16;
};

struct alignas(1024) CbSmem {
  uint8_t C[2][kL * 64 * 2];  // [atom][t][64 n] bf16, SW128
  uint8_t B[2][kL * 64 * 2];  // [atom][s][64 n]
  uint64_t full, done;
  uint32_t tmem_slot;
};
static_assert(sizeof(CbSmem) <= sizeof(ScanSmem<2>), "a CB tile runs in a scan CTA's shared memory");

__device__ __forceinline__ void cb_tile(const CbJob& job, int k, uint8_t* smem) {
  CbSmem& sm = *reinterpret_cast<CbSmem*>(smem);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int g = k % job.G, bc = k / job.G;
  const int c = bc % job.nc, b = bc / job.nc;
  int* status = job.status;
  if (tid == 0) {
    mbar_init(&sm.full, 1);
    mbar_init(&sm.done, 1);
    mbar_init_fence();
  }
  if (warp == 0) tmem_alloc(&sm.tmem_slot, 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_slot;
  if (tid == 0) {
    mbar_expect_tx(&sm.full, 4 * kL * 64 * 2);
    for (int a = 0; a < 2; ++a) {
      tma_load_4d(sm.C[a], &job.c, 64 * a, g, c * kL, b, &sm.full);
      tma_load_4d(sm.B[a], &job.b, 64 * a, g, c * kL, b, &sm.full);
    }
    if (mbar_wait(&sm.full, 0, status, 61)) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kN; kk += 16)
        mma_bf16(tmem, kdesc(sm.C[0], kL, kk), kdesc(sm.B[0], kL, kk), idesc_bf16(64, 64, false, false), kk > 0);
    }
    mma_commit(&sm.done);  // arrives even when nothing was issued, so the readers below never wait forever
  }
  if (warp < 4) {
    __syncwarp();
    const bool ok = mbar_wait(&sm.done, 0, status, 62);
    tc_fence_after();
    if (ok && *status == 0) {
      // M = 64 accumulator: row t = 16 warp + (lane & 15) in lane 32 warp + (lane & 15); lanes 16-31 take
      // columns 32-63
      const int lane = tid & 31, t = 16 * warp + (lane & 15), s0 = 32 * (lane >> 4);
      uint32_t v[32];
      tmem_ld_pair32(taddr(tmem, 32 * warp, 0), v);
      tmem_wait_ld();
      const size_t o = ((size_t)k * kL + t) * kL + s0;
      if (job.bf16) {
        uint4* out = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(job.CB) + o);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          out[e] = make_uint4(pack_bf16(__uint_as_float(v[8 * e]), __uint_as_float(v[8 * e + 1])),
                              pack_bf16(__uint_as_float(v[8 * e + 2]), __uint_as_float(v[8 * e + 3])),
                              pack_bf16(__uint_as_float(v[8 * e + 4]), __uint_as_float(v[8 * e + 5])),
                              pack_bf16(__uint_as_float(v[8 * e + 6]), __uint_as_float(v[8 * e + 7])));
      } else {
        float4* out = reinterpret_cast<float4*>(job.CB + o);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          out[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]), __uint_as_float(v[4 * e + 2]),
                               __uint_as_float(v[4 * e + 3]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// Everything one launch runs, and how the grid splits: blocks [0, n_fwd) are forward chains, the next n_rev
// reverse chains (chain i is (batch i / H, head i % H)), the last n_cb CB tiles (tile i is (chunk, group) i).
struct ScanLaunch {
  ScanJob fwd, rev;
  CbJob cb;
  int n_fwd, n_rev, n_cb, H;
  int nk;         // forward blocks per (batch, head): its segments, or 1
  int rev_first;  // the reverse chains come first in the grid (the forward ones are short segments)
};

template <int kStU>
__global__ void __launch_bounds__(kThreads, 3) k_scan(const __grid_constant__ ScanLaunch job) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  pdl_trigger();  // the chunk kernel after this launch may take SMs as they free up (it waits for this launch)
  int i = blockIdx.x;
  if (job.rev_first) {
    if (i < job.n_rev) {
      scan_chain<true, kStU>(job.rev, i % job.H, i / job.H, 0, smem);
      return;
    }
    i -= job.n_rev;
  }
  if (i < job.n_fwd) {
    const int unit = i / job.nk;
    scan_chain<false, kStU>(job.fwd, unit % job.H, unit / job.H, i - unit * job.nk, smem);
    return;
  }
  i -= job.n_fwd;
  if (!job.rev_first) {
    if (i < job.n_rev) {
      scan_chain<true, kStU>(job.rev, i % job.H, i / job.H, 0, smem);
      return;
    }
    i -= job.n_rev;
  }
  cb_tile(job.cb, i, smem);
}

// Three x / dy stages when three CTAs of them still fit an SM (all (batch, head) chains of one direction stay
// resident at once), else two.
template <int kStU>
cudaError_t launch_stages(const ScanLaunch& job, const char* name, cudaStream_t st, bool* fits) {
  const int smem = (int)sizeof(ScanSmem<kStU>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(k_scan<kStU>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_scan<kStU>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  if (fits) {  // shared memory of three CTAs (each with the per-block reservation) against the SM's
    int dev = 0, per_sm = 0, reserved = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess) return e;
    *fits = 3ll * (smem + reserved) <= per_sm;
    if (!*fits) return cudaSuccess;
  }
  const unsigned grid = (unsigned)(job.n_fwd + job.n_rev + job.n_cb);
  SSD_LAUNCH(name, st, k_scan<kStU><<<grid, kThreads, smem, st>>>(job));
  return cudaGetLastError();
}

}  // namespace

size_t tc_scan_states_bytes(const Dims& d) { return (size_t)d.b * d.H * d.nc * kN * kP * sizeof(__nv_bfloat16); }

size_t tc_checkpoints_bytes(const Dims& d, int every) {
  const size_t nk = ((size_t)d.nc + every - 1) / every;
  return (size_t)d.b * d.H * nk * kP * kN * sizeof(float);
}

cudaError_t tc_scans(const Dims& d, const ScanSide* fwd, const ScanSide* rev, const void* B, const void* C,
                     const float* dt_raw, const float* A, float* CB, int* status, cudaStream_t st) {
  const uint64_t srows = (uint64_t)d.b * d.H * d.nc * kN;
  const long long chains = (long long)d.b * d.H, tiles = (long long)d.b * d.nc * d.G;
  const bool segmented = fwd && fwd->ckpt_in;
  const int every = fwd && (fwd->ckpt_in || fwd->ckpt_out) ? fwd->every : 0;
  if (every < 0 || (fwd && (fwd->ckpt_in || fwd->ckpt_out) && every < 1)) return cudaErrorInvalidValue;
  const int nk = every > 0 ? (d.nc + every - 1) / every : 1;
  const long long fwd_blocks = fwd ? chains * (segmented ? nk : 1) : 0;
  if (fwd_blocks + (rev ? chains : 0) + tiles > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  ScanLaunch job;
  memset(&job, 0, sizeof(job));
  cudaError_t e = cudaSuccess;
  const ScanSide* sides[2] = {fwd, rev};
  ScanJob* jobs[2] = {&job.fwd, &job.rev};
  for (int r = 0; r < 2 && e == cudaSuccess; ++r) {
    const ScanSide* s = sides[r];
    if (!s) continue;
    ScanJob& j = *jobs[r];
    e = make_tmap_seq_bf16(&j.u, s->u, d, (uint64_t)d.H * kP);
    if (e == cudaSuccess) e = make_tmap_bc_bf16(&j.k, r == 0 ? B : C, d);
    if (e == cudaSuccess) e = make_tmap_2d_bf16(&j.out, s->states, kP, srows, 64, 32);
    j.prm = ScanParams{dt_raw, A,  s->init, s->fin, status, d.T, d.H, d.hpg, d.nc, d.variant == kMimo, d.rs,
                       s->ckpt_out, s->ckpt_in, every, nk};
  }
  if (e == cudaSuccess) e = make_tmap_bc_bf16(&job.cb.c, C, d);
  if (e == cudaSuccess) e = make_tmap_bc_bf16(&job.cb.b, B, d);
  if (e != cudaSuccess) return e;
  job.cb.CB = CB;
  job.cb.status = status;
  job.cb.G = d.G;
  job.cb.nc = d.nc;
  job.cb.bf16 = d.variant == kMimo;
  job.n_fwd = (int)fwd_blocks;
  job.n_rev = rev ? (int)chains : 0;
  job.nk = segmented ? nk : 1;
  job.rev_first = segmented ? 1 : 0;
  job.n_cb = (int)tiles;
  job.H = d.H;
  const char* name = fwd && rev ? "k_tc_scan_pair_cb" : fwd ? "k_tc_states_cb" : "k_tc_dstates_cb";
  bool fits = false;
  e = launch_stages<3>(job, name, st, &fits);
  if (e != cudaSuccess || fits) return e;
  return launch_stages<2>(job, name, st, nullptr);
}

}  // namespace ssd
