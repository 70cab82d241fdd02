/*
 * Float64 CPU oracle for the selective state-space scan and its VJP.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file (through oracle/__init__.py).  The CUDA
 * library neither includes, links nor calls anything here, and nothing here
 * includes or calls the CUDA library.
 *
 * What it computes is the plain definition of the method, one (batch, head)
 * unit at a time, in the order the method states it:
 *
 *   dt'_t = softplus(dt_raw_t)
 *   s_t   = exp(dt'_t * A) * s_{t-1} + dt'_t * x_t (outer) B_t
 *   y_t   = s_t . C_t                      (the updated state s_t)
 *
 * ("S1-31: SSM_SCAN_BACK — Mamba has a backward", opening paragraph: the
 * Mamba-2 branch has one scalar decay per head, the Mamba-1 branch one decay
 * per state.)  The MIMO-rank form of the Mamba-3 page (combined_backward.rs,
 * "ORANGE backward" and "BLUE backward" formulas) takes a pre-combined
 * da = dt'*A and R (v, B, C) triples per step:
 *
 *   s_t     = exp(da_t) * s_{t-1} + sum_r v_{t,r} (outer) B_{t,r}
 *   y_{t,r} = s_t . C_{t,r}
 *
 * The backward is the store-all reverse-time VJP of the SSM_SCAN_BACK page
 * ("Two things that are easy to get wrong"): all T+1 states are recomputed
 * and kept, the state gradient is seeded with the (nonzero) upstream gradient
 * of the final state, and t walks from T-1 down to 0.  The loop shape
 * (accumulate the output's contribution into dS, read out the per-step
 * gradients, then decay dS) is that of the KDA notes, section
 * "反向传播推导", steps 1-5.
 *
 * Per-head outputs that a group of heads shares (dB, dC in the Mamba-2
 * branch, and dB, dC over all channels in the Mamba-1 branch) and the
 * per-head dA summed over batch and time are reduced in a fixed order that
 * does not depend on the number of threads ("Threaded by sequence, not by
 * head": one owner per output, no atomics).
 *
 * A `mutation` argument plants exactly one of the five defects of the
 * SSM_SCAN_BACK page's verification table, so that a test can show that its
 * finite-difference check catches each of them:
 *   1  drop the dA path from d(dt)
 *   2  seed the state gradient with zeros
 *   3  drop y's own contribution to dS
 *   4  use s_{t-1} where s_t belongs in dC
 *   5  drop the softplus derivative
 * mutation = 0 is the correct VJP.
 *
 * Build: gcc -O2 -fPIC -shared -pthread (no -ffast-math); exp/log1p are the
 * C library's double-precision functions.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- helpers */

static double softplus(double z) { return fmax(z, 0.0) + log1p(exp(-fabs(z))); }

/* d softplus / dz */
static double sigmoid(double z) {
  if (z >= 0.0) return 1.0 / (1.0 + exp(-z));
  double e = exp(z);
  return e / (1.0 + e);
}

typedef void (*task_fn)(void* ctx, int64_t task, double* scratch);

typedef struct {
  task_fn fn;
  void* ctx;
  int64_t ntasks;
  int64_t next; /* shared counter, atomically incremented */
  size_t scratch_doubles;
  int failed;
} pool_t;

static void* pool_worker(void* arg) {
  pool_t* pl = (pool_t*)arg;
  double* scratch = (double*)malloc(pl->scratch_doubles * sizeof(double) + 64);
  if (!scratch) {
    __atomic_store_n(&pl->failed, 1, __ATOMIC_SEQ_CST);
    return NULL;
  }
  for (;;) {
    int64_t t = __atomic_fetch_add(&pl->next, 1, __ATOMIC_SEQ_CST);
    if (t >= pl->ntasks) break;
    pl->fn(pl->ctx, t, scratch);
  }
  free(scratch);
  return NULL;
}

/* Run fn(ctx, task, scratch) for task in [0, ntasks) on up to nthreads
 * threads; each thread owns one scratch buffer.  Returns 0 on success. */
static int parallel_for(int64_t ntasks, int nthreads, size_t scratch_doubles, task_fn fn, void* ctx) {
  pool_t pl = {fn, ctx, ntasks, 0, scratch_doubles, 0};
  if (nthreads < 1) nthreads = 1;
  if (nthreads > ntasks) nthreads = (int)(ntasks > 0 ? ntasks : 1);
  if (nthreads == 1) {
    pool_worker(&pl);
    return pl.failed ? -1 : 0;
  }
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!th) return -1;
  int started = 0;
  for (int i = 0; i < nthreads; ++i) {
    if (pthread_create(&th[i], NULL, pool_worker, &pl) != 0) break;
    ++started;
  }
  if (started == 0) { free(th); pool_worker(&pl); return pl.failed ? -1 : 0; }
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  return pl.failed ? -1 : 0;
}

/* Heads (or channels) of one group are handled in fixed blocks of this many
 * consecutive heads; each block owns one partial sum for dB/dC, and the
 * blocks are then added in ascending order.  The result is therefore
 * independent of the thread count. */
#define HEAD_BLOCK 4
#define CHAN_BLOCK 16

/* =========================================================== Mamba-2 branch
 * Layouts (row-major): x, y [b,T,H,P]; dt_raw [b,T,H]; A [H]; B, C [b,T,G,N];
 * s0, s_final [b,H,P,N].  Head h reads group g = h / (H/G).                */

typedef struct {
  int64_t b, T, H, P, N, G;
  const double *x, *dt_raw, *A, *B, *C, *s0, *dy, *ds_final;
  double *y, *s_final;
  double *dx, *ddt_raw, *ds0;
  double *dB_part, *dC_part; /* [b][G][nblk][T][N] */
  double *dA_part;           /* [b][H] */
  int64_t nblk;
  int mutation;
} m2_ctx;

static void m2_forward_task(void* vctx, int64_t task, double* s) {
  const m2_ctx* c = (const m2_ctx*)vctx;
  const int64_t T = c->T, H = c->H, P = c->P, N = c->N, G = c->G;
  const int64_t b = task / H, h = task % H, g = h / (H / G);
  const double A = c->A[h];
  if (c->s0) memcpy(s, c->s0 + (b * H + h) * P * N, sizeof(double) * P * N);
  else memset(s, 0, sizeof(double) * P * N);
  for (int64_t t = 0; t < T; ++t) {
    const double d = softplus(c->dt_raw[(b * T + t) * H + h]);
    const double a = exp(d * A);
    const double* xt = c->x + ((b * T + t) * H + h) * P;
    const double* Bt = c->B + ((b * T + t) * G + g) * N;
    const double* Ct = c->C + ((b * T + t) * G + g) * N;
    double* yt = c->y + ((b * T + t) * H + h) * P;
    for (int64_t p = 0; p < P; ++p) {
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n) {
        double v = a * s[p * N + n] + d * xt[p] * Bt[n];
        s[p * N + n] = v;
        acc += v * Ct[n];
      }
      yt[p] = acc;
    }
  }
  memcpy(c->s_final + (b * H + h) * P * N, s, sizeof(double) * P * N);
}

/* One block of consecutive heads of group g in batch b; scratch holds the
 * (T+1) stored states, the running state gradient and one P-vector. */
static void m2_backward_task(void* vctx, int64_t task, double* scratch) {
  const m2_ctx* c = (const m2_ctx*)vctx;
  const int64_t T = c->T, H = c->H, P = c->P, N = c->N, G = c->G;
  const int64_t Hg = H / G, nblk = c->nblk;
  const int64_t b = task / (G * nblk), g = (task / nblk) % G, k = task % nblk;
  const int mut = c->mutation;
  double* S = scratch;                 /* [(T+1)][P][N] */
  double* dS = S + (T + 1) * P * N;    /* [P][N] */
  double* u = dS + P * N;              /* [P] */
  double* acc_n = u + P;               /* [N] */
  double* dBp = c->dB_part + ((b * G + g) * nblk + k) * T * N;
  double* dCp = c->dC_part + ((b * G + g) * nblk + k) * T * N;
  memset(dBp, 0, sizeof(double) * T * N);
  memset(dCp, 0, sizeof(double) * T * N);

  for (int64_t hh = k * HEAD_BLOCK; hh < (k + 1) * HEAD_BLOCK && hh < Hg; ++hh) {
    const int64_t h = g * Hg + hh;
    const double A = c->A[h];
    /* replay the forward, keeping every state: S[t+1] = s_t, S[0] = s0 */
    if (c->s0) memcpy(S, c->s0 + (b * H + h) * P * N, sizeof(double) * P * N);
    else memset(S, 0, sizeof(double) * P * N);
    for (int64_t t = 0; t < T; ++t) {
      const double d = softplus(c->dt_raw[(b * T + t) * H + h]);
      const double a = exp(d * A);
      const double* xt = c->x + ((b * T + t) * H + h) * P;
      const double* Bt = c->B + ((b * T + t) * G + g) * N;
      const double* Sp = S + t * P * N;
      double* Sn = S + (t + 1) * P * N;
      for (int64_t p = 0; p < P; ++p)
        for (int64_t n = 0; n < N; ++n) Sn[p * N + n] = a * Sp[p * N + n] + d * xt[p] * Bt[n];
    }
    /* seed with the upstream gradient of the final state */
    if (mut == 2) memset(dS, 0, sizeof(double) * P * N);
    else memcpy(dS, c->ds_final + (b * H + h) * P * N, sizeof(double) * P * N);
    double dA_acc = 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
      const double z = c->dt_raw[(b * T + t) * H + h];
      const double d = softplus(z);
      const double a = exp(d * A);
      const double* xt = c->x + ((b * T + t) * H + h) * P;
      const double* Bt = c->B + ((b * T + t) * G + g) * N;
      const double* Ct = c->C + ((b * T + t) * G + g) * N;
      const double* dyt = c->dy + ((b * T + t) * H + h) * P;
      const double* s_prev = S + t * P * N;       /* s_{t-1} */
      const double* s_cur = S + (t + 1) * P * N;  /* s_t */
      /* y_t = s_t . C_t : y's contribution to the state gradient */
      if (mut != 3)
        for (int64_t p = 0; p < P; ++p)
          for (int64_t n = 0; n < N; ++n) dS[p * N + n] += dyt[p] * Ct[n];
      /* dC_t = sum_p dy_t[p] s_t[p, :] */
      const double* s_for_dC = (mut == 4) ? s_prev : s_cur;
      for (int64_t n = 0; n < N; ++n) acc_n[n] = 0.0;
      for (int64_t p = 0; p < P; ++p)       /* per n, p ascending */
        for (int64_t n = 0; n < N; ++n) acc_n[n] += dyt[p] * s_for_dC[p * N + n];
      for (int64_t n = 0; n < N; ++n) dCp[t * N + n] += acc_n[n];
      /* s_t = a s_{t-1} + d x_t (outer) B_t */
      double dd = 0.0; /* d J / d dt' */
      for (int64_t p = 0; p < P; ++p) {
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) acc += dS[p * N + n] * Bt[n];
        u[p] = acc;
        c->dx[((b * T + t) * H + h) * P + p] = d * acc;
        dd += acc * xt[p];
      }
      for (int64_t n = 0; n < N; ++n) acc_n[n] = 0.0;
      for (int64_t p = 0; p < P; ++p)
        for (int64_t n = 0; n < N; ++n) acc_n[n] += dS[p * N + n] * xt[p];
      for (int64_t n = 0; n < N; ++n) dBp[t * N + n] += d * acc_n[n];
      /* the decay path: a = exp(d A), d a / d(dA) = a */
      double dda = 0.0;
      for (int64_t i = 0; i < P * N; ++i) dda += dS[i] * s_prev[i];
      dda *= a;
      if (mut != 1) dd += A * dda;
      dA_acc += d * dda;
      c->ddt_raw[(b * T + t) * H + h] = (mut == 5) ? dd : dd * sigmoid(z);
      for (int64_t i = 0; i < P * N; ++i) dS[i] *= a;
    }
    memcpy(c->ds0 + (b * H + h) * P * N, dS, sizeof(double) * P * N);
    c->dA_part[b * H + h] = dA_acc;
  }
}

int oracle_m2_forward(int64_t b, int64_t T, int64_t H, int64_t P, int64_t N, int64_t G,
                      const double* x, const double* dt_raw, const double* A, const double* B,
                      const double* C, const double* s0, double* y, double* s_final, int nthreads) {
  if (b < 0 || T < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G) return -1;
  m2_ctx c;
  memset(&c, 0, sizeof c);
  c.b = b; c.T = T; c.H = H; c.P = P; c.N = N; c.G = G;
  c.x = x; c.dt_raw = dt_raw; c.A = A; c.B = B; c.C = C; c.s0 = s0;
  c.y = y; c.s_final = s_final;
  return parallel_for(b * H, nthreads, (size_t)(P * N), m2_forward_task, &c);
}

int oracle_m2_backward(int64_t b, int64_t T, int64_t H, int64_t P, int64_t N, int64_t G,
                       const double* x, const double* dt_raw, const double* A, const double* B,
                       const double* C, const double* s0, const double* dy, const double* ds_final,
                       double* dx, double* ddt_raw, double* dA, double* dB, double* dC, double* ds0,
                       int nthreads, int mutation) {
  if (b < 0 || T < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G) return -1;
  m2_ctx c;
  memset(&c, 0, sizeof c);
  c.b = b; c.T = T; c.H = H; c.P = P; c.N = N; c.G = G;
  c.x = x; c.dt_raw = dt_raw; c.A = A; c.B = B; c.C = C; c.s0 = s0;
  c.dy = dy; c.ds_final = ds_final;
  c.dx = dx; c.ddt_raw = ddt_raw; c.ds0 = ds0;
  c.mutation = mutation;
  const int64_t Hg = H / G;
  c.nblk = (Hg + HEAD_BLOCK - 1) / HEAD_BLOCK;
  c.dB_part = (double*)malloc(sizeof(double) * (size_t)(b * G * c.nblk * T * N) + 8);
  c.dC_part = (double*)malloc(sizeof(double) * (size_t)(b * G * c.nblk * T * N) + 8);
  c.dA_part = (double*)malloc(sizeof(double) * (size_t)(b * H) + 8);
  int rc = -1;
  if (c.dB_part && c.dC_part && c.dA_part) {
    rc = parallel_for(b * G * c.nblk, nthreads, (size_t)((T + 2) * P * N + P + N), m2_backward_task, &c);
    if (rc == 0) {
      /* fixed-order reductions: head blocks ascending, then batches ascending */
      for (int64_t bb = 0; bb < b; ++bb)
        for (int64_t t = 0; t < T; ++t)
          for (int64_t g = 0; g < G; ++g)
            for (int64_t n = 0; n < N; ++n) {
              double sb = 0.0, sc = 0.0;
              for (int64_t k = 0; k < c.nblk; ++k) {
                sb += c.dB_part[((bb * G + g) * c.nblk + k) * T * N + t * N + n];
                sc += c.dC_part[((bb * G + g) * c.nblk + k) * T * N + t * N + n];
              }
              dB[((bb * T + t) * G + g) * N + n] = sb;
              dC[((bb * T + t) * G + g) * N + n] = sc;
            }
      for (int64_t h = 0; h < H; ++h) {
        double acc = 0.0;
        for (int64_t bb = 0; bb < b; ++bb) acc += c.dA_part[bb * H + h];
        dA[h] = acc;
      }
    }
  }
  free(c.dB_part);
  free(c.dC_part);
  free(c.dA_part);
  return rc;
}

/* =========================================================== Mamba-1 branch
 * One decay per state.  Layouts: x, y, dt_raw [b,T,D]; A [D,N]; B, C [b,T,N];
 * s0, s_final [b,D,N].  Every channel reads the same B_t, C_t.              */

typedef struct {
  int64_t b, T, D, N;
  const double *x, *dt_raw, *A, *B, *C, *s0, *dy, *ds_final;
  double *y, *s_final;
  double *dx, *ddt_raw, *ds0;
  double *dB_part, *dC_part; /* [b][nblk][T][N] */
  double *dA_part;           /* [b][D][N] */
  int64_t nblk;
  int mutation;
} m1_ctx;

static void m1_forward_task(void* vctx, int64_t task, double* s) {
  const m1_ctx* c = (const m1_ctx*)vctx;
  const int64_t T = c->T, D = c->D, N = c->N;
  const int64_t b = task / D, dch = task % D;
  const double* A = c->A + dch * N;
  if (c->s0) memcpy(s, c->s0 + (b * D + dch) * N, sizeof(double) * N);
  else memset(s, 0, sizeof(double) * N);
  for (int64_t t = 0; t < T; ++t) {
    const double d = softplus(c->dt_raw[(b * T + t) * D + dch]);
    const double xt = c->x[(b * T + t) * D + dch];
    const double* Bt = c->B + (b * T + t) * N;
    const double* Ct = c->C + (b * T + t) * N;
    double acc = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      s[n] = exp(d * A[n]) * s[n] + d * xt * Bt[n];
      acc += s[n] * Ct[n];
    }
    c->y[(b * T + t) * D + dch] = acc;
  }
  memcpy(c->s_final + (b * D + dch) * N, s, sizeof(double) * N);
}

static void m1_backward_task(void* vctx, int64_t task, double* scratch) {
  const m1_ctx* c = (const m1_ctx*)vctx;
  const int64_t T = c->T, D = c->D, N = c->N, nblk = c->nblk;
  const int64_t b = task / nblk, k = task % nblk;
  const int mut = c->mutation;
  double* S = scratch;              /* [(T+1)][N] */
  double* dS = S + (T + 1) * N;     /* [N] */
  double* dBp = c->dB_part + (b * nblk + k) * T * N;
  double* dCp = c->dC_part + (b * nblk + k) * T * N;
  memset(dBp, 0, sizeof(double) * T * N);
  memset(dCp, 0, sizeof(double) * T * N);
  for (int64_t dch = k * CHAN_BLOCK; dch < (k + 1) * CHAN_BLOCK && dch < D; ++dch) {
    const double* A = c->A + dch * N;
    double* dA = c->dA_part + (b * D + dch) * N;
    if (c->s0) memcpy(S, c->s0 + (b * D + dch) * N, sizeof(double) * N);
    else memset(S, 0, sizeof(double) * N);
    for (int64_t t = 0; t < T; ++t) {
      const double d = softplus(c->dt_raw[(b * T + t) * D + dch]);
      const double xt = c->x[(b * T + t) * D + dch];
      const double* Bt = c->B + (b * T + t) * N;
      for (int64_t n = 0; n < N; ++n) S[(t + 1) * N + n] = exp(d * A[n]) * S[t * N + n] + d * xt * Bt[n];
    }
    if (mut == 2) memset(dS, 0, sizeof(double) * N);
    else memcpy(dS, c->ds_final + (b * D + dch) * N, sizeof(double) * N);
    for (int64_t n = 0; n < N; ++n) dA[n] = 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
      const double z = c->dt_raw[(b * T + t) * D + dch];
      const double d = softplus(z);
      const double xt = c->x[(b * T + t) * D + dch];
      const double dyt = c->dy[(b * T + t) * D + dch];
      const double* Bt = c->B + (b * T + t) * N;
      const double* Ct = c->C + (b * T + t) * N;
      const double* s_prev = S + t * N;
      const double* s_cur = S + (t + 1) * N;
      const double* s_for_dC = (mut == 4) ? s_prev : s_cur;
      if (mut != 3)
        for (int64_t n = 0; n < N; ++n) dS[n] += dyt * Ct[n];
      for (int64_t n = 0; n < N; ++n) dCp[t * N + n] += dyt * s_for_dC[n];
      double u = 0.0;
      for (int64_t n = 0; n < N; ++n) u += dS[n] * Bt[n];
      c->dx[(b * T + t) * D + dch] = d * u;
      double dd = u * xt;
      for (int64_t n = 0; n < N; ++n) dBp[t * N + n] += d * xt * dS[n];
      for (int64_t n = 0; n < N; ++n) {
        const double a = exp(d * A[n]);
        const double dda = a * dS[n] * s_prev[n];
        if (mut != 1) dd += A[n] * dda;
        dA[n] += d * dda;
        dS[n] *= a;
      }
      c->ddt_raw[(b * T + t) * D + dch] = (mut == 5) ? dd : dd * sigmoid(z);
    }
    memcpy(c->ds0 + (b * D + dch) * N, dS, sizeof(double) * N);
  }
}

int oracle_m1_forward(int64_t b, int64_t T, int64_t D, int64_t N, const double* x, const double* dt_raw,
                      const double* A, const double* B, const double* C, const double* s0, double* y,
                      double* s_final, int nthreads) {
  if (b < 0 || T < 0 || D <= 0 || N <= 0) return -1;
  m1_ctx c;
  memset(&c, 0, sizeof c);
  c.b = b; c.T = T; c.D = D; c.N = N;
  c.x = x; c.dt_raw = dt_raw; c.A = A; c.B = B; c.C = C; c.s0 = s0;
  c.y = y; c.s_final = s_final;
  return parallel_for(b * D, nthreads, (size_t)N, m1_forward_task, &c);
}

int oracle_m1_backward(int64_t b, int64_t T, int64_t D, int64_t N, const double* x, const double* dt_raw,
                       const double* A, const double* B, const double* C, const double* s0, const double* dy,
                       const double* ds_final, double* dx, double* ddt_raw, double* dA, double* dB, double* dC,
                       double* ds0, int nthreads, int mutation) {
  if (b < 0 || T < 0 || D <= 0 || N <= 0) return -1;
  m1_ctx c;
  memset(&c, 0, sizeof c);
  c.b = b; c.T = T; c.D = D; c.N = N;
  c.x = x; c.dt_raw = dt_raw; c.A = A; c.B = B; c.C = C; c.s0 = s0;
  c.dy = dy; c.ds_final = ds_final;
  c.dx = dx; c.ddt_raw = ddt_raw; c.ds0 = ds0;
  c.mutation = mutation;
  c.nblk = (D + CHAN_BLOCK - 1) / CHAN_BLOCK;
  c.dB_part = (double*)malloc(sizeof(double) * (size_t)(b * c.nblk * T * N) + 8);
  c.dC_part = (double*)malloc(sizeof(double) * (size_t)(b * c.nblk * T * N) + 8);
  c.dA_part = (double*)malloc(sizeof(double) * (size_t)(b * D * N) + 8);
  int rc = -1;
  if (c.dB_part && c.dC_part && c.dA_part) {
    rc = parallel_for(b * c.nblk, nthreads, (size_t)((T + 2) * N), m1_backward_task, &c);
    if (rc == 0) {
      for (int64_t bb = 0; bb < b; ++bb)
        for (int64_t t = 0; t < T; ++t)
          for (int64_t n = 0; n < N; ++n) {
            double sb = 0.0, sc = 0.0;
            for (int64_t k = 0; k < c.nblk; ++k) {
              sb += c.dB_part[(bb * c.nblk + k) * T * N + t * N + n];
              sc += c.dC_part[(bb * c.nblk + k) * T * N + t * N + n];
            }
            dB[(bb * T + t) * N + n] = sb;
            dC[(bb * T + t) * N + n] = sc;
          }
      for (int64_t i = 0; i < D * N; ++i) {
        double acc = 0.0;
        for (int64_t bb = 0; bb < b; ++bb) acc += c.dA_part[bb * D * N + i];
        dA[i] = acc;
      }
    }
  }
  free(c.dB_part);
  free(c.dC_part);
  free(c.dA_part);
  return rc;
}

/* ============================================================== MIMO rank R
 * Layouts: v, y [b,T,R,H,P]; da [b,T,H]; B, C [b,T,R,H,N]; s0, s_final
 * [b,H,P,N].  B and C are per head, so nothing is reduced across heads.    */

typedef struct {
  int64_t b, T, R, H, P, N;
  const double *v, *da, *B, *C, *s0, *dy, *ds_final;
  double *y, *s_final;
  double *dv, *dda, *dB, *dC, *ds0;
  int mutation;
} mimo_ctx;

#define MIMO_IDX(b, t, r, h, k, K) (((((b) * T + (t)) * R + (r)) * H + (h)) * (K) + (k))

static void mimo_forward_task(void* vctx, int64_t task, double* s) {
  const mimo_ctx* c = (const mimo_ctx*)vctx;
  const int64_t T = c->T, R = c->R, H = c->H, P = c->P, N = c->N;
  const int64_t b = task / H, h = task % H;
  if (c->s0) memcpy(s, c->s0 + (b * H + h) * P * N, sizeof(double) * P * N);
  else memset(s, 0, sizeof(double) * P * N);
  for (int64_t t = 0; t < T; ++t) {
    const double a = exp(c->da[(b * T + t) * H + h]);
    for (int64_t i = 0; i < P * N; ++i) s[i] *= a;
    for (int64_t r = 0; r < R; ++r) {
      const double* vt = c->v + MIMO_IDX(b, t, r, h, 0, P);
      const double* Bt = c->B + MIMO_IDX(b, t, r, h, 0, N);
      for (int64_t p = 0; p < P; ++p)
        for (int64_t n = 0; n < N; ++n) s[p * N + n] += vt[p] * Bt[n];
    }
    for (int64_t r = 0; r < R; ++r) {
      const double* Ct = c->C + MIMO_IDX(b, t, r, h, 0, N);
      double* yt = c->y + MIMO_IDX(b, t, r, h, 0, P);
      for (int64_t p = 0; p < P; ++p) {
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) acc += s[p * N + n] * Ct[n];
        yt[p] = acc;
      }
    }
  }
  memcpy(c->s_final + (b * H + h) * P * N, s, sizeof(double) * P * N);
}

static void mimo_backward_task(void* vctx, int64_t task, double* scratch) {
  const mimo_ctx* c = (const mimo_ctx*)vctx;
  const int64_t T = c->T, R = c->R, H = c->H, P = c->P, N = c->N;
  const int64_t b = task / H, h = task % H;
  const int mut = c->mutation;
  double* S = scratch;
  double* dS = S + (T + 1) * P * N;
  if (c->s0) memcpy(S, c->s0 + (b * H + h) * P * N, sizeof(double) * P * N);
  else memset(S, 0, sizeof(double) * P * N);
  for (int64_t t = 0; t < T; ++t) {
    const double a = exp(c->da[(b * T + t) * H + h]);
    const double* Sp = S + t * P * N;
    double* Sn = S + (t + 1) * P * N;
    for (int64_t i = 0; i < P * N; ++i) Sn[i] = a * Sp[i];
    for (int64_t r = 0; r < R; ++r) {
      const double* vt = c->v + MIMO_IDX(b, t, r, h, 0, P);
      const double* Bt = c->B + MIMO_IDX(b, t, r, h, 0, N);
      for (int64_t p = 0; p < P; ++p)
        for (int64_t n = 0; n < N; ++n) Sn[p * N + n] += vt[p] * Bt[n];
    }
  }
  if (mut == 2) memset(dS, 0, sizeof(double) * P * N);
  else memcpy(dS, c->ds_final + (b * H + h) * P * N, sizeof(double) * P * N);
  for (int64_t t = T - 1; t >= 0; --t) {
    const double a = exp(c->da[(b * T + t) * H + h]);
    const double* s_prev = S + t * P * N;
    const double* s_cur = S + (t + 1) * P * N;
    const double* s_for_dC = (mut == 4) ? s_prev : s_cur;
    /* every y_{t,r} reads s_t */
    for (int64_t r = 0; r < R; ++r) {
      const double* dyt = c->dy + MIMO_IDX(b, t, r, h, 0, P);
      const double* Ct = c->C + MIMO_IDX(b, t, r, h, 0, N);
      double* dCt = c->dC + MIMO_IDX(b, t, r, h, 0, N);
      if (mut != 3)
        for (int64_t p = 0; p < P; ++p)
          for (int64_t n = 0; n < N; ++n) dS[p * N + n] += dyt[p] * Ct[n];
      for (int64_t n = 0; n < N; ++n) dCt[n] = 0.0;
      for (int64_t p = 0; p < P; ++p)       /* per n, p ascending */
        for (int64_t n = 0; n < N; ++n) dCt[n] += dyt[p] * s_for_dC[p * N + n];
    }
    /* s_t = a s_{t-1} + sum_r v_r (outer) B_r */
    for (int64_t r = 0; r < R; ++r) {
      const double* vt = c->v + MIMO_IDX(b, t, r, h, 0, P);
      const double* Bt = c->B + MIMO_IDX(b, t, r, h, 0, N);
      double* dvt = c->dv + MIMO_IDX(b, t, r, h, 0, P);
      double* dBt = c->dB + MIMO_IDX(b, t, r, h, 0, N);
      for (int64_t p = 0; p < P; ++p) {
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) acc += dS[p * N + n] * Bt[n];
        dvt[p] = acc;
      }
      for (int64_t n = 0; n < N; ++n) dBt[n] = 0.0;
      for (int64_t p = 0; p < P; ++p)
        for (int64_t n = 0; n < N; ++n) dBt[n] += dS[p * N + n] * vt[p];
    }
    double dda = 0.0;
    for (int64_t i = 0; i < P * N; ++i) dda += dS[i] * s_prev[i];
    c->dda[(b * T + t) * H + h] = (mut == 1) ? 0.0 : a * dda;
    for (int64_t i = 0; i < P * N; ++i) dS[i] *= a;
  }
  memcpy(c->ds0 + (b * H + h) * P * N, dS, sizeof(double) * P * N);
}

int oracle_mimo_forward(int64_t b, int64_t T, int64_t R, int64_t H, int64_t P, int64_t N, const double* v,
                        const double* da, const double* B, const double* C, const double* s0, double* y,
                        double* s_final, int nthreads) {
  if (b < 0 || T < 0 || R <= 0 || H <= 0 || P <= 0 || N <= 0) return -1;
  mimo_ctx c;
  memset(&c, 0, sizeof c);
  c.b = b; c.T = T; c.R = R; c.H = H; c.P = P; c.N = N;
  c.v = v; c.da = da; c.B = B; c.C = C; c.s0 = s0; c.y = y; c.s_final = s_final;
  return parallel_for(b * H, nthreads, (size_t)(P * N), mimo_forward_task, &c);
}

int oracle_mimo_backward(int64_t b, int64_t T, int64_t R, int64_t H, int64_t P, int64_t N, const double* v,
                         const double* da, const double* B, const double* C, const double* s0, const double* dy,
                         const double* ds_final, double* dv, double* dda, double* dB, double* dC, double* ds0,
                         int nthreads, int mutation) {
  if (b < 0 || T < 0 || R <= 0 || H <= 0 || P <= 0 || N <= 0) return -1;
  mimo_ctx c;
  memset(&c, 0, sizeof c);
  c.b = b; c.T = T; c.R = R; c.H = H; c.P = P; c.N = N;
  c.v = v; c.da = da; c.B = B; c.C = C; c.s0 = s0; c.dy = dy; c.ds_final = ds_final;
  c.dv = dv; c.dda = dda; c.dB = dB; c.dC = dC; c.ds0 = ds0;
  c.mutation = mutation;
  return parallel_for(b * H, nthreads, (size_t)((T + 2) * P * N), mimo_backward_task, &c);
}
