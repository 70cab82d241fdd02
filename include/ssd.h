/*
 * ssd.h — C ABI of the GB300 (sm_103a) selective state-space scan library.
 *
 * The library computes one selective state-space scan and its vector-Jacobian
 * product (VJP) on the GPU, for three forms of the recurrence:
 *
 *   Mamba-2 (SSD_MAMBA2), one scalar decay per head, B and C shared by the
 *   heads of a group:
 *       dt'_t = softplus(dt_raw_t)
 *       s_t   = exp(dt'_t * A_h) * s_{t-1} + dt'_t * x_t (outer) B_t
 *       y_t   = s_t . C_t                     (the updated state s_t)
 *   Mamba-1 (SSD_MAMBA1), one decay per state:
 *       s_t[n] = exp(dt'_t * A[d,n]) * s_{t-1}[n] + dt'_t * x_t * B_t[n]
 *       y_t    = sum_n s_t[n] * C_t[n]
 *   MIMO rank R (SSD_MIMO), the form of one pass of the Mamba-3 scan:
 *       s_t     = exp(da_t) * s_{t-1} + sum_r v_{t,r} (outer) B_{t,r}
 *       y_{t,r} = s_t . C_{t,r}
 *
 * Sources (the pages the method is taken from):
 *   - "S1-31: SSM_SCAN_BACK — Mamba has a backward" (llama.cpp PR text),
 *     opening paragraph: the reverse recurrence, the Mamba-2 and Mamba-1
 *     branches and the five gradients; "Two things that are easy to get
 *     wrong", item 1: the final-state gradient is a nonzero seed; item 2:
 *     the backward needs s_{t-1} and recomputes the states; verification
 *     table: the softplus derivative belongs in d(dt_raw).
 *   - burn-mamba "combined_backward.rs" (Mamba-3 double-SSD, serial
 *     recalculated): CombinedGrads (one gradient per input, including the
 *     initial state), the chunkwise K1..K5 forward and the recompute backward
 *     (replay K1..K4 from the saved leaf inputs, reverse per-chunk loop
 *     fusing the K5 and K4 backwards, then batched K3/K2/K1 backwards).
 *
 * Conventions for every call:
 *   - All tensor arguments are DEVICE pointers to contiguous row-major
 *     arrays owned by the caller.  The library allocates nothing: scratch
 *     memory is the caller's workspace, sized by ssd_workspace_size().
 *   - Work is enqueued asynchronously on `cuda_stream` (a cudaStream_t; NULL
 *     is the legacy default stream).  A call returns once its kernels are
 *     enqueued.  Buffers must stay valid until the stream reaches them.
 *   - Arguments are validated before anything is launched; on any error no
 *     kernel runs and no output is written.
 *   - Results are bitwise reproducible: the same inputs on the same GPU give
 *     the same bits on every call (all reductions run in a fixed order; no
 *     floating-point atomics).
 *   - Calls on different streams with different buffers (including different
 *     workspaces) may run concurrently.  A workspace must not be shared by
 *     calls that may overlap on the GPU.
 */
#ifndef SSD_GB300_H
#define SSD_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1, /* NULL where a buffer is required, unknown enum, negative size */
  SSD_ERR_SHAPE = 2,       /* sizes the method does not allow (H % G, limits of this build) */
  SSD_ERR_DTYPE = 3,       /* io dtype not supported for this variant */
  SSD_ERR_ALIGNMENT = 4,   /* a pointer is not 16-byte aligned */
  SSD_ERR_WORKSPACE = 5,   /* ws_bytes smaller than ssd_workspace_size() */
  SSD_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed */
  SSD_ERR_TIMEOUT = 7,     /* the device status word is nonzero: a bounded device-side wait gave up */
  SSD_ERR_INTERNAL = 8,    /* a device-side consistency check failed */
  SSD_ERR_TOO_LARGE = 9    /* ssd_forward_static: the problem needs more scratch than its fixed array */
} ssd_status;

typedef enum { SSD_MAMBA2 = 0, SSD_MAMBA1 = 1, SSD_MIMO = 2 } ssd_variant;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

/*
 * Problem description.
 *   variant    ssd_variant.
 *   io_dtype   ssd_dtype of x, B, C, y, dy, dx, dB, dC (and of v, dv for
 *              MIMO).  dt_raw, A, s0, s_final, ds_final, ds0, ddt_raw, dA are
 *              always fp32.  Mamba-1 supports SSD_F32 only.
 *   batch      b >= 1 independent sequences.
 *   seqlen     T >= 1 steps.
 *   nheads     H heads (Mamba-2, MIMO) or D channels (Mamba-1).
 *   headdim    P (Mamba-2, MIMO); must be 1 for Mamba-1.
 *   dstate     N state size.
 *   ngroups    G groups of consecutive heads sharing B and C (Mamba-2;
 *              H % G == 0, head h reads group h / (H/G)).  Ignored for
 *              Mamba-1 (B, C are shared by all channels) and MIMO (B, C are
 *              per head).
 *   chunk      L, the chunk length of the chunkwise algorithm (Mamba-2,
 *              MIMO), 1 <= L <= 256.  Mamba-1 has no chunkwise form: its
 *              kernels walk the sequence step by step (checkpointing the
 *              state every 8 steps in the backward) and accept any
 *              1 <= L <= 256 here.  T need not be a multiple of L: the sequence is cut
 *              into nc = ceil(T / L) chunks, and the last one holds the
 *              remaining T - (nc - 1) L steps (a tail chunk).  The kernels
 *              treat its missing steps as steps with dt' = 0 (da = 0) and
 *              x = B = C = dy = 0, which leave the state unchanged, and store
 *              nothing for them, so every output equals the serial recurrence
 *              over the T real steps.  The chunked layout of the pages builds T
 *              as nchunks * chunk_len; the tail chunk is this library's
 *              widening, which lets a caller stream a sequence in pieces of
 *              any length through s0 / ds_final.
 *   mimo_rank  R (MIMO); must be 1 for the other variants.
 * Limits of this build: P <= 256, N <= 256, L * R <= 256 (Mamba-2, MIMO);
 * N <= 32, L <= 256 (Mamba-1).  Larger sizes return SSD_ERR_SHAPE.
 */
typedef struct {
  int32_t variant;
  int32_t io_dtype;
  int64_t batch;
  int64_t seqlen;
  int64_t nheads;
  int64_t headdim;
  int64_t dstate;
  int64_t ngroups;
  int64_t chunk;
  int64_t mimo_rank;
} ssd_problem;

/*
 * Bytes of device workspace that ssd_forward (backward == 0) or ssd_backward
 * (backward != 0) needs for `prob`.  Writes *bytes and returns SSD_OK, or
 * returns a validation error and leaves *bytes untouched.  Host-only; touches
 * no device.
 */
ssd_status ssd_workspace_size(const ssd_problem* prob, int backward, size_t* bytes);

/*
 * Forward scan: y and s_final from (x, dt_raw, A, B, C, s0).
 *
 * Layouts (row-major):
 *   Mamba-2: x, y [b,T,H,P]; dt_raw [b,T,H]; A [H]; B, C [b,T,G,N];
 *            s0, s_final [b,H,P,N].
 *   Mamba-1: x, y, dt_raw [b,T,D]; A [D,N]; B, C [b,T,N]; s0, s_final [b,D,N].
 *   MIMO:    the x slot carries v [b,T,R,H,P]; the dt_raw slot carries the
 *            pre-combined decay exponent da [b,T,H] (no softplus is applied);
 *            A must be NULL; B, C [b,T,R,H,N]; y [b,T,R,H,P];
 *            s0, s_final [b,H,P,N].
 * s0 may be NULL (a zero initial state).  Every other pointer is required
 * (except A for MIMO) and must be 16-byte aligned.
 * ws / ws_bytes: caller-owned device workspace of at least
 * ssd_workspace_size(prob, 0) bytes (always >= 256, never NULL).  Its first
 * 4 bytes are a device status word (int32): the call resets it to 0, and a
 * kernel whose bounded wait on an internal barrier gives up writes a nonzero
 * code there (the outputs are then invalid).  Read it after the stream
 * reaches the call if that check is wanted.
 */
ssd_status ssd_forward(const ssd_problem* prob, const void* x, const float* dt_raw, const float* A,
                       const void* B, const void* C, const float* s0, void* y, float* s_final, void* ws,
                       size_t ws_bytes, void* cuda_stream);

/*
 * Backward (VJP) of ssd_forward.  Inputs: the upstream gradients dy (layout
 * and dtype of y) and ds_final (fp32, layout of s_final; required, it is the
 * nonzero seed of the reverse recurrence), and the saved leaf inputs of the
 * forward (x, dt_raw, A, B, C, s0 exactly as passed to ssd_forward).  No
 * forward intermediate is needed: the backward recomputes the chunk states.
 *
 * Outputs (each takes its primal's layout and dtype):
 *   dx [like x], ddt_raw [like dt_raw, fp32], dA [like A, fp32],
 *   dB [like B], dC [like C], ds0 [like s0, fp32].
 * dB, dC (Mamba-2: over the heads of each group; Mamba-1: over all
 * channels) and dA (over batch and time) are full reductions written once.
 * MIMO: dx returns dv, ddt_raw returns d(da), and dA must be NULL.
 * s0 may be NULL (zero initial state); ds0 is still written.
 * ws / ws_bytes: at least ssd_workspace_size(prob, 1) bytes, with the same
 * device status word in its first 4 bytes as for ssd_forward.
 */
ssd_status ssd_backward(const ssd_problem* prob, const void* dy, const float* ds_final, const void* x,
                        const float* dt_raw, const float* A, const void* B, const void* C, const float* s0,
                        void* dx, float* ddt_raw, float* dA, void* dB, void* dC, float* ds0, void* ws,
                        size_t ws_bytes, void* cuda_stream);

/*
 * Stashed chunk states: a forward that keeps every chunk-input state S_c for
 * the backward, and a backward that reads them instead of replaying the
 * forward scan (the "Two things that are easy to get wrong" section, item 2,
 * of the "S1-31: SSM_SCAN_BACK" page: the backward needs the states the
 * forward overwrote; storing all of them is the reference, a cheaper scheme
 * must give the same bits).  The stash holds the same bf16 tiles the
 * recompute path writes to its workspace, produced by the same kernel from the
 * same inputs, so ssd_backward_stashed returns bit for bit what ssd_backward
 * returns for the same leaf inputs.  It saves the backward one pass of the
 * state scan (about an eighth of a forward + backward step at the Mamba-2
 * 2.7B layer shape) for b*H*ceil(T/L)*N*P*2 bytes of device memory held from the
 * forward to the backward.
 *
 * Available where the tensor-core path runs: Mamba-2, bf16 io, chunk 64,
 * headdim 64, dstate 128 (other problems return SSD_ERR_SHAPE).
 *
 * ssd_states_size: bytes of the stash for `prob` (bf16 [b, H, ceil(T/L)][N][P],
 *   row-major; tile (b, h, c) is the state entering chunk c, S_0 = s0 rounded
 *   to bf16).  Host-only.
 * ssd_forward_stash: ssd_forward, plus the stash written to `states`
 *   (caller-owned device buffer of at least ssd_states_size bytes, 16-byte
 *   aligned; a smaller states_bytes returns SSD_ERR_WORKSPACE).  y and s_final
 *   are bit for bit those of ssd_forward.  ws as for ssd_forward.
 * ssd_backward_stashed: ssd_backward without s0, reading `states` as written
 *   by ssd_forward_stash for the same x, dt_raw, A, B, s0 (the caller keeps
 *   the buffer unchanged in between; nothing checks it).  ws as for
 *   ssd_backward.
 * Errors and the device status word are those of ssd_forward / ssd_backward.
 */
ssd_status ssd_states_size(const ssd_problem* prob, size_t* bytes);
ssd_status ssd_forward_stash(const ssd_problem* prob, const void* x, const float* dt_raw, const float* A,
                             const void* B, const void* C, const float* s0, void* y, float* s_final, void* states,
                             size_t states_bytes, void* ws, size_t ws_bytes, void* cuda_stream);
ssd_status ssd_backward_stashed(const ssd_problem* prob, const void* dy, const float* ds_final, const void* x,
                                const float* dt_raw, const float* A, const void* B, const void* C,
                                const void* states, size_t states_bytes, void* dx, float* ddt_raw, float* dA,
                                void* dB, void* dC, float* ds0, void* ws, size_t ws_bytes, void* cuda_stream);

/*
 * Checkpoint every K chunks: a forward that keeps the fp32 chain state at
 * every K-th chunk boundary, and a backward that replays the chunk states from
 * those checkpoints in independent segments of K chunks instead of one
 * sequential scan over the whole sequence (the "Two things that are easy to
 * get wrong" section, item 2, of the "S1-31: SSM_SCAN_BACK" page: checkpoints
 * every K steps are the cheaper scheme, and must give the bits of storing every
 * state).  The checkpoints are the exact fp32 states of the forward's scan, and
 * each segment applies the same operations to them as the whole-sequence
 * replay, so ssd_backward_checkpointed returns bit for bit what ssd_backward
 * returns, for any K.  Memory held from the forward to the backward:
 * b*H*ceil(nc/K)*P*N*4 bytes (nc = ceil(T/L); 84 MB at K = 8 for the Mamba-2
 * 2.7B layer shape, against 336 MB for the stash of every state).
 *
 * Available where the tensor-core path runs: Mamba-2, bf16 io, chunk 64,
 * headdim 64, dstate 128 (other problems return SSD_ERR_SHAPE).  every = K,
 * 1 <= K <= 2^30 (SSD_ERR_INVALID_ARG otherwise); K >= nc keeps only s0.
 *
 * ssd_checkpoints_size: bytes of the checkpoints (fp32 [b, H, ceil(nc/K)][P][N],
 *   row-major; entry (b, h, k) is the state entering chunk k*K, entry 0 = s0,
 *   zeros for a NULL s0).  Host-only.
 * ssd_forward_checkpointed: ssd_forward, plus the checkpoints written to
 *   `ckpt` (caller-owned device buffer of at least ssd_checkpoints_size bytes,
 *   16-byte aligned; a smaller ckpt_bytes returns SSD_ERR_WORKSPACE).  y and
 *   s_final are bit for bit those of ssd_forward.  ws as for ssd_forward.
 * ssd_backward_checkpointed: ssd_backward without s0, reading the checkpoints
 *   written by ssd_forward_checkpointed with the same K for the same x,
 *   dt_raw, A, B, s0 (the caller keeps the buffer unchanged in between; nothing
 *   checks it).  ws as for ssd_backward.
 * Errors and the device status word are those of ssd_forward / ssd_backward.
 */
ssd_status ssd_checkpoints_size(const ssd_problem* prob, int64_t every, size_t* bytes);
ssd_status ssd_forward_checkpointed(const ssd_problem* prob, const void* x, const float* dt_raw, const float* A,
                                    const void* B, const void* C, const float* s0, void* y, float* s_final,
                                    int64_t every, float* ckpt, size_t ckpt_bytes, void* ws, size_t ws_bytes,
                                    void* cuda_stream);
ssd_status ssd_backward_checkpointed(const ssd_problem* prob, const void* dy, const float* ds_final, const void* x,
                                     const float* dt_raw, const float* A, const void* B, const void* C,
                                     int64_t every, const float* ckpt, size_t ckpt_bytes, void* dx, float* ddt_raw,
                                     float* dA, void* dB, void* dC, float* ds0, void* ws, size_t ws_bytes,
                                     void* cuda_stream);

/*
 * Forward scan without a caller workspace, for callers that cannot allocate
 * device memory.  (The pages describe no such call; it is an addition of this
 * library.)
 *
 * Who needs it: code that runs where device allocation is not available or
 * not allowed once it has started, for example an inference engine or plugin
 * whose host framework owns all GPU memory and hands out only the tensors, or
 * a latency-critical loop that has a rule of no allocation after start-up.
 * ssd_forward needs a workspace from ssd_workspace_size(); this call takes
 * none.  Its scratch is one fixed array of 32 MiB in device memory, declared
 * at file scope in the library, so every GPU that loads the library keeps
 * those 32 MiB until the process exits.
 *
 * Arguments, layouts, results and validation are those of ssd_forward,
 * without ws / ws_bytes.  A problem whose ssd_workspace_size(prob, 0) exceeds
 * 32 MiB is rejected with SSD_ERR_TOO_LARGE before anything runs.  The call
 * allocates nothing (no cudaMalloc, no allocating library routine).
 *
 * Start-up: the array belongs to this library's device module, which the
 * CUDA runtime loads on a device the first time the library needs it there
 * (lazy loading, the default).  Loading reserves the 32 MiB, so a caller that
 * forbids device allocation after start-up calls
 * ssd_forward_static_status(NULL, stream) once per device at start-up, with
 * that device current and before any stream capture: it loads the module and
 * looks up the array's address and does nothing else.  Later calls allocate
 * nothing.
 *
 * All calls share the one array, which keeps the last call's contents (its
 * first 4 bytes are the device status word, reset to 0 by every call):
 * calls that may overlap on the GPU, on any streams, race on it and must be
 * serialized by the caller.
 *
 * ssd_forward_static_status(code, stream): with code == NULL, the start-up
 * step above only.  Otherwise it also copies the status word into *code (a
 * caller-owned host int32) on `stream`, after the work already enqueued
 * there, and waits for that stream.  Returns SSD_OK when the word is 0,
 * SSD_ERR_TIMEOUT when a bounded wait of the last call gave up (its outputs
 * are then invalid; *code holds the code), SSD_ERR_CUDA if a CUDA call fails.
 */
ssd_status ssd_forward_static(const ssd_problem* prob, const void* x, const float* dt_raw, const float* A,
                              const void* B, const void* C, const float* s0, void* y, float* s_final,
                              void* cuda_stream);
ssd_status ssd_forward_static_status(int32_t* code, void* cuda_stream);

/*
 * The device status word of a workspace, and a test of the bounded waits.
 *
 * Every wait of a kernel of this library on one of its barriers is bounded
 * (two seconds).  One that runs out writes a nonzero code into the status
 * word (the first 4 bytes of the call's workspace), stops issuing work and
 * returns; the host learns of it only from the word, since the call itself
 * returned before the GPU ran it.  (The pages ask for none of this; it is the
 * failure detection of this library.)
 *
 * ssd_read_status(ws, code, stream): copies the status word at the start of
 * the device workspace `ws` into *code (host int32) on `stream`, after the
 * work already enqueued there, and waits for that stream.  Returns SSD_OK for
 * 0, SSD_ERR_TIMEOUT for a nonzero word, SSD_ERR_INVALID_ARG for NULL
 * arguments, SSD_ERR_CUDA if a CUDA call fails.  Allocates nothing.
 *
 * ssd_wait_selftest(ws, limit_us, stream): resets the status word of `ws`
 * (device, 16-byte aligned, at least 4 bytes) and launches one warp in which
 * one thread waits on a barrier that nothing ever completes, with a limit of
 * limit_us microseconds (1 .. 2 000 000) instead of two seconds.  The wait
 * runs out, writes code 1 into the word and the kernel returns: a following
 * ssd_read_status returns SSD_ERR_TIMEOUT with *code == 1, and the stream and
 * context stay usable.  Returns SSD_ERR_INVALID_ARG for a NULL ws or a limit
 * outside the range, SSD_ERR_ALIGNMENT, or SSD_ERR_CUDA if the launch fails.
 */
ssd_status ssd_read_status(const void* ws, int32_t* code, void* cuda_stream);
ssd_status ssd_wait_selftest(void* ws, uint32_t limit_us, void* cuda_stream);

/*
 * KDA: the gated delta-rule recurrence of the notes page "sec-10.tex"
 * (section "反向传播推导"), a second workload beside the selective scan, and
 * its BPTT backward (the page's reverse-time steps 1-6).  fp32 io and
 * arithmetic.  Per batch element and value head, with state S [K, V]:
 *     S_dec = exp(g_t) (.) S_{t-1}     (one log-decay per key row)
 *     r_t   = v_t - k_t^T S_dec
 *     S_t   = S_dec + beta_t k_t (x) r_t
 *     o_t   = (scale q_t)^T S_t
 * Value head hv reads query / key head hv / G, G = value_heads / nheads (the
 * page's grouped value heads); dq, dk of a query / key head are the sums over
 * its G value heads.
 *
 * Layouts (row-major, fp32, 16-byte aligned): q, k, dq, dk [b,T,H,K];
 * v, o, do, dv [b,T,HV,V]; g, dg [b,T,HV,K]; beta, dbeta [b,T,HV];
 * s0, s_final, ds_final, ds0 [b,HV,K,V].  s0 may be NULL (zeros).
 * Limits of this build: key_dim <= 128, value_dim <= 128 (SSD_ERR_SHAPE);
 * value_heads a multiple of nheads (SSD_ERR_SHAPE).
 *
 * ssd_kda_workspace_size: device workspace of the forward (backward == 0) or
 *   backward; host-only.  The backward's holds fp32 checkpoints of the state
 *   every 8 steps (b*HV*ceil(T/8)*K*V*4 bytes), the per-step row sums of its
 *   CTAs and the per-value-head dq, dk.  Its first 4 bytes are the device
 *   status word, as for ssd_forward.
 * ssd_kda_forward: o and s_final.
 * ssd_kda_backward: dq, dk, dv, dg, dbeta and ds0 of <do, o> + <ds_final,
 *   s_final> (ds_final required); recomputes the states from the leaf inputs
 *   (no forward intermediate is needed).  Deterministic: every sum has a
 *   fixed order.
 * Errors as for ssd_forward; every error is returned before anything is
 * enqueued.
 */
typedef struct {
  int64_t batch;
  int64_t seqlen;
  int64_t nheads;      /* H: query / key heads */
  int64_t value_heads; /* HV: a multiple of H */
  int64_t key_dim;     /* K */
  int64_t value_dim;   /* V */
} ssd_kda_problem;

ssd_status ssd_kda_workspace_size(const ssd_kda_problem* prob, int backward, size_t* bytes);
ssd_status ssd_kda_forward(const ssd_kda_problem* prob, const float* q, const float* k, const float* v,
                           const float* g, const float* beta, const float* s0, float scale, float* o, float* s_final,
                           void* ws, size_t ws_bytes, void* cuda_stream);
ssd_status ssd_kda_backward(const ssd_kda_problem* prob, const float* dout, const float* ds_final, const float* q,
                            const float* k, const float* v, const float* g, const float* beta, const float* s0,
                            float scale, float* dq, float* dk, float* dv, float* dg, float* dbeta, float* ds0,
                            void* ws, size_t ws_bytes, void* cuda_stream);

/*
 * Per-launch timing, for diagnostics and roofline measurement.
 *
 * ssd_profile_start(capacity): every later ssd_forward / ssd_backward call
 * (from any host thread) records a pair of CUDA events around each kernel it
 * enqueues, on that call's stream, for up to `capacity` launches.  Returns
 * SSD_ERR_INVALID_ARG if capacity < 1.  Events are created with
 * cudaEventCreate on the current device; no device memory is allocated.
 *
 * ssd_profile_stop(out, capacity, count): waits for the recorded events,
 * writes one {kernel name, milliseconds} record per launch in launch order
 * (at most `capacity`), sets *count to the number written, destroys the
 * events and turns recording off.  The names are static strings.  Returns
 * SSD_ERR_CUDA if an event query fails.
 */
typedef struct {
  const char* kernel;
  float ms;
} ssd_kernel_time;

ssd_status ssd_profile_start(int capacity);
ssd_status ssd_profile_stop(ssd_kernel_time* out, int capacity, int* count);

/* Static, human-readable name of a status code (never NULL). */
const char* ssd_status_string(ssd_status status);

/* Version of this library as MAJOR*10000 + MINOR*100 + PATCH. */
int ssd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSD_GB300_H */
