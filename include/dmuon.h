/*
 * dmuon.h - C ABI of the owner-side batched Muon update on one GB300 GPU.
 *
 * The library runs, for a whole batch of 2-D weight matrices in one pass, the
 * update that a DMuon owner performs on the matrices it owns ("DMuon:
 * Efficient Distributed Muon Training with Near-Adam Overhead", gist.science
 * technical summary, section 2.1 "Owner-Centric Executiestrategie": the owner
 * keeps the optimizer state and runs the Newton-Schulz iteration and the
 * update once per matrix; section 1 "Probleemstelling": Newton-Schulz on the
 * momentum-aggregated gradient, built on the product X X^T). Per matrix W
 * (rows x cols, row-major, rows = dim 0), gradient G and momentum M:
 *
 *   M  <- mu*M + G;   U = G + mu*M (Nesterov) or U = M
 *   X  <- U / (||U||_F + eps), transposed when rows > cols (short side first)
 *   repeat ns_steps:  A = X X^T;  B = b*A + c*A*A;  X <- a*X + B*X
 *   W  <- W - lr * sqrt(max(1, rows/cols)) * X     (X back in W's orientation)
 *
 * The two calls follow the problem statement of the pages: a plan built once
 * from the list of matrix shapes, the Newton-Schulz step count, coefficients
 * and dtypes ("dmuon_plan"), and a step taking params, grads and momenta
 * ("dmuon_step"). Matrices of equal shape are batched into one bucket and
 * every phase runs all buckets in one launch (summary section 2,
 * "Batching"); tiles are ordered by computational cost, largest first, the
 * greedy fallback of the cost-based balancing in summary section 2.3.
 *
 * Conventions for every entry point:
 *  - Every call returns a dmuon_status; nothing else crosses the ABI. On an
 *    error, dmuon_last_error() returns a message (thread-local, valid until
 *    the next call on the same thread).
 *  - Argument errors are detected on the host before anything is launched.
 *  - "stream" is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - Device pointers must address memory of the current CUDA device.
 *  - The library never allocates device memory: the caller owns the
 *    workspace and every parameter, gradient and momentum buffer.
 *  - Device-detected conditions (non-finite norm, a pipeline wait that ran
 *    out of time) are bits of a status word in the workspace, never traps;
 *    read them with dmuon_read_device_status().
 */
#ifndef DMUON_H
#define DMUON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DMUON_OK = 0,
  DMUON_ERR_INVALID_ARG = -1, /* bad shape, count, pointer, size or value      */
  DMUON_ERR_UNSUPPORTED = -2, /* dtype combination or flag not supported       */
  DMUON_ERR_WORKSPACE = -3,   /* workspace NULL, too small or misaligned       */
  DMUON_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed             */
  DMUON_ERR_NOT_BOUND = -5,   /* dmuon_step before dmuon_plan_bind             */
  DMUON_ERR_DEVICE = -6       /* a device-side result is wrong: a status bit is
                                 set, or a DMUON_FLAG_DEBUG_CHECKS check failed */
} dmuon_status;

typedef enum { DMUON_F32 = 0, DMUON_BF16 = 1 } dmuon_dtype;

/* Stored shape of one matrix: rows = dim 0, row-major, contiguous. */
typedef struct {
  int64_t rows;
  int64_t cols;
} dmuon_shape;

/* Storage dtypes of the step's tensors and the arithmetic mode.
 *   param:    DMUON_F32 or DMUON_BF16 (weights, updated in place)
 *   grad:     DMUON_F32 or DMUON_BF16 (read only)
 *   momentum: DMUON_F32 only (updated in place)
 *   compute:  DMUON_F32  = fp32 operands and fp32 accumulation everywhere;
 *             DMUON_BF16 = bf16 Newton-Schulz operands (X, A, B stored bf16)
 *                          with fp32 accumulation on the tensor cores.      */
typedef struct {
  int32_t param;
  int32_t grad;
  int32_t momentum;
  int32_t compute;
} dmuon_dtypes;

/* Plan flags. */
#define DMUON_FLAG_CAPTURE_UPDATE 0x1u /* keep the fp32 update X of the last step
                                          (read it with dmuon_read_update)      */
#define DMUON_FLAG_GRAM_NS 0x2u        /* matrices with max(rows,cols) >= 2*min(rows,cols)
                                          iterate in the m x m Gram space: G = X X^T
                                          once, then per step P = aI + bG + cG^2,
                                          Q <- P Q, G <- P G P; finally X = Q X0
                                          ("DMuon: Efficient Distributed Muon
                                          Training with Near-Adam Overhead",
                                          gist.science summary section 2, "Gram
                                          Space Recurrence"). Fewer flops when the
                                          matrix is wide (>= 26% fewer at 2:1);
                                          others keep the standard form.          */
#define DMUON_FLAG_PAIR_TILES 0x8u    /* 256 x 256 tiles on pairs of SMs (two-SM
                                          UMMA, thread-block clusters of 2; bf16
                                          only) for every bucket whose short side
                                          is a multiple of 256 and whose products
                                          run 256 wide. Without the flag the same
                                          holds for short sides of at least 1024
                                          (the default); other buckets use one-SM
                                          tiles. Test hook: with the environment
                                          variable DMUON_TEST_FORCE_PAIRS=1, every
                                          bucket with a short side >= 256 gets
                                          pairs (as DMUON_FLAG_TUNE may choose).  */
#define DMUON_FLAG_EPILOGUE_AX 0x10u   /* standard form: add the a*X_k term of the
                                          quintic step in the epilogue of the
                                          product B X_k (reading the X_k tile),
                                          with B = bA + cA^2. Without the flag
                                          the step runs as X_{k+1} = P X_k with
                                          P = aI + bA + cA^2 formed by the
                                          symmetric-product epilogue (a on the
                                          diagonal), and the last product reads
                                          no X_k tile: the same polynomial, one
                                          bf16 rounding of a + B_ii instead of
                                          an fp32 a*X term.                      */
#define DMUON_FLAG_STATIC_TILES 0x20u  /* tensor-core launches deal the cost-ordered
                                          tile list round-robin (CTA b, or CTA pair b,
                                          takes tiles b, b + grid, ...) instead of
                                          letting each CTA (pair) claim the next tile
                                          from the launch's counter as it becomes free.
                                          Same results bit for bit; kept to compare the
                                          two schedules.                           */
#define DMUON_FLAG_DEBUG_CHECKS 0x40u /* debugging aid: after every launch of a step
                                          the host waits for it, copies back the
                                          operands of a few sampled output elements
                                          (momentum, U, s, product elements, one on
                                          the diagonal, one mirror, updated weights)
                                          and recomputes them in double precision;
                                          dmuon_step returns DMUON_ERR_DEVICE, with
                                          the launch, matrix and element in
                                          dmuon_last_error(), when one is off by more
                                          than its rounding allows. Makes every step
                                          synchronous and slow; not for capture.
                                          Test hook: with the environment variable
                                          DMUON_TEST_SKIP_LAUNCH=<i>, launch i of
                                          each step is left out, so its outputs are
                                          stale and the checks must report them.  */
#define DMUON_FLAG_ONE_SM_TILES 0x80u /* every bucket uses one-SM tiles (128 rows,
                                          128 or 256 columns): no CTA pairs. Not
                                          together with DMUON_FLAG_PAIR_TILES or
                                          DMUON_FLAG_TUNE.                        */
#define DMUON_FLAG_TUNE 0x4u           /* at bind, time three tile configurations per
                                          bucket on the bound workspace (one-SM
                                          128 x 128 and 128 x 256 tiles, two-SM
                                          256 x 256 pairs where the short side is
                                          >= 256; each with its ring depth), keep
                                          the cheapest, and order tiles by measured
                                          time (see dmuon_plan_costs). Timings are
                                          cached for the process by (short side,
                                          long side, weight dtype, SM count,
                                          compute capability): a later plan with
                                          the same shapes binds without timing.
                                          bf16 only.                              */

/* Device status bits (dmuon_read_device_status). */
#define DMUON_DEV_NONFINITE_NORM 0x1u  /* ||U||_F was NaN or Inf for some matrix  */
#define DMUON_DEV_WAIT_TIMEOUT 0x2u    /* a pipeline wait ran out of time; the
                                          kernel returned early, results invalid */

/* Launch kinds reported by the profiler. */
#define DMUON_KIND_MOMENTUM 0 /* momentum + per-unit sums of squares + cast/transposed copy */
#define DMUON_KIND_GRAM 1     /* A = X X^T, upper tiles, mirrored                  */
#define DMUON_KIND_POLY 2     /* B = b*A + c*A A^T, upper tiles, mirrored          */
#define DMUON_KIND_GEMM 3     /* X' = a*X + B X (last step: W update epilogue)     */
#define DMUON_KIND_UPDATE0 4  /* W update straight from U (ns_steps == 0)          */
#define DMUON_KIND_SYMM 5     /* Gram-space form: product of two commuting
                                 symmetric m x m matrices, upper tiles, mirrored   */
#define DMUON_KIND_NORM 6     /* s = 1/(||U||_F + eps) per matrix from the partials */

typedef struct dmuon_plan_s* dmuon_plan_t;

/*
 * dmuon_plan - validate a batch description and build the host-side plan.
 *
 *  shapes[n_mats]     stored shape of each matrix; 1 <= rows, cols <= 2^20 and
 *                     rows*cols < 2^31.
 *  ns_steps           number of Newton-Schulz steps, 0..16.
 *  coeffs             host array of 3*n_coeff_triples floats (a, b, c, ...);
 *                     n_coeff_triples is 1 (same triple every step) or
 *                     ns_steps (one triple per step). NULL with 0 triples
 *                     selects (3.4445, -4.7750, 2.0315).
 *  eps                added to the Frobenius norm (not its square); >= 0.
 *  dtypes, flags      see above. momentum must be DMUON_F32.
 *  out                receives the plan handle (host memory, owned by the
 *                     library until dmuon_plan_destroy).
 *
 * Needs no GPU: only host memory is touched. Matrices with equal (short, long)
 * shape share a bucket; per phase the tiles of all buckets are listed and
 * sorted by cost (largest first).
 */
dmuon_status dmuon_plan(const dmuon_shape* shapes, int32_t n_mats, int32_t ns_steps,
                        const float* coeffs, int32_t n_coeff_triples, float eps,
                        dmuon_dtypes dtypes, uint32_t flags, dmuon_plan_t* out);

/* Bytes of device workspace the plan needs (host only). */
dmuon_status dmuon_plan_workspace_bytes(dmuon_plan_t plan, size_t* bytes);

/*
 * dmuon_plan_bind - attach a caller-owned device workspace and upload the
 * plan's tables into it (asynchronously, on stream).
 *
 *  d_workspace  device pointer, 1024-byte aligned, at least
 *               dmuon_plan_workspace_bytes() bytes; owned by the caller and
 *               used exclusively by this plan until it is destroyed or bound
 *               again. Its contents need not be initialised.
 *  Builds the TMA tensor maps for the workspace buffers. The plan's host
 *  staging of the tables must outlive the copies: it does (it is owned by the
 *  plan). Returns DMUON_ERR_WORKSPACE if the buffer is NULL, misaligned, too
 *  small or not memory of the current device, DMUON_ERR_UNSUPPORTED for bf16 compute on a GPU other than
 *  sm_103. Any failing bind leaves the plan unbound, also a plan that was
 *  bound before (dmuon_step then returns DMUON_ERR_NOT_BOUND until a bind
 *  succeeds). For tests, the environment variable DMUON_TEST_FAIL set to
 *  bind_check, bind_tables, bind_maps or bind_staging makes the bind fail at
 *  that point (before any CUDA call, after the tables are uploaded, while the
 *  tensor maps are built, or before the host staging is allocated).
 */
dmuon_status dmuon_plan_bind(dmuon_plan_t plan, void* d_workspace, size_t bytes, void* stream);

/*
 * dmuon_step - one Muon step for every matrix of the plan, asynchronous on
 * stream.
 *
 *  params[n_mats]   host array of device pointers; W_i, rows x cols,
 *                   param dtype, updated in place.
 *  grads[n_mats]    host array of device pointers; G_i, grad dtype, read only.
 *  momenta[n_mats]  host array of device pointers; M_i, fp32, updated in place.
 *  lr, mu           learning rate and momentum coefficient (finite).
 *  nesterov         0 = heavy ball (U = M), 1 = Nesterov (U = G + mu*M).
 *
 * Each pointer must be 16-byte aligned and the matrices must not overlap.
 * The host pointer arrays are read during the call only. The plan keeps the
 * last 4 distinct pointer sets resident on the device: a call whose pointers
 * equal one of them copies nothing (alternating gradient buffers cost no
 * copy after their first steps); otherwise the least recently used set is
 * replaced by a cudaMemcpyAsync from host memory on `stream`. With bf16
 * weights on the tensor-core path a resident set also holds a TMA tensor map
 * of every W (encoded on the host when the set is first seen, copied with the
 * pointers): the last Newton-Schulz product stores its updated W boxes
 * through them. Under CUDA-graph
 * capture, make one uncaptured call with the same pointers first so that none
 * is needed; the captured graph stays valid while that pointer set remains
 * one of the 4 resident ones.
 * Launches the momentum kernel and the per-matrix norm kernel, then
 * 3*ns_steps kernels per chunk of standard-form buckets and 4*ns_steps - 1
 * per chunk of Gram-space buckets (a chunk: up to 7 buckets sharing form and
 * tile widths); 2 + 1 kernels when ns_steps == 0. dmuon_plan_describe lists
 * them.
 */
dmuon_status dmuon_step(dmuon_plan_t plan, void* const* params, const void* const* grads,
                        void* const* momenta, float lr, float mu, int32_t nesterov, void* stream);

/*
 * dmuon_set_weight_events - order the weight writes of later steps against
 * work on other streams. Only the launches that write W (the last
 * Newton-Schulz product of each launch chunk, or the update kernel when
 * ns_steps == 0) touch the weights; the momentum pass and every earlier
 * product read only the gradients, the momenta and the workspace.
 *
 *  wait_before_write  a cudaEvent_t (as void*) or NULL: every later
 *                     dmuon_step makes its stream wait on it
 *                     (cudaStreamWaitEvent, on the event's most recent
 *                     record at the time of that dmuon_step call) just
 *                     before its first launch that writes W.
 *  after_write        a cudaEvent_t or NULL: every later dmuon_step
 *                     records it on its stream right after its last launch
 *                     that writes W.
 *
 * With both, a copy of step k's weights (to the host, say) can run on
 * another stream while step k+1's momentum pass and its first ns_steps - 1
 * Newton-Schulz steps run: the copy waits on after_write and records
 * wait_before_write. The events stay the caller's; they must stay valid
 * while set (NULL, NULL clears them). Host only; no effect on the results.
 */
dmuon_status dmuon_set_weight_events(dmuon_plan_t plan, void* wait_before_write, void* after_write);

/*
 * dmuon_read_device_status - synchronise stream, return the device status
 * bits accumulated since the last read (DMUON_DEV_*) in *bits, and clear
 * them. Returns DMUON_OK even when bits are set. The word travels through a
 * one-thread kernel into mapped page-locked host memory owned by the plan,
 * not through a copy, so the read does not wait behind large transfers that
 * other streams have in flight.
 */
dmuon_status dmuon_read_device_status(dmuon_plan_t plan, void* stream, uint32_t* bits);

/*
 * dmuon_read_update - copy the fp32 update X of matrix `mat` from the last
 * step (before lr and the shape scale, in W's rows x cols orientation) to
 * d_dst (device, rows*cols floats), asynchronously on stream. Needs a plan
 * made with DMUON_FLAG_CAPTURE_UPDATE.
 */
dmuon_status dmuon_read_update(dmuon_plan_t plan, int32_t mat, float* d_dst, void* stream);

/*
 * dmuon_plan_describe - JSON text describing the plan (buckets, tiles per
 * phase, launches per step, algorithmic flops and bytes per launch) written
 * to buf (at most len bytes, NUL-terminated); *needed receives the full
 * length + 1. Host only.
 */
dmuon_status dmuon_plan_describe(dmuon_plan_t plan, char* buf, size_t len, size_t* needed);

/*
 * Profiling: dmuon_profile_begin(plan, max_launches) makes the following
 * steps record a CUDA event pair around each launch (on the step's stream),
 * for up to max_launches launches (it creates the events: host-side CUDA
 * objects, no device memory). dmuon_profile_end synchronises the events and
 * writes, for each recorded launch i < cap, its kind (DMUON_KIND_*), its
 * duration in ms and its algorithmic work (flops for GEMM kinds, bytes for
 * streaming kinds); *n receives the number recorded. Profiling then stops.
 */
dmuon_status dmuon_profile_begin(dmuon_plan_t plan, int32_t max_launches);
dmuon_status dmuon_profile_end(dmuon_plan_t plan, int32_t* kinds, float* ms, double* work,
                               int32_t cap, int32_t* n);

/*
 * dmuon_plan_costs - predicted GPU milliseconds of each matrix's
 * Newton-Schulz work (its tiles times the measured time per tile, spread over
 * all SMs), from the timings a DMUON_FLAG_TUNE bind made. n must equal the
 * plan's matrix count; per_matrix_ms is a host array. Returns
 * DMUON_ERR_UNSUPPORTED for a plan that was not tuned. The costs can be
 * passed to dmuon_assign_owners ("DMuon: Efficient Distributed Muon Training
 * with Near-Adam Overhead", gist.science summary section 2.3: owners are
 * balanced on measured, not theoretical, costs).
 */
dmuon_status dmuon_plan_costs(dmuon_plan_t plan, double* per_matrix_ms, int32_t n);

/*
 * Per-CTA timing of the tensor-core launches (profiling). After
 * dmuon_profile_cta_times(plan, 1), every tensor-core launch of the following
 * steps records, per CTA, the global timer (ns) when the CTA started and when
 * it finished, in the workspace (each step overwrites the previous one's);
 * dmuon_profile_cta_times(plan, 0) stops it. dmuon_read_cta_times copies the
 * records of launch `launch` (its index in dmuon_plan_describe's launch list)
 * of the last recorded step to out[2*i] (start) and out[2*i+1] (end) for CTA
 * i < min(cap, *n_ctas), host memory, synchronising stream; *n_ctas receives
 * the launch's CTA count (both CTAs of each pair for two-SM tiles; 0 for
 * launches that keep no records: streaming kernels and fp32 mode).
 */
dmuon_status dmuon_profile_cta_times(dmuon_plan_t plan, int32_t enable);
dmuon_status dmuon_read_cta_times(dmuon_plan_t plan, int32_t launch, uint64_t* out, int32_t cap, int32_t* n_ctas,
                                  void* stream);

/* Number of kernels the library has launched through this plan so far. */
dmuon_status dmuon_launch_count(dmuon_plan_t plan, int64_t* count);

/*
 * dmuon_selftest_wait_timeout - run one small kernel whose pipeline wait can
 * never complete (nothing arrives on its barrier), with a wait limit of
 * limit_ns nanoseconds (1e6..5e9). The kernel gives up, records
 * DMUON_DEV_WAIT_TIMEOUT and returns; *bits receives the status it wrote.
 * Exercises the bounded-wait path of the pipelined kernels without a fault.
 * Synchronises stream. d_scratch: 256 device bytes owned by the caller.
 */
dmuon_status dmuon_selftest_wait_timeout(void* d_scratch, int64_t limit_ns, void* stream,
                                         uint32_t* bits);

/*
 * dmuon_momentum_norm_noalloc - the momentum and normalisation pass of ONE
 * matrix for callers that cannot allocate device memory: a framework whose
 * allocator already holds the whole GPU, a plugin handed only the tensors it
 * must update, or a runtime that forbids allocation in its steady state.
 * The pages have no counterpart; it is the plan-free form of the first
 * launch of dmuon_step, with its reduction scratch (per-tile partial sums)
 * in a static device array of the library instead of a workspace.
 *
 *  grad       device, rows x cols, grad_dtype (DMUON_F32 or DMUON_BF16), read only.
 *  momentum   device, rows x cols fp32, updated in place: M <- mu*M + G.
 *  u_out      device, m x u_ld elements of u_dtype, m = min(rows, cols),
 *             u_ld = round_up(max(rows, cols), 8): U = G + mu*M (Nesterov) or
 *             U = M, stored transposed when rows > cols (short side first).
 *  s_out      device, one float: 1 / (||U||_F + eps).
 *
 * Limit: ceil(rows/64) * ceil(cols/128) <= 65536 (e.g. 8192 x 8192 fits);
 * larger matrices return DMUON_ERR_UNSUPPORTED. The static array (256 KiB +
 * 256 B) stays allocated on every GPU that loads the library until the
 * process exits. The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current, and so does the
 * first call after the device's context was replaced (cudaDeviceReset); make
 * that first call before any stream capture. A CUDA error that earlier work
 * left pending is reported (DMUON_ERR_CUDA, left pending) before anything is
 * launched. The call allocates nothing: it launches two
 * kernels on stream (the tile pass, which writes one partial sum per tile,
 * and a one-block kernel that adds them in a fixed order and writes s_out).
 * 16-byte aligned grad, momentum and u_out (with cols % 4 == 0) take the
 * vectorised path; other alignments are accepted and go element by element.
 * Every call shares the array and it keeps the last call's contents; calls
 * that overlap on the GPU race and give wrong results.
 */
dmuon_status dmuon_momentum_norm_noalloc(const void* grad, float* momentum, void* u_out, float* s_out,
                                         int64_t rows, int64_t cols, int32_t grad_dtype, int32_t u_dtype,
                                         float mu, int32_t nesterov, float eps, void* stream);

/*
 * dmuon_assign_owners - choose one owner rank for every matrix so that the
 * largest predicted per-rank load is small ("DMuon: Efficient Distributed
 * Muon Training with Near-Adam Overhead", gist.science summary section 2.1:
 * one owner per matrix runs its update; section 2.3: minimise the predicted
 * makespan over owner ranks, greedy when the search space is large).
 *
 *  shapes[n_mats]   stored shapes (host).
 *  ns_steps         0..16; with costs == NULL the cost of a matrix is its
 *                   Newton-Schulz flops (symmetric products counted once;
 *                   ns_steps 0 counts as 1).
 *  costs            optional host array of n_mats finite costs >= 0 (e.g.
 *                   measured times); NULL = the flop count above.
 *  n_ranks          >= 1.
 *  owner_out        host array of n_mats: the owner rank of each matrix.
 *  load_out         optional host array of n_ranks: the summed cost per rank.
 *
 * Longest-processing-time-first greedy, then moves and swaps out of the
 * most-loaded rank while they lower the makespan. Deterministic: every rank
 * that calls it with the same arguments gets the same assignment. Host only.
 */
dmuon_status dmuon_assign_owners(const dmuon_shape* shapes, int32_t n_mats, int32_t ns_steps,
                                 const double* costs, int32_t n_ranks, int32_t* owner_out,
                                 double* load_out);

/*
 * dmuon_adamw_flat - one AdamW step over a flat buffer of n elements, for the
 * parameters the Muon predicate leaves out ("DMuon" project docs, section
 * "DMuon 能做什么": everything else is optimised by AdamW with its own
 * learning rate, adamw_lr). Decoupled weight decay and bias correction:
 *   p <- p*(1 - lr*wd);  m <- b1*m + (1-b1)*g;  v <- b2*v + (1-b2)*g^2
 *   p <- p - lr/(1-b1^t) * m / (sqrt(v)/sqrt(1-b2^t) + eps)
 *
 *  param        device, n elements of param_dtype (DMUON_F32/DMUON_BF16), in place.
 *  grad         device, n elements of grad_dtype, read only.
 *  exp_avg, exp_avg_sq  device, n fp32 each (m and v), in place.
 *  step         t >= 1 (the step being taken); 0 <= beta1, beta2 < 1; eps >= 0.
 * All four pointers 16-byte aligned. One kernel on stream; no allocation.
 */
dmuon_status dmuon_adamw_flat(void* param, const void* grad, float* exp_avg, float* exp_avg_sq, int64_t n,
                              int32_t param_dtype, int32_t grad_dtype, float lr, float beta1, float beta2,
                              float eps, float weight_decay, int32_t step, void* stream);

/* Free the host-side plan (the workspace stays the caller's). NULL is a no-op. */
void dmuon_plan_destroy(dmuon_plan_t plan);

/* Message of the last error on this thread ("" if none). */
const char* dmuon_last_error(void);

/* Library version: major*10000 + minor*100 + patch. */
int32_t dmuon_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DMUON_H */
