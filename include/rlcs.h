/*
 * rlcs.h — C ABI of the GB300 affine-scan library for RL credit assignment.
 *
 * Seven estimators, each one batched first-order linear recurrence over
 * [N, T] rollouts (N environments, T steps), solved on the GPU as an
 * associative scan over affine pairs:
 *
 *   backward estimators:  A_t = alpha_t + beta_t * A_{t+1}
 *   forward estimators:   e_t = alpha_t + beta_t * e_{t-1}
 *   pair operator:        (alpha_B, beta_B) (+) (alpha_A, beta_A)
 *                         = (alpha_B + beta_B*alpha_A, beta_A*beta_B)
 *
 * (rl-triton technical summary, Methodology 1 "Unified Algebraic Framework".)
 * Each entry point builds its own (alpha_t, beta_t) in registers from the raw
 * inputs and writes only the final outputs (same page, Methodology 2).
 *
 * ---------------------------------------------------------------------------
 * Conventions common to every entry point
 * ---------------------------------------------------------------------------
 * Memory.    Every array pointer is DEVICE memory owned by the caller, on
 *            the current CUDA device (launches go there). The library
 *            allocates nothing and frees nothing. Every per-step array,
 *            outputs included, must hold N*T elements from its pointer: the
 *            library cannot see a buffer's size, so a shorter output is
 *            written past its end.
 * Layout.    Per-step arrays are [N, T], row-major, time-contiguous
 *            (element (n, t) at offset n*T + t). float32, except the prefix
 *            sum's int32 input and output. bootstrap_value is [N].
 *            Rows whose start is 16-byte aligned (T % 4 == 0 and 16-byte
 *            aligned base pointers) take the vectorised / bulk-copy path;
 *            anything else takes a scalar path with the same results.
 * Masks.     terminateds / truncateds / dones are 0/1 float32; an entry
 *            counts as set when it is nonzero.
 * Scalars.   gamma, lambda, rho_bar and c_bar are double. Every step is
 *            computed in fp32 with the scalars rounded to fp32, but where
 *            an estimator's multiplier between cuts is one constant beta
 *            (discounted returns: gamma; GAE, TD(lambda) returns, traces:
 *            gamma*lambda) the multiplier of a 4-, 8- or 16-step span is
 *            beta^k raised in double and rounded once. Over long undamped
 *            horizons (1/(1-beta) steps) the fp32 rounding of beta itself,
 *            and of products of it, would otherwise add up: at gamma = 0.997
 *            over 16384 steps the rounding of gamma alone moves discounted
 *            returns by 2e-4 of max(1, |G|).
 * Boundary.  (Methodology 3 "Explicit Boundary Semantics".) The successor
 *            value of step t is: 0 if terminateds[t] is set; otherwise
 *            next_values[t] if truncateds[t] is set; otherwise
 *            bootstrap_value[n] when t = T-1; otherwise values[t+1].
 *            Termination wins when both masks are set. A step with any of
 *            these three conditions is a cut: nothing is carried across it.
 *            truncateds and next_values must be both NULL (no truncation)
 *            or both non-NULL. bootstrap_value may be NULL (taken as 0).
 * Aliasing.  Outputs must not overlap any input or each other; identical
 *            input/output pointers are rejected with RLCS_ERR_INVALID_ARG.
 * Streams.   Every call is asynchronous on `stream` (a cudaStream_t; NULL is
 *            the legacy default stream) and never synchronises the host,
 *            except rlcs_check_status. Calls can be captured in CUDA graphs.
 * Workspace. Long rows are split across thread blocks that pass carries
 *            through `workspace`. Size it with rlcs_workspace_bytes(N, T)
 *            and zero it once (rlcs_workspace_init, or any memset to 0)
 *            before its first use; afterwards every call leaves it ready for
 *            the next one. One workspace must not be used by two calls that
 *            can run at the same time (give each stream its own). It may be
 *            NULL with workspace_bytes = 0 only when the call needs none;
 *            otherwise the call returns RLCS_ERR_WORKSPACE and launches
 *            nothing.
 * Errors.    Argument errors (N <= 0, T <= 0, NULL required pointer, half a
 *            truncation pair, aliasing, workspace too small) return before
 *            anything is launched. A launch failure returns RLCS_ERR_CUDA.
 *            Device-side conditions (a bounded wait that ran out) are
 *            recorded in the workspace and reported by rlcs_check_status.
 * Device.    The library is built for sm_103a (GB300) only.
 */
#ifndef RLCS_H_
#define RLCS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so the header needs no CUDA. */
typedef struct CUstream_st *rlcs_stream_t;

typedef enum {
  RLCS_OK = 0,
  RLCS_ERR_INVALID_ARG = 1, /* bad size, NULL pointer, aliasing, half pair */
  RLCS_ERR_MISALIGNED = 2,  /* reserved: misalignment selects a scalar path */
  RLCS_ERR_WORKSPACE = 3,   /* workspace missing, too small or corrupted    */
  RLCS_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed         */
  RLCS_ERR_TIMEOUT = 5      /* a device-side bounded wait ran out           */
} rlcs_status;

/* Bytes of workspace any entry point needs for an [N, T] call: a small
 * header plus 32 bytes per possible row chunk. Depends only on N and T.
 * Returns 0 if N <= 0 or T <= 0. */
size_t rlcs_workspace_bytes(int64_t N, int64_t T);

/* Zero `bytes` of `workspace` on `stream` (asynchronous). */
rlcs_status rlcs_workspace_init(void *workspace, size_t bytes,
                                rlcs_stream_t stream);

/* Synchronise `stream`, then read and clear the device-side status that
 * calls using `workspace` recorded (RLCS_ERR_TIMEOUT when a bounded wait ran
 * out, RLCS_ERR_WORKSPACE when the workspace was not initialised; the higher
 * code wins when both happened). Returns
 * RLCS_ERR_CUDA if the stream reported an error. workspace may be NULL, in
 * which case only the stream is checked. */
rlcs_status rlcs_check_status(void *workspace, rlcs_stream_t stream);

/* Static, human-readable name of a status code. */
const char *rlcs_status_string(rlcs_status status);

/* Generalized Advantage Estimation.
 * rl-triton README, Kernels table, compute_gae: the one-step TD errors
 * accumulated backward with weight gamma*lambda; boundary rules of
 * Methodology 3.
 *   delta_t = r_t + gamma*S_t - V_t          (S_t: successor value above)
 *   A_t     = delta_t + gamma*lambda*A_{t+1} (nothing carried across a cut)
 * Inputs rewards, values, terminateds [N,T]; optional truncateds and
 * next_values [N,T]; optional bootstrap_value [N]. Output advantages [N,T]. */
rlcs_status rlcs_gae(const float *rewards, const float *values,
                     const float *terminateds, const float *truncateds,
                     const float *next_values, const float *bootstrap_value,
                     float *advantages, int64_t N, int64_t T, double gamma,
                     double lambda, void *workspace, size_t workspace_bytes,
                     rlcs_stream_t stream);

/* TD(lambda) returns.
 * README Kernels table, compute_lambda_returns: the lambda-weighted blend
 * of n-step returns, written as a backward recursion:
 *   G_t = r_t + gamma*((1-lambda)*V_{t+1} + lambda*G_{t+1})
 *   G_t = r_t + gamma*S_t                                   at a cut
 * Same inputs as rlcs_gae; output returns [N,T] (equals GAE + values). */
rlcs_status rlcs_lambda_returns(const float *rewards, const float *values,
                                const float *terminateds,
                                const float *truncateds,
                                const float *next_values,
                                const float *bootstrap_value, float *returns,
                                int64_t N, int64_t T, double gamma,
                                double lambda, void *workspace,
                                size_t workspace_bytes, rlcs_stream_t stream);

/* Discounted reward-to-go.
 * README Kernels table, compute_discounted_returns:
 *   G_t = r_t + gamma*G_{t+1};   G_t = r_t + gamma*S_t at a cut.
 * Takes no values array: the successor value at a cut is 0 (terminated),
 * next_values[t] (truncated) or bootstrap_value[n] (t = T-1). */
rlcs_status rlcs_discounted_returns(const float *rewards,
                                    const float *terminateds,
                                    const float *truncateds,
                                    const float *next_values,
                                    const float *bootstrap_value,
                                    float *returns, int64_t N, int64_t T,
                                    double gamma, void *workspace,
                                    size_t workspace_bytes,
                                    rlcs_stream_t stream);

/* V-trace targets and policy-gradient advantages.
 * README Kernels table, compute_vtrace: value targets and advantages
 * corrected by clipped importance ratios; definition of IMPALA V-trace with
 * lambda in the trace:
 *   ratio_t = exp(log_rhos_t), rho_t = min(rho_bar, ratio_t),
 *   c_t = lambda*min(c_bar, ratio_t)
 *   vs_t - V_t = rho_t*(r_t + gamma*S_t - V_t) + gamma*c_t*(vs_{t+1} - V_{t+1})
 *   pg_t = rho_t*(r_t + gamma*W_t - V_t),  W_t = S_t at a cut, else vs_{t+1}
 * log_rhos = log pi(a_t|s_t) - log mu(a_t|s_t), [N,T]. Outputs vs [N,T] and
 * pg_advantages [N,T] (may be NULL to skip it). */
rlcs_status rlcs_vtrace(const float *rewards, const float *values,
                        const float *log_rhos, const float *terminateds,
                        const float *truncateds, const float *next_values,
                        const float *bootstrap_value, float *vs,
                        float *pg_advantages, int64_t N, int64_t T,
                        double gamma, double lambda, double rho_bar, double c_bar,
                        void *workspace, size_t workspace_bytes,
                        rlcs_stream_t stream);

/* Retrace(lambda) targets.
 * README Kernels table, compute_retrace: an off-policy Q target whose
 * traces are clipped importance ratios; definition of Munos et al. (2016):
 *   c_t = lambda*min(c_bar, exp(log_rhos_t))
 *   Q_t = r_t + gamma*(values_{t+1} + c_{t+1}*(Q_{t+1} - q_values_{t+1}))
 *   Q_t = r_t + gamma*S_t                                     at a cut
 * values = E_pi Q(s_t, .), q_values = Q(s_t, a_t), log_rhos of a_t; all
 * [N,T]. Output q_ret [N,T]. Note the trace at t+1 weighs the carry into t. */
rlcs_status rlcs_retrace(const float *rewards, const float *values,
                         const float *q_values, const float *log_rhos,
                         const float *terminateds, const float *truncateds,
                         const float *next_values,
                         const float *bootstrap_value, float *q_ret,
                         int64_t N, int64_t T, double gamma, double lambda,
                         double c_bar, void *workspace, size_t workspace_bytes,
                         rlcs_stream_t stream);

/* Accumulating eligibility traces, forward in time.
 * README Kernels table, compute_eligibility_traces:
 *   e_t = x_t + gamma*lambda*(1 - d_{t-1})*e_{t-1},   e_{-1} = 0.
 * Inputs x, dones [N,T]; output traces [N,T]. To cut at truncations too, OR
 * them into dones. */
rlcs_status rlcs_eligibility_traces(const float *x, const float *dones,
                                    float *traces, int64_t N, int64_t T,
                                    double gamma, double lambda,
                                    void *workspace, size_t workspace_bytes,
                                    rlcs_stream_t stream);

/* Episodic prefix sum, forward in time, int32.
 * README Kernels table, compute_episodic_prefix_sum: a running sum that
 * restarts after every done step; reset index as for the traces:
 *   s_t = x_t + (1 - d_{t-1})*s_{t-1},   s_{-1} = 0,   modulo 2^32.
 * Bit-exact. Inputs x (int32) and dones (float) [N,T]; output out (int32). */
rlcs_status rlcs_episodic_prefix_sum(const int32_t *x, const float *dones,
                                     int32_t *out, int64_t N, int64_t T,
                                     void *workspace, size_t workspace_bytes,
                                     rlcs_stream_t stream);

/* GAE advantages and TD(lambda) returns in one pass.
 * README Kernels table, compute_gae and compute_lambda_returns; the two share
 * their coefficients, and TD(lambda) returns = GAE + values. Same inputs and
 * conventions as rlcs_gae; writes advantages [N,T] and returns [N,T] from a
 * single read of the inputs (20 bytes per step instead of 32 for two calls).
 * The outputs must not overlap each other or any input. */
rlcs_status rlcs_gae_and_returns(const float *rewards, const float *values,
                                 const float *terminateds, const float *truncateds,
                                 const float *next_values, const float *bootstrap_value,
                                 float *advantages, float *returns, int64_t N, int64_t T,
                                 double gamma, double lambda, void *workspace,
                                 size_t workspace_bytes, rlcs_stream_t stream);

/* GAE on compact inputs: the same estimator, conventions and fp32 output as
 * rlcs_gae, reading rewards, values and next_values as bf16 (raw bf16 bit
 * patterns, 2 bytes each) and terminateds and truncateds as uint8 masks (a
 * byte counts as set when nonzero): 9 bytes per step read and written
 * instead of 16 (13 instead of 24 with truncation). bootstrap_value stays
 * float32 [N]. bf16 to fp32 conversion is exact; the arithmetic is fp32.
 * Rows with T % 8 == 0 and 16-byte aligned arrays run eight steps per lane
 * (one 16-byte load per bf16 input): up to T = 4096 whole rows share a tile
 * of 1024, 2048 or 4096 steps and the call needs no workspace; longer rows
 * chain tiles through the workspace. Other calls take the warp-row shape
 * (T <= 512) or the register tiles. */
rlcs_status rlcs_gae_compact(const uint16_t *rewards, const uint16_t *values,
                             const uint8_t *terminateds, const uint8_t *truncateds,
                             const uint16_t *next_values, const float *bootstrap_value,
                             float *advantages, int64_t N, int64_t T, double gamma,
                             double lambda, void *workspace, size_t workspace_bytes,
                             rlcs_stream_t stream);

/* Generic segmented first-order affine recurrence on raw coefficients.
 * The recurrence of the technical summary, Methodology 1, with a and b given
 * directly (its Significance section points to other segmented affine
 * recurrences):
 *   reverse = 0:  x_t = a_t * x_{t-1} + b_t,   x_{-1} = x_init[n]
 *   reverse = 1:  x_t = a_t * x_{t+1} + b_t,   x_T    = x_init[n]
 * a, b, x are [N,T] float32; reset [N,T] is optional (NULL: no resets) and
 * where it is nonzero the step does not depend on its neighbour (x_t = b_t);
 * x_init [N] is optional (NULL: 0). Same layout, stream, workspace and error
 * conventions as the estimators. */
rlcs_status rlcs_affine_scan(const float *a, const float *b, const float *reset,
                             const float *x_init, float *x, int64_t N, int64_t T,
                             int reverse, void *workspace, size_t workspace_bytes,
                             rlcs_stream_t stream);

/* Time-major layout. The technical summary's Problem Statement fixes the
 * estimators' operands as [num_envs, seq_len] tensors; many RL rollout
 * buffers store the same data time-major instead. Each function below is its
 * row-major namesake for arrays stored [T, N] (element (t, n) at offset
 * t*N + n; bootstrap_value and x_init stay [N]): the same estimator,
 * arguments, results and errors, without a transpose. Lane l of a warp owns
 * environment 32*g + l, so every access moves whole 128-byte row segments; a
 * block owns 32 environments and one chunk of steps, and chunks of the same
 * environments are linked by a decoupled look-back.
 *
 * Workspace: rlcs_workspace_bytes_tm(N, T) bytes, prepared as for the
 * row-major entries (zeroed once, one per stream, never shared by calls that
 * may overlap). It is required only when T spans more than one chunk (the
 * size function still answers nonzero for shorter rows); when it is missing
 * or short the call returns RLCS_ERR_WORKSPACE and launches nothing. */
size_t rlcs_workspace_bytes_tm(int64_t N, int64_t T);

rlcs_status rlcs_gae_tm(const float *rewards, const float *values, const float *terminateds,
                        const float *truncateds, const float *next_values,
                        const float *bootstrap_value, float *advantages, int64_t N, int64_t T,
                        double gamma, double lambda, void *workspace, size_t workspace_bytes,
                        rlcs_stream_t stream);
rlcs_status rlcs_lambda_returns_tm(const float *rewards, const float *values,
                                   const float *terminateds, const float *truncateds,
                                   const float *next_values, const float *bootstrap_value,
                                   float *returns, int64_t N, int64_t T, double gamma,
                                   double lambda, void *workspace, size_t workspace_bytes,
                                   rlcs_stream_t stream);
rlcs_status rlcs_discounted_returns_tm(const float *rewards, const float *terminateds,
                                       const float *truncateds, const float *next_values,
                                       const float *bootstrap_value, float *returns, int64_t N,
                                       int64_t T, double gamma, void *workspace,
                                       size_t workspace_bytes, rlcs_stream_t stream);
rlcs_status rlcs_vtrace_tm(const float *rewards, const float *values, const float *log_rhos,
                           const float *terminateds, const float *truncateds,
                           const float *next_values, const float *bootstrap_value, float *vs,
                           float *pg_advantages, int64_t N, int64_t T, double gamma,
                           double lambda, double rho_bar, double c_bar, void *workspace,
                           size_t workspace_bytes, rlcs_stream_t stream);
rlcs_status rlcs_retrace_tm(const float *rewards, const float *values, const float *q_values,
                            const float *log_rhos, const float *terminateds,
                            const float *truncateds, const float *next_values,
                            const float *bootstrap_value, float *q_ret, int64_t N, int64_t T,
                            double gamma, double lambda, double c_bar, void *workspace,
                            size_t workspace_bytes, rlcs_stream_t stream);
rlcs_status rlcs_eligibility_traces_tm(const float *x, const float *dones, float *traces,
                                       int64_t N, int64_t T, double gamma, double lambda,
                                       void *workspace, size_t workspace_bytes,
                                       rlcs_stream_t stream);
rlcs_status rlcs_episodic_prefix_sum_tm(const int32_t *x, const float *dones, int32_t *out,
                                        int64_t N, int64_t T, void *workspace,
                                        size_t workspace_bytes, rlcs_stream_t stream);
rlcs_status rlcs_gae_and_returns_tm(const float *rewards, const float *values,
                                    const float *terminateds, const float *truncateds,
                                    const float *next_values, const float *bootstrap_value,
                                    float *advantages, float *returns, int64_t N, int64_t T,
                                    double gamma, double lambda, void *workspace,
                                    size_t workspace_bytes, rlcs_stream_t stream);
rlcs_status rlcs_affine_scan_tm(const float *a, const float *b, const float *reset,
                                const float *x_init, float *x, int64_t N, int64_t T, int reverse,
                                void *workspace, size_t workspace_bytes, rlcs_stream_t stream);

/* Grouped calls. Up to RLCS_MAX_GROUP estimator calls run in as few kernel
 * launches as possible instead of one launch each: every call computes
 * exactly what its namesake entry point computes (same definitions, same
 * validation), on its own arrays and sizes. A launch has a fixed cost of a
 * few microseconds whatever its size, which dominates calls of a few MB
 * (4096 x 128 rows), and each long-row launch ends in a partly idle wave;
 * one grid for the group pays both once. The paper has no counterpart: it is
 * a launch-level convenience for the seven estimators.
 *
 * rlcs_call: one call. `estimator` selects the namesake; the pointer fields
 * are that entry point's arguments (rewards holds x for the two forward
 * estimators, int32 for the prefix sum; terminateds holds their dones; out
 * is the first output, out2 V-trace's pg_advantages (may be NULL) or the
 * fused call's returns). Fields the estimator does not take are ignored;
 * `reserved` must be 0. All pointers are device memory owned by the caller.
 *
 * Classes and launches: short rows (T <= 512) are grouped by strips per row
 * (T <= 128, <= 256, <= 512) and by whether their truncation inputs are
 * present; long rows (T > 512) by tile length (chosen from the rows of all
 * the group's long calls together) and the same flag. Each class is one
 * launch, in the order of first appearance, on `stream`.
 *
 * Workspace: rlcs_group_workspace_bytes(calls, n) bytes (0 when no long call
 * spans several tiles; NULL is then allowed), prepared like the other
 * workspaces (zeroed once, one per stream, never shared by calls that may
 * overlap). Long calls of one group share it.
 *
 * Errors: RLCS_ERR_INVALID_ARG for more than RLCS_MAX_GROUP calls, any
 * argument a call's namesake would reject, an output of one call overlapping
 * any array of another call (the calls run concurrently), or a workspace
 * overlapping any array; RLCS_ERR_WORKSPACE for a missing, short or
 * misaligned workspace; nothing is launched then. RLCS_ERR_CUDA if a launch
 * fails. */
#define RLCS_MAX_GROUP 16
typedef enum {
  RLCS_EST_GAE = 0,
  RLCS_EST_LAMBDA_RETURNS = 1,
  RLCS_EST_DISCOUNTED_RETURNS = 2,
  RLCS_EST_VTRACE = 3,
  RLCS_EST_RETRACE = 4,
  RLCS_EST_ELIGIBILITY_TRACES = 5,
  RLCS_EST_EPISODIC_PREFIX_SUM = 6,
  RLCS_EST_GAE_AND_RETURNS = 7
} rlcs_estimator;

typedef struct {
  int32_t estimator; /* rlcs_estimator */
  int32_t reserved;  /* must be 0 */
  const void *rewards;
  const float *values;
  const float *q_values;
  const float *log_rhos;
  const float *terminateds;
  const float *truncateds;
  const float *next_values;
  const float *bootstrap_value;
  void *out;
  float *out2;
  int64_t N, T;
  double gamma, lambda, rho_bar, c_bar;
} rlcs_call;

size_t rlcs_group_workspace_bytes(const rlcs_call *calls, int n_calls);
rlcs_status rlcs_run_group(const rlcs_call *calls, int n_calls, void *workspace,
                           size_t workspace_bytes, rlcs_stream_t stream);

/* GAE for callers that cannot allocate device memory.
 * The paper has no counterpart: this is a library convenience. Some callers
 * cannot call cudaMalloc, such as a plugin inside a host program that owns
 * every device allocation, or a real-time loop that forbids allocating after
 * start-up; they cannot provide the workspace long rows need. This entry
 * point takes the same arguments as rlcs_gae minus the workspace and gives
 * the same results; long rows pass their carries through a fixed scratch
 * array that the library keeps in device memory (64 + 32*65536 bytes, about
 * 2 MiB, held on every GPU that loads the library until the process exits).
 * It calls no allocation routine.
 *  - Sizes: returns RLCS_ERR_WORKSPACE, launching nothing, when
 *    N * ceil(T / 1024) > 65536, the array's capacity in chunk records
 *    (the same count rlcs_workspace_bytes(N, T) is based on).
 *  - Set-up: the first call on each device looks up the array's device
 *    address and zeroes it, synchronously; make that first call before any
 *    CUDA stream capture.
 *  - Sharing: every call on a device uses the same array and leaves its
 *    contents behind, so calls that can overlap on the GPU (other streams,
 *    other threads) race; the caller must serialise them. Device-side wait
 *    timeouts are recorded in the array; read them, and repair the array,
 *    with rlcs_gae_noalloc_recover. */
rlcs_status rlcs_gae_noalloc(const float *rewards, const float *values,
                             const float *terminateds, const float *truncateds,
                             const float *next_values, const float *bootstrap_value,
                             float *advantages, int64_t N, int64_t T, double gamma,
                             double lambda, rlcs_stream_t stream);

/* Status and repair of rlcs_gae_noalloc's scratch array on the current
 * device (the paper has no counterpart). Synchronises `stream`, reads the
 * status that earlier rlcs_gae_noalloc calls recorded in the array
 * (RLCS_ERR_TIMEOUT when a bounded wait ran out, RLCS_ERR_WORKSPACE when the
 * array's counters were found inconsistent), then zeroes the whole array on
 * `stream` and waits for that, which returns it to its initial state: the
 * header counters and every chunk record, so no flag of an earlier call can
 * match a later one. Returns the status it read (RLCS_OK if none), or
 * RLCS_ERR_CUDA if a CUDA call failed. Call it after a call reported an
 * error, after calls may have overlapped, or whenever a caller wants to
 * check; no rlcs_gae_noalloc call may be in flight on the device meanwhile.
 * It allocates nothing. */
rlcs_status rlcs_gae_noalloc_recover(rlcs_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RLCS_H_ */
