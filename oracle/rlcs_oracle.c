/*
 * Float64 CPU oracle for the seven RL credit-assignment estimators.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may include, link or
 * call this file: only the tests, the package smoke check and the bench's CPU
 * baseline leg use it. It shares no code, header, table or constant with the
 * CUDA library.
 *
 * Each function is the estimator's *defining sequential recursion*, evaluated
 * in double, one row at a time, in the direction the definition runs. No scan,
 * no blocking, no reassociation.
 *
 * Source pages (rl-triton):
 *   - "rl-triton" technical summary, Methodology 1 (Unified Algebraic
 *     Framework): the recurrence A_t = alpha_t + beta_t * A_{t+1} and its
 *     forward-time mirror.
 *   - same page, Methodology 3 (Explicit Boundary Semantics): a terminated
 *     step has successor value zero; a truncated step bootstraps from a
 *     supplied value; the rollout-window end t = T-1 takes the bootstrap value
 *     exactly once.
 *   - rl-triton README, "Kernels" table: one row per estimator (GAE,
 *     V-Trace, Retrace, TD(lambda), discounted returns, eligibility traces
 *     e[t] = x[t] + gamma*lambda*(1-d[t-1])*e[t-1], episodic prefix sum).
 * Where the pages name an estimator but do not print its recursion (V-Trace,
 * Retrace), the published definitions the names refer to are used:
 * IMPALA V-trace (Espeholt et al., 2018, eq. 1 and the policy-gradient
 * advantage of sec. 4.2) and Retrace(lambda) (Munos et al., 2016, eq. 3 with
 * c_s = lambda * min(c_bar, pi/mu)).
 *
 * Conventions shared by every backward estimator (readings of the pages):
 *   - A mask entry counts as set when it is nonzero (0/1 floats in practice).
 *   - Successor value S_t: 0 if terminated[t]; else next_values[t] if
 *     truncated[t]; else bootstrap[n] (0 when no bootstrap array) if t = T-1;
 *     else values[t+1]. Termination wins over truncation.
 *   - A step is a cut when it is terminated, truncated, or t = T-1: the
 *     recursion does not reach past a cut; it uses S_t instead.
 * Forward estimators (eligibility traces, prefix sum) reset when the
 * *previous* step was done: d[t-1] != 0, and start from 0 before t = 0.
 *
 * Layout: every per-step array is [N, T], row-major, time-contiguous, fp32
 * (int32 for the prefix-sum input and output); outputs are float64 so the
 * comparison sees the oracle at full precision. The prefix sum wraps modulo
 * 2^32 like int32 two's-complement addition.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#define SET(mask, i) ((mask)[i] != 0.0f)

/* Successor value S_t of the boundary rules (Methodology 3). `values` may be
 * NULL only when the caller never reaches the values[t+1] case itself
 * (discounted returns ask for S_t only at cut steps). */
static double successor(const float *values, const float *term,
                        const float *trunc, const float *next_values,
                        double boot, int64_t t, int64_t T) {
  if (SET(term, t)) return 0.0;
  if (trunc != NULL && SET(trunc, t)) return (double)next_values[t];
  if (t == T - 1) return boot;
  return (double)values[t + 1];
}

static int is_cut(const float *term, const float *trunc, int64_t t,
                  int64_t T) {
  if (SET(term, t)) return 1;
  if (trunc != NULL && SET(trunc, t)) return 1;
  return t == T - 1;
}

static double row_boot(const float *bootstrap, int64_t n) {
  return bootstrap != NULL ? (double)bootstrap[n] : 0.0;
}

/* GAE (README Kernels table, compute_gae: one-step TD errors accumulated
 * backward with weight gamma*lambda):
 *   delta_t = r_t + gamma*S_t - V_t
 *   A_t     = delta_t + gamma*lambda*A_{t+1}   (A_{t+1} dropped at a cut). */
void oracle_gae(int64_t N, int64_t T, const float *rewards,
                const float *values, const float *terminateds,
                const float *truncateds, const float *next_values,
                const float *bootstrap, double gamma, double lambda,
                double *advantages) {
  for (int64_t n = 0; n < N; ++n) {
    const float *r = rewards + n * T, *v = values + n * T;
    const float *d = terminateds + n * T;
    const float *tr = truncateds ? truncateds + n * T : NULL;
    const float *nv = next_values ? next_values + n * T : NULL;
    double *out = advantages + n * T;
    double boot = row_boot(bootstrap, n);
    double a_next = 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
      double s = successor(v, d, tr, nv, boot, t, T);
      double delta = (double)r[t] + gamma * s - (double)v[t];
      double a = delta;
      if (!is_cut(d, tr, t, T)) a += gamma * lambda * a_next;
      out[t] = a;
      a_next = a;
    }
  }
}

/* TD(lambda) returns (README Kernels table, compute_lambda_returns: the
 * lambda-weighted blend of n-step returns), recursive form:
 *   G_t = r_t + gamma*((1-lambda)*V_{t+1} + lambda*G_{t+1})   not a cut
 *   G_t = r_t + gamma*S_t                                       at a cut  */
void oracle_lambda_returns(int64_t N, int64_t T, const float *rewards,
                           const float *values, const float *terminateds,
                           const float *truncateds, const float *next_values,
                           const float *bootstrap, double gamma,
                           double lambda, double *returns) {
  for (int64_t n = 0; n < N; ++n) {
    const float *r = rewards + n * T, *v = values + n * T;
    const float *d = terminateds + n * T;
    const float *tr = truncateds ? truncateds + n * T : NULL;
    const float *nv = next_values ? next_values + n * T : NULL;
    double *out = returns + n * T;
    double boot = row_boot(bootstrap, n);
    double g_next = 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
      double g;
      if (is_cut(d, tr, t, T)) {
        g = (double)r[t] + gamma * successor(v, d, tr, nv, boot, t, T);
      } else {
        g = (double)r[t] +
            gamma * ((1.0 - lambda) * (double)v[t + 1] + lambda * g_next);
      }
      out[t] = g;
      g_next = g;
    }
  }
}

/* Discounted reward-to-go (README Kernels table):
 *   G_t = r_t + gamma*G_{t+1}   not a cut
 *   G_t = r_t + gamma*S_t       at a cut (S_t never needs values here). */
void oracle_discounted_returns(int64_t N, int64_t T, const float *rewards,
                               const float *terminateds,
                               const float *truncateds,
                               const float *next_values,
                               const float *bootstrap, double gamma,
                               double *returns) {
  for (int64_t n = 0; n < N; ++n) {
    const float *r = rewards + n * T;
    const float *d = terminateds + n * T;
    const float *tr = truncateds ? truncateds + n * T : NULL;
    const float *nv = next_values ? next_values + n * T : NULL;
    double *out = returns + n * T;
    double boot = row_boot(bootstrap, n);
    double g_next = 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
      double g;
      if (is_cut(d, tr, t, T))
        g = (double)r[t] + gamma * successor(NULL, d, tr, nv, boot, t, T);
      else
        g = (double)r[t] + gamma * g_next;
      out[t] = g;
      g_next = g;
    }
  }
}

/* V-trace (README Kernels table, compute_vtrace: value targets and
 * advantages corrected by clipped importance ratios;
 * IMPALA eq. 1 in recursive form, lambda folded into the trace weight):
 *   rho_t = min(rho_bar, exp(log_rho_t)),  c_t = lambda*min(c_bar, exp(log_rho_t))
 *   vs_t - V_t = rho_t*(r_t + gamma*S_t - V_t)
 *                + gamma*c_t*(vs_{t+1} - V_{t+1})           (dropped at a cut)
 *   pg_t = rho_t*(r_t + gamma*W_t - V_t),  W_t = S_t at a cut, else vs_{t+1}.
 * pg may be NULL. */
void oracle_vtrace(int64_t N, int64_t T, const float *rewards,
                   const float *values, const float *log_rhos,
                   const float *terminateds, const float *truncateds,
                   const float *next_values, const float *bootstrap,
                   double gamma, double lambda, double rho_bar, double c_bar,
                   double *vs, double *pg) {
  for (int64_t n = 0; n < N; ++n) {
    const float *r = rewards + n * T, *v = values + n * T;
    const float *lr = log_rhos + n * T;
    const float *d = terminateds + n * T;
    const float *tr = truncateds ? truncateds + n * T : NULL;
    const float *nv = next_values ? next_values + n * T : NULL;
    double *vs_row = vs + n * T;
    double *pg_row = pg ? pg + n * T : NULL;
    double boot = row_boot(bootstrap, n);
    double vs_next = 0.0, v_next = 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
      double ratio = exp((double)lr[t]);
      double rho = fmin(rho_bar, ratio);
      double c = lambda * fmin(c_bar, ratio);
      double s = successor(v, d, tr, nv, boot, t, T);
      int cut = is_cut(d, tr, t, T);
      double diff = rho * ((double)r[t] + gamma * s - (double)v[t]);
      if (!cut) diff += gamma * c * (vs_next - v_next);
      double vs_t = (double)v[t] + diff;
      if (pg_row != NULL) {
        double w = cut ? s : vs_next;
        pg_row[t] = rho * ((double)r[t] + gamma * w - (double)v[t]);
      }
      vs_row[t] = vs_t;
      vs_next = vs_t;
      v_next = (double)v[t];
    }
  }
}

/* Retrace(lambda) (README Kernels table, compute_retrace: an off-policy Q
 * target with clipped importance-ratio traces; Munos et al. 2016 in
 * recursive form):
 *   values_t = E_pi Q(s_t, .),  q_values_t = Q(s_t, a_t)
 *   c_{t+1} = lambda*min(c_bar, exp(log_rho_{t+1}))
 *   Qret_t = r_t + gamma*(values_{t+1} + c_{t+1}*(Qret_{t+1} - q_values_{t+1}))
 *   Qret_t = r_t + gamma*S_t                                        at a cut */
void oracle_retrace(int64_t N, int64_t T, const float *rewards,
                    const float *values, const float *q_values,
                    const float *log_rhos, const float *terminateds,
                    const float *truncateds, const float *next_values,
                    const float *bootstrap, double gamma, double lambda,
                    double c_bar, double *q_ret) {
  for (int64_t n = 0; n < N; ++n) {
    const float *r = rewards + n * T, *v = values + n * T;
    const float *q = q_values + n * T, *lr = log_rhos + n * T;
    const float *d = terminateds + n * T;
    const float *tr = truncateds ? truncateds + n * T : NULL;
    const float *nv = next_values ? next_values + n * T : NULL;
    double *out = q_ret + n * T;
    double boot = row_boot(bootstrap, n);
    double qret_next = 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
      double g;
      if (is_cut(d, tr, t, T)) {
        g = (double)r[t] + gamma * successor(v, d, tr, nv, boot, t, T);
      } else {
        double c_next = lambda * fmin(c_bar, exp((double)lr[t + 1]));
        g = (double)r[t] +
            gamma * ((double)v[t + 1] +
                     c_next * (qret_next - (double)q[t + 1]));
      }
      out[t] = g;
      qret_next = g;
    }
  }
}

/* Accumulating eligibility traces, forward in time (README Kernels table):
 *   e_t = x_t + gamma*lambda*(1 - d_{t-1})*e_{t-1},   e_{-1} = 0. */
void oracle_eligibility_traces(int64_t N, int64_t T, const float *x,
                               const float *dones, double gamma,
                               double lambda, double *traces) {
  for (int64_t n = 0; n < N; ++n) {
    const float *xr = x + n * T, *d = dones + n * T;
    double *out = traces + n * T;
    double e_prev = 0.0;
    for (int64_t t = 0; t < T; ++t) {
      double e = (double)xr[t];
      if (t > 0 && !SET(d, t - 1)) e += gamma * lambda * e_prev;
      out[t] = e;
      e_prev = e;
    }
  }
}

/* Episodic prefix sum, forward in time (README Kernels table,
 * compute_episodic_prefix_sum: a running sum restarted after each done
 * step), same reset index as the traces:
 *   s_t = x_t + (1 - d_{t-1})*s_{t-1},   s_{-1} = 0,   modulo 2^32. */
void oracle_episodic_prefix_sum(int64_t N, int64_t T, const int32_t *x,
                                const float *dones, int32_t *out) {
  for (int64_t n = 0; n < N; ++n) {
    const int32_t *xr = x + n * T;
    const float *d = dones + n * T;
    int32_t *o = out + n * T;
    uint32_t s_prev = 0u;
    for (int64_t t = 0; t < T; ++t) {
      uint32_t s = (uint32_t)xr[t];
      if (t > 0 && !SET(d, t - 1)) s += s_prev;
      o[t] = (int32_t)s;
      s_prev = s;
    }
  }
}

/* Generic segmented first-order affine recurrence on raw coefficients
 * (technical summary, Methodology 1: A_t = alpha_t + beta_t*A_{t+1} and its
 * forward mirror, here with the multiplier a and addend b given directly;
 * the Significance section points to other segmented affine recurrences):
 *   reverse = 0:  x_t = a_t*x_{t-1} + b_t,  x_{-1} = x_init[n]
 *   reverse = 1:  x_t = a_t*x_{t+1} + b_t,  x_T    = x_init[n]
 * Where reset[t] is set the neighbour term is dropped: x_t = b_t.
 * reset and x_init may be NULL (no resets, x_init = 0). */
void oracle_affine_scan(int64_t N, int64_t T, const float *a, const float *b,
                        const float *reset, const float *x_init, int reverse,
                        double *x) {
  for (int64_t n = 0; n < N; ++n) {
    const float *ar = a + n * T, *br = b + n * T;
    const float *rr = reset ? reset + n * T : NULL;
    double *out = x + n * T;
    double prev = x_init ? (double)x_init[n] : 0.0;
    for (int64_t i = 0; i < T; ++i) {
      int64_t t = reverse ? T - 1 - i : i;
      double v = (double)br[t];
      if (rr == NULL || !SET(rr, t)) v += (double)ar[t] * prev;
      out[t] = v;
      prev = v;
    }
  }
}
