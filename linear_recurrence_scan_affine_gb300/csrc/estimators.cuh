// Per-estimator coefficient functors: each turns the raw inputs of one step
// into its affine pair (beta_t, alpha_t) in registers, and turns the scanned
// value back into the estimator's output(s). Nothing here touches memory.
//
// Boundary rules (rl-triton technical summary, Methodology 3): the successor
// value S_t of step t is 0 if the step terminated, next_values[t] if it was
// truncated, bootstrap[n] at the window end t = T-1, else values[t+1]; such a
// step is a cut and carries nothing across (beta_t = 0). Termination wins.
#pragma once

#include "scan_core.cuh"

namespace rlcs {

// Input slots. Backward estimators use R, V, Q, LR, D (+ TAU, NV with
// truncation); forward ones put x in R and the done mask in D.
enum Slot : int { kR = 0, kV = 1, kQ = 2, kLR = 3, kD = 4, kTau = 5, kNV = 6, kNumSlots = 7 };

constexpr uint32_t bit(int s) { return 1u << s; }

struct Params {
  const float *in[kNumSlots];  // device pointers, [N, T]; unused slots NULL
  const float *boot;           // [N] or NULL
  void *out0;                  // [N, T] float (int32 for the prefix sum)
  float *out1;                 // [N, T] second output (V-trace pg) or NULL
  int64_t N, T;
  float gamma, lambda, rho_bar, c_bar;  // the call's scalars, rounded to fp32
  // beta^4, beta^8, beta^16 for estimators whose multiplier between cuts is
  // one constant beta (kConstBeta): raised in double from the call's double
  // scalars and rounded once. Unused (0) for the others.
  float beta4, beta8, beta16;
  int vec;                     // 1: rows 16-byte aligned (T % 4 == 0, aligned bases)
};

// What a functor sees for step t. Fields an estimator does not use are never
// loaded (their slots are absent from its masks) and fold away.
struct StepIn {
  float r, v, q, lr, d, tau, nv;  // at t
  float vn, qn, lrn;              // at t+1 (backward, only where needed)
  float dp;                       // done mask at t-1 (forward)
  bool last;                      // t == T-1
  bool first;                     // t == 0
};

template <bool TRUNC>
__device__ __forceinline__ float successor(const StepIn &s, float boot, bool &cut) {
  const bool term = s.d != 0.0f;
  const bool trunc = TRUNC && s.tau != 0.0f;
  cut = term || trunc || s.last;
  return term ? 0.0f : (trunc ? s.nv : (s.last ? boot : s.vn));
}

constexpr uint32_t kTruncSlots = bit(kTau) | bit(kNV);

// Element formats of the input slots. By default every slot is float32; a
// functor that takes compact inputs names its bf16 slots (raw bf16 bits) and
// its uint8 slots (0/1 masks), and the kernels convert them on load.
struct F32Slots {
  static constexpr uint32_t kBF16Slots = 0u;
  static constexpr uint32_t kU8Slots = 0u;
  // The multiplier between cuts is one constant beta (0 at a cut): spans of
  // 4, 8 or 16 steps then take beta^k from Params instead of a product of k
  // fp32 factors (see span_multiplier in kernels.cuh).
  static constexpr bool kConstBeta = false;
};

// ---------------------------------------------------------------------------
// GAE: alpha = r + gamma*S - V, beta = gamma*lambda (0 at a cut). Out: A.
// ---------------------------------------------------------------------------
struct Gae : F32Slots {
  static constexpr bool kConstBeta = true;  // beta = gamma*lambda
  static constexpr uint32_t kOptSlots = kTruncSlots;  // slots added when the optional input is given
  static constexpr bool kUsesRowValue = true;  // reads bootstrap_value[n]
  static constexpr bool kPrevD = false;         // reads the done mask at t-1
  static constexpr bool kBackward = true;
  static constexpr uint32_t kSlots = bit(kR) | bit(kV) | bit(kD);
  static constexpr uint32_t kNext = bit(kV);
  static constexpr int kOuts = 1;
  using Pair = FPair;
  template <bool TRUNC>
  __device__ static __forceinline__ void coeff(const Params &p, const StepIn &s, float boot,
                                               Pair &e, float &, float &) {
    bool cut;
    const float S = successor<TRUNC>(s, boot, cut);
    e.c = fmaf(p.gamma, S, s.r) - s.v;
    e.m = cut ? 0.0f : p.gamma * p.lambda;
  }
  __device__ static __forceinline__ float out0(float A, float, const Pair &, float, float) {
    return A;
  }
};

// ---------------------------------------------------------------------------
// TD(lambda) returns: alpha = r + gamma*(1-lambda)*V_{t+1}, beta = gamma*lambda;
// at a cut alpha = r + gamma*S, beta = 0. Out: G.
// ---------------------------------------------------------------------------
struct LambdaReturns : F32Slots {
  static constexpr bool kConstBeta = true;  // beta = gamma*lambda
  static constexpr uint32_t kOptSlots = kTruncSlots;  // slots added when the optional input is given
  static constexpr bool kUsesRowValue = true;  // reads bootstrap_value[n]
  static constexpr bool kPrevD = false;         // reads the done mask at t-1
  static constexpr bool kBackward = true;
  static constexpr uint32_t kSlots = bit(kR) | bit(kV) | bit(kD);
  static constexpr uint32_t kNext = bit(kV);
  static constexpr int kOuts = 1;
  using Pair = FPair;
  template <bool TRUNC>
  __device__ static __forceinline__ void coeff(const Params &p, const StepIn &s, float boot,
                                               Pair &e, float &, float &) {
    bool cut;
    const float S = successor<TRUNC>(s, boot, cut);
    const float w = cut ? p.gamma : p.gamma * (1.0f - p.lambda);
    e.c = fmaf(w, S, s.r);  // S == V_{t+1} when not a cut
    e.m = cut ? 0.0f : p.gamma * p.lambda;
  }
  __device__ static __forceinline__ float out0(float A, float, const Pair &, float, float) {
    return A;
  }
};

// ---------------------------------------------------------------------------
// Discounted returns: alpha = r (+ gamma*S at a cut), beta = gamma (0 at a cut).
// ---------------------------------------------------------------------------
struct DiscountedReturns : F32Slots {
  static constexpr uint32_t kOptSlots = kTruncSlots;  // slots added when the optional input is given
  static constexpr bool kConstBeta = true;  // beta = gamma
  static constexpr bool kUsesRowValue = true;  // reads bootstrap_value[n]
  static constexpr bool kPrevD = false;         // reads the done mask at t-1
  static constexpr bool kBackward = true;
  static constexpr uint32_t kSlots = bit(kR) | bit(kD);
  static constexpr uint32_t kNext = 0;
  static constexpr int kOuts = 1;
  using Pair = FPair;
  template <bool TRUNC>
  __device__ static __forceinline__ void coeff(const Params &p, const StepIn &s, float boot,
                                               Pair &e, float &, float &) {
    const bool term = s.d != 0.0f;
    const bool trunc = TRUNC && s.tau != 0.0f;
    const bool cut = term || trunc || s.last;
    const float S = term ? 0.0f : (trunc ? s.nv : boot);  // only used at a cut
    e.c = cut ? fmaf(p.gamma, S, s.r) : s.r;
    e.m = cut ? 0.0f : p.gamma;
  }
  __device__ static __forceinline__ float out0(float A, float, const Pair &, float, float) {
    return A;
  }
};

// ---------------------------------------------------------------------------
// V-trace (IMPALA, lambda in the trace weight):
//   rho = min(rho_bar, e^lr), c = lambda*min(c_bar, e^lr)   (e^lr by __expf)
//   alpha = rho*(r + gamma*S - V), beta = gamma*c (0 at a cut), A = vs - V.
// Outputs vs = V + A and pg = alpha + [not cut]*gamma*rho*A_{t+1}, which is
// rho*(r + gamma*W - V) with W = vs_{t+1} (or S at a cut).
// aux0 = gamma*rho (0 at a cut), aux1 = V.
// ---------------------------------------------------------------------------
struct VTrace : F32Slots {
  static constexpr uint32_t kOptSlots = kTruncSlots;  // slots added when the optional input is given
  static constexpr bool kUsesRowValue = true;  // reads bootstrap_value[n]
  static constexpr bool kPrevD = false;         // reads the done mask at t-1
  static constexpr bool kBackward = true;
  static constexpr uint32_t kSlots = bit(kR) | bit(kV) | bit(kLR) | bit(kD);
  static constexpr uint32_t kNext = bit(kV);
  static constexpr int kOuts = 2;
  using Pair = FPair;
  template <bool TRUNC>
  __device__ static __forceinline__ void coeff(const Params &p, const StepIn &s, float boot,
                                               Pair &e, float &aux0, float &aux1) {
    bool cut;
    const float S = successor<TRUNC>(s, boot, cut);
    const float ratio = __expf(s.lr);  // fast exponential: ~1e-6 relative error
    const float rho = fminf(p.rho_bar, ratio);
    const float c = p.lambda * fminf(p.c_bar, ratio);
    e.c = rho * (fmaf(p.gamma, S, s.r) - s.v);
    e.m = cut ? 0.0f : p.gamma * c;
    aux0 = cut ? 0.0f : p.gamma * rho;
    aux1 = s.v;
  }
  __device__ static __forceinline__ float out0(float A, float, const Pair &, float, float v) {
    return v + A;
  }
  __device__ static __forceinline__ float out1(float, float A_next, const Pair &e, float g_rho,
                                               float) {
    return fmaf(g_rho, A_next, e.c);
  }
};

// ---------------------------------------------------------------------------
// Retrace(lambda) (Munos et al.), values = E_pi Q(s_t,.), q = Q(s_t, a_t):
//   c_{t+1} = lambda*min(c_bar, e^{lr_{t+1}})
//   alpha = r + gamma*(V_{t+1} - c_{t+1}*Q_{t+1}), beta = gamma*c_{t+1};
//   at a cut alpha = r + gamma*S, beta = 0. Out: Q^ret.
// ---------------------------------------------------------------------------
struct Retrace : F32Slots {
  static constexpr uint32_t kOptSlots = kTruncSlots;  // slots added when the optional input is given
  static constexpr bool kUsesRowValue = true;  // reads bootstrap_value[n]
  static constexpr bool kPrevD = false;         // reads the done mask at t-1
  static constexpr bool kBackward = true;
  static constexpr uint32_t kSlots = bit(kR) | bit(kV) | bit(kQ) | bit(kLR) | bit(kD);
  static constexpr uint32_t kNext = bit(kV) | bit(kQ) | bit(kLR);
  static constexpr int kOuts = 1;
  using Pair = FPair;
  template <bool TRUNC>
  __device__ static __forceinline__ void coeff(const Params &p, const StepIn &s, float boot,
                                               Pair &e, float &, float &) {
    bool cut;
    const float S = successor<TRUNC>(s, boot, cut);
    if (cut) {
      e.c = fmaf(p.gamma, S, s.r);
      e.m = 0.0f;
    } else {
      const float c_next = p.lambda * fminf(p.c_bar, __expf(s.lrn));
      e.c = fmaf(p.gamma, fmaf(-c_next, s.qn, s.vn), s.r);
      e.m = p.gamma * c_next;
    }
  }
  __device__ static __forceinline__ float out0(float A, float, const Pair &, float, float) {
    return A;
  }
};

// ---------------------------------------------------------------------------
// Eligibility traces (forward): alpha = x, beta = gamma*lambda*(1 - d_{t-1}),
// beta_0 = 0 (e_{-1} = 0). Out: e.
// ---------------------------------------------------------------------------
struct EligibilityTraces : F32Slots {
  static constexpr bool kConstBeta = true;  // beta = gamma*lambda
  static constexpr uint32_t kOptSlots = 0u;  // slots added when the optional input is given
  static constexpr bool kUsesRowValue = false;  // reads bootstrap_value[n]
  static constexpr bool kPrevD = true;         // reads the done mask at t-1
  static constexpr bool kBackward = false;
  static constexpr uint32_t kSlots = bit(kR) | bit(kD);
  static constexpr uint32_t kNext = 0;
  static constexpr int kOuts = 1;
  using Pair = FPair;
  template <bool TRUNC>
  __device__ static __forceinline__ void coeff(const Params &p, const StepIn &s, float,
                                               Pair &e, float &, float &) {
    e.c = s.r;
    e.m = (s.first || s.dp != 0.0f) ? 0.0f : p.gamma * p.lambda;
  }
  __device__ static __forceinline__ float out0(float A, float, const Pair &, float, float) {
    return A;
  }
};

// ---------------------------------------------------------------------------
// Episodic prefix sum (forward, int32 modulo 2^32): alpha = x, carry flag
// m = (1 - d_{t-1}), m_0 = 0. The int32 input travels in slot R as raw bits.
// ---------------------------------------------------------------------------
struct EpisodicPrefixSum : F32Slots {
  static constexpr uint32_t kOptSlots = 0u;  // slots added when the optional input is given
  static constexpr bool kUsesRowValue = false;  // reads bootstrap_value[n]
  static constexpr bool kPrevD = true;         // reads the done mask at t-1
  static constexpr bool kBackward = false;
  static constexpr uint32_t kSlots = bit(kR) | bit(kD);
  static constexpr uint32_t kNext = 0;
  static constexpr int kOuts = 1;
  using Pair = IPair;
  template <bool TRUNC>
  __device__ static __forceinline__ void coeff(const Params &, const StepIn &s, float, Pair &e,
                                               float &, float &) {
    e.c = __float_as_uint(s.r);
    e.m = (s.first || s.dp != 0.0f) ? 0u : 1u;
  }
};

// ---------------------------------------------------------------------------
// GAE and TD(lambda) returns in one pass: the GAE pairs, with outputs
// A_t and G_t = A_t + V_t (the identity TD(lambda) = GAE + V).
// ---------------------------------------------------------------------------
struct GaeAndReturns : F32Slots {
  static constexpr bool kConstBeta = true;  // beta = gamma*lambda
  static constexpr uint32_t kOptSlots = kTruncSlots;
  static constexpr bool kUsesRowValue = true;
  static constexpr bool kPrevD = false;
  static constexpr bool kBackward = true;
  static constexpr uint32_t kSlots = bit(kR) | bit(kV) | bit(kD);
  static constexpr uint32_t kNext = bit(kV);
  static constexpr int kOuts = 2;
  using Pair = FPair;
  template <bool TRUNC>
  __device__ static __forceinline__ void coeff(const Params &p, const StepIn &s, float boot,
                                               Pair &e, float &, float &aux1) {
    Gae::coeff<TRUNC>(p, s, boot, e, aux1, aux1);
    aux1 = s.v;
  }
  __device__ static __forceinline__ float out0(float A, float, const Pair &, float, float) {
    return A;
  }
  __device__ static __forceinline__ float out1(float A, float, const Pair &, float, float v) {
    return v + A;
  }
};

// ---------------------------------------------------------------------------
// Generic first-order affine recurrence on raw coefficients (the segmented
// affine scan the technical summary's Significance section points to):
//   forward   x_t = a_t * x_{t-1} + b_t,   x_{-1} = x_init[n]
//   backward  x_t = a_t * x_{t+1} + b_t,   x_T    = x_init[n]
// b travels in slot R, a in slot Q, the optional reset mask in slot D. Where
// reset[t] is set the step does not depend on its neighbour: x_t = b_t. The
// step at the scan origin folds x_init into its addend.
// ---------------------------------------------------------------------------
template <bool BACKWARD>
struct Affine : F32Slots {
  static constexpr uint32_t kOptSlots = bit(kD);
  static constexpr bool kUsesRowValue = true;
  static constexpr bool kPrevD = false;
  static constexpr bool kBackward = BACKWARD;
  static constexpr uint32_t kSlots = bit(kR) | bit(kQ);
  static constexpr uint32_t kNext = 0;
  static constexpr int kOuts = 1;
  using Pair = FPair;
  template <bool RESET>
  __device__ static __forceinline__ void coeff(const Params &, const StepIn &s, float x_init,
                                               Pair &e, float &, float &) {
    const bool cut = RESET && s.d != 0.0f;
    const bool origin = BACKWARD ? s.last : s.first;
    e.m = (cut || origin) ? 0.0f : s.q;
    e.c = (origin && !cut) ? fmaf(s.q, x_init, s.r) : s.r;
  }
  __device__ static __forceinline__ float out0(float A, float, const Pair &, float, float) {
    return A;
  }
};

// ---------------------------------------------------------------------------
// GAE on compact inputs: rewards, values and next_values as bf16, terminated
// and truncated masks as uint8 (9 bytes per step read+written instead of 16
// without truncation). The arithmetic is GAE's, in fp32, on the converted
// values (bf16 -> fp32 is exact; a mask byte counts as set when nonzero).
// ---------------------------------------------------------------------------
struct GaeCompact : Gae {
  static constexpr uint32_t kBF16Slots = bit(kR) | bit(kV) | bit(kNV);
  static constexpr uint32_t kU8Slots = bit(kD) | bit(kTau);
};

}  // namespace rlcs
