// The launch shapes of the scan, templated on an estimator functor.
//
// Data layout on chip ("strip-major"): a warp walks its span of a row in
// strips of 128 steps; in strip j lane l owns the four consecutive steps
// 128*j + 4*l .. +3, so each warp-wide float4 access covers 512 contiguous
// bytes. Per strip: each lane composes its four pairs (lane-serial
// sub-scan), a 5-round shuffle scan composes the lanes, and the strips of a
// warp are chained by their totals.
//
//  * warp_row_kernel    one warp per row (T <= 512): inputs go straight to
//                       registers with 128-bit loads; no shared memory.
//  * block_tile_kernel  the default for longer rows: one block per row tile
//                       (8 warps of 1 or 2 strips: 1024 or 2048 steps; 16 or
//                       32 warps of 2 strips: 4096 or 8192 steps), inputs in registers,
//                       warp aggregates composed in shared memory, the tiles of a
//                       row chained in a single pass by a decoupled look-back
//                       through the workspace (self-validating 64-bit
//                       records, epoch tags, bounded waits), tiles in
//                       row-interleaved order.
//  * block_chunk_kernel the selectable alternative: chunks staged into shared
//                       memory by cp.async.bulk (1-D TMA) completing on an
//                       mbarrier, chained in ticket order.
//  * eight_step_tile_kernel light calls (compact GAE; float32 discounted
//                       returns) with T % 8 == 0:
//                       eight steps per lane, whole rows packed into a tile
//                       up to 4096 steps (no look-back), chained tiles
//                       beyond.
//  * group_row_kernel, group_tile_kernel: several calls in one launch, the
//                       warp-row or block-tile body per call.
//  * time_major_kernel, time_major_short_kernel: [T, N] arrays, one
//                       environment per lane, chunks of 128 steps chained
//                       by a per-lane look-back (no look-back for T <= 128).
#pragma once

#include <type_traits>

#include "estimators.cuh"

namespace rlcs {

constexpr int kStrip = 128;              // steps per warp strip
constexpr int kChunkWarps = 8;           // warps per block in the chunk tier
constexpr int kChunkThreads = kChunkWarps * 32;
#ifndef RLCS_ROW_WARPS
#define RLCS_ROW_WARPS 4
#endif
constexpr int kRowWarps = RLCS_ROW_WARPS;  // rows (warps) per block, warp-row tier
constexpr uint64_t kWaitLimitNs = 1ull << 30;  // ~1.07 s bound on every wait

// Workspace: a 64-byte header, then one 32-byte record per chunk.
struct WsHeader {
  uint32_t epoch;   // bumped by the last block of every chunked launch
  uint32_t ticket;  // next chunk ticket
  uint32_t done;    // blocks of the current launch that finished
  uint32_t status;  // sticky device-side error (an rlcs_status code)
  uint32_t pad[12];
};
// A chunk record holds self-validating 64-bit words, each
// (tag << 32) | payload with tag = (epoch tag << 2) | state: the aggregate
// pair (m, c) in two words of state 1, the inclusive value in one word of
// state 2. Each word is written and read with one strong 64-bit access,
// which is single-copy atomic, so a reader that sees a matching tag has that
// word's payload whole. No fence orders the words, and none is needed: the
// aggregate counts only when both of its words carry the current tag.
struct WsRecord {
  uint64_t m;    // aggregate multiplier bits, state 1
  uint64_t c;    // aggregate addend bits, state 1
  uint64_t inc;  // inclusive value bits (value at the chunk's far end), state 2
  uint64_t pad;
};
static_assert(sizeof(WsHeader) == 64 && sizeof(WsRecord) == 32, "workspace layout");
constexpr uint32_t kStateAgg = 1u, kStateInc = 2u;
__device__ __forceinline__ uint64_t tagged(uint32_t tag, uint32_t payload) {
  return ((uint64_t)tag << 32) | payload;
}
constexpr uint32_t kTagMask = 0x3fffffffu;
constexpr uint32_t kStatusWorkspace = 3u, kStatusTimeout = 5u;

struct ChunkShape {
  WsHeader *ws;            // workspace header (records follow it); may be
                           // NULL when chunks_per_row == 1
  int64_t chunks_per_row;  // Q
  int64_t total_chunks;    // N * Q = grid size
};

// ---------------------------------------------------------------------------
// Small helpers
// ---------------------------------------------------------------------------
// q = a / b for 0 <= a, 0 < b: in 32 bits when both fit (the usual case),
// a fraction of the cost of the 64-bit routine.
__device__ __forceinline__ int64_t div_nonneg(int64_t a, int64_t b) {
  if ((((uint64_t)a | (uint64_t)b) >> 32) == 0) return (int64_t)((uint32_t)a / (uint32_t)b);
  return a / b;
}

__device__ __forceinline__ float4 f4zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }

__device__ __forceinline__ float f4get(const float4 &v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}
__device__ __forceinline__ void f4set(float4 &v, int i, float x) {
  if (i == 0) v.x = x; else if (i == 1) v.y = x; else if (i == 2) v.z = x; else v.w = x;
}

// Four consecutive steps of one row starting at t (t % 4 == 0); steps past T
// read as 0. vec: the row is 16-byte aligned and T % 4 == 0.
__device__ __forceinline__ float4 load4(const float *row, int64_t t, int64_t T, bool vec) {
  if (vec) return t < T ? __ldg(reinterpret_cast<const float4 *>(row + t)) : f4zero();
  float4 v = f4zero();
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (t + i < T) f4set(v, i, __ldg(row + t + i));
  return v;
}

__device__ __forceinline__ void store4(float *row, int64_t t, int64_t T, bool vec, float4 v) {
  if (vec) {
    if (t < T) *reinterpret_cast<float4 *>(row + t) = v;
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (t + i < T) row[t + i] = f4get(v, i);
}

// Typed access to input slot k of estimator E (float32, bf16 bits or uint8
// masks), converting to float. `off` counts elements from the slot's start.
template <class E>
__host__ __device__ constexpr int slot_bytes(int k) {
  return (E::kBF16Slots & bit(k)) ? 2 : ((E::kU8Slots & bit(k)) ? 1 : 4);
}
__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }
__device__ __forceinline__ float mask_byte(uint32_t b) { return (b & 0xffu) ? 1.0f : 0.0f; }

// Four consecutive steps starting at row + t (t % 4 == 0); steps past T read 0.
template <class E>
__device__ __forceinline__ float4 load_slot4(const Params &p, int k, int64_t row, int64_t t,
                                             int64_t T, bool vec) {
  if (E::kBF16Slots & bit(k)) {
    const uint16_t *r = reinterpret_cast<const uint16_t *>(p.in[k]) + row;
    float4 v = f4zero();
    if (vec) {
      if (t < T) {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(r + t));
        v = make_float4(bf16_bits_to_float(u.x & 0xffffu), bf16_bits_to_float(u.x >> 16),
                        bf16_bits_to_float(u.y & 0xffffu), bf16_bits_to_float(u.y >> 16));
      }
      return v;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (t + i < T) f4set(v, i, bf16_bits_to_float(__ldg(r + t + i)));
    return v;
  }
  if (E::kU8Slots & bit(k)) {
    const uint8_t *r = reinterpret_cast<const uint8_t *>(p.in[k]) + row;
    float4 v = f4zero();
    if (vec) {
      if (t < T) {
        const uint32_t u = __ldg(reinterpret_cast<const unsigned int *>(r + t));
        v = make_float4(mask_byte(u), mask_byte(u >> 8), mask_byte(u >> 16), mask_byte(u >> 24));
      }
      return v;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (t + i < T) f4set(v, i, mask_byte(__ldg(r + t + i)));
    return v;
  }
  return load4(p.in[k] + row, t, T, vec);
}

// Vector path for register-loaded spans: the lane's four steps of strip j,
// at element offset lane_off + 128*j of slot k; `left` = steps from the
// lane's first step to the row end (the strip is past the end when
// 128*j >= left). The slot pointer plus lane_off is formed once per slot and
// every strip adds an immediate, so a load costs one instruction and the
// bounds test one compare per strip.
template <class E>
__device__ __forceinline__ float4 load_lane4(const Params &p, int k, int64_t lane_off, int j,
                                             int left) {
  if (j * kStrip >= left) return f4zero();
  if (E::kBF16Slots & bit(k)) {
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(
        reinterpret_cast<const uint16_t *>(p.in[k]) + lane_off + j * kStrip));
    return make_float4(bf16_bits_to_float(u.x & 0xffffu), bf16_bits_to_float(u.x >> 16),
                       bf16_bits_to_float(u.y & 0xffffu), bf16_bits_to_float(u.y >> 16));
  }
  if (E::kU8Slots & bit(k)) {
    const uint32_t u = __ldg(reinterpret_cast<const unsigned int *>(
        reinterpret_cast<const uint8_t *>(p.in[k]) + lane_off + j * kStrip));
    return make_float4(mask_byte(u), mask_byte(u >> 8), mask_byte(u >> 16), mask_byte(u >> 24));
  }
  return __ldg(reinterpret_cast<const float4 *>(p.in[k] + lane_off + j * kStrip));
}

__device__ __forceinline__ void store_lane4(float *out, int64_t lane_off, int j, int left,
                                            float4 v) {
  if (j * kStrip < left) *reinterpret_cast<float4 *>(out + lane_off + j * kStrip) = v;
}

// One step of slot k at element offset `off` from the slot's start.
template <class E>
__device__ __forceinline__ float load_slot1(const Params &p, int k, int64_t off) {
  if (E::kBF16Slots & bit(k))
    return bf16_bits_to_float(__ldg(reinterpret_cast<const uint16_t *>(p.in[k]) + off));
  if (E::kU8Slots & bit(k))
    return mask_byte(__ldg(reinterpret_cast<const uint8_t *>(p.in[k]) + off));
  return __ldg(p.in[k] + off);
}

// L2 bulk prefetch of n elements of slot k from element offset `off`, when
// the range is 16-byte aligned in start and length (a hint: skipped if not).
template <class E>
__device__ __forceinline__ void prefetch_slot(const Params &p, int k, int64_t off, int64_t n) {
  const char *a = reinterpret_cast<const char *>(p.in[k]) + off * slot_bytes<E>(k);
  const int64_t bytes = n * slot_bytes<E>(k);
  if (((reinterpret_cast<uintptr_t>(a) | (uintptr_t)bytes) & 15u) == 0 && bytes > 0)
    prefetch_l2(a, (uint32_t)bytes);
}

// The step after each of a lane's four steps: lanes pass their first element
// down; lane 31 takes `following` (first step after the strip).
__device__ __forceinline__ float4 next4(const float4 &a, float following, int lane) {
  float n = __shfl_down_sync(kFull, a.x, 1);
  if (lane == 31) n = following;
  return make_float4(a.y, a.z, a.w, n);
}
// The step before each of a lane's four steps; lane 0 takes `preceding`.
__device__ __forceinline__ float4 prev4(const float4 &a, float preceding, int lane) {
  float q = __shfl_up_sync(kFull, a.w, 1);
  if (lane == 0) q = preceding;
  return make_float4(q, a.x, a.y, a.z);
}

template <class P>
__device__ __forceinline__ P lane_aggregate(const P (&e)[4], bool backward) {
  P a;
  if (backward) {  // e0 ∘ e1 ∘ e2 ∘ e3
    a = compose(e[2], e[3]);
    a = compose(e[1], a);
    a = compose(e[0], a);
  } else {  // e3 ∘ e2 ∘ e1 ∘ e0
    a = compose(e[1], e[0]);
    a = compose(e[2], a);
    a = compose(e[3], a);
  }
  return a;
}

// Estimators with kConstBeta: the multiplier of k consecutive steps is
// beta^k unless one of them is a cut (multiplier exactly 0). beta^k comes
// from the host, raised in double from the call's scalars and rounded once,
// so the span's multiplier carries neither the fp32 rounding of beta nor
// k-1 fp32 roundings of a product. A product's roundings are the same in
// every span without a cut, so over an undamped horizon of ~1/(1-beta)
// steps they add up (discounted returns at gamma = 0.997: a plain four-step
// product doubled the worst error). Identity padding past a row end (m = 1)
// also reads as "no cut"; such spans only compose behind the row's last
// step (a cut) or after every real step, so they never reach an output.
template <int K>
__device__ __forceinline__ float span_multiplier(const FPair (&e)[K], float beta_k) {
  bool nz = true;
#pragma unroll
  for (int j = 0; j < K; ++j) nz = nz && (e[j].m != 0.0f);
  return nz ? beta_k : 0.0f;
}
template <int K>
__device__ __forceinline__ float const_beta_power(const Params &p) {
  static_assert(K == 4 || K == 8 || K == 16, "the powers the host provides");
  return K == 4 ? p.beta4 : (K == 8 ? p.beta8 : p.beta16);
}

template <class P> struct ValueOf;
template <> struct ValueOf<FPair> { using type = float; };
template <> struct ValueOf<IPair> { using type = uint32_t; };

__device__ __forceinline__ uint32_t vbits(float x) { return __float_as_uint(x); }
__device__ __forceinline__ uint32_t vbits(uint32_t x) { return x; }
__device__ __forceinline__ void vfrom(uint32_t b, float &x) { x = __uint_as_float(b); }
__device__ __forceinline__ void vfrom(uint32_t b, uint32_t &x) { x = b; }

// Where a warp's raw inputs come from.
//  RegSource: every strip already in registers (warp-row tier).
//  SmemSource: the block's staged chunk in shared memory (chunk tier).
template <int S>
struct RegSource {
  const float4 (&raw)[kNumSlots][S];
  const float (&halo_next)[kNumSlots];  // first step after the span
  float halo_prev_d;                    // done mask just before the span
  int lane;
  __device__ __forceinline__ float4 get(int k, int j) const { return raw[k][j]; }
  __device__ __forceinline__ float following(int k, int j) const {
    return (j + 1 < S) ? __shfl_sync(kFull, raw[k][j + 1].x, 0) : halo_next[k];
  }
  __device__ __forceinline__ float preceding_d(int j) const {
    return (j > 0) ? __shfl_sync(kFull, raw[kD][j - 1].w, 31) : halo_prev_d;
  }
};

template <int S>
struct SmemSource {
  const float *slot[kNumSlots];         // per slot: the chunk's staged steps
  int span_off;                         // warp's first step within the chunk
  int chunk;                            // steps per chunk
  const float (&halo_next)[kNumSlots];  // first step after the chunk
  float halo_prev_d;                    // done mask before the chunk
  int lane;
  __device__ __forceinline__ float4 get(int k, int j) const {
    return *reinterpret_cast<const float4 *>(slot[k] + span_off + j * kStrip + 4 * lane);
  }
  __device__ __forceinline__ float following(int k, int j) const {
    const int pos = span_off + (j + 1) * kStrip;
    return pos < chunk ? slot[k][pos] : halo_next[k];
  }
  __device__ __forceinline__ float preceding_d(int j) const {
    const int pos = span_off + j * kStrip - 1;
    return pos >= 0 ? slot[kD][pos] : halo_prev_d;
  }
};

// ---------------------------------------------------------------------------
// Strip engine for one warp's span of S strips.
// ---------------------------------------------------------------------------
template <class E, bool TRUNC, int S>
struct Strips {
  using P = typename E::Pair;
  using V = typename ValueOf<P>::type;
  static constexpr uint32_t kUse = E::kSlots | (TRUNC ? E::kOptSlots : 0u);

  P el[S][4];
  float aux0[S][4], aux1[S][4];
  P excl[S], tot[S];
  float beta4;  // Params::beta4 (kConstBeta estimators)

  // t_span: the span's first step within the row; T: the row length.
  // ZERO_PAD: steps past the row end arrive as zeros (register-loaded spans).
  // Their coefficients are then finite, and they never reach a real output:
  // a backward row's last step has beta = 0 (it is a cut), and a forward
  // row's padding comes after every real step. So they need no per-step
  // identity mask. Spans staged in shared memory (uninitialised past the end)
  // keep the mask.
  template <bool ZERO_PAD = false, class Src>
  __device__ __forceinline__ void build(const Params &p, const Src &src, float boot,
                                        int64_t t_span, int64_t T, int lane) {
    beta4 = p.beta4;
    // Per-element bounds in 32-bit offsets from the span start: steps left in
    // the row (clamped; a span is at most a few thousand steps long).
    const int64_t left = T - t_span;
    const int rem = left > (int64_t)(1 << 30) ? (1 << 30) : (int)left;
    const bool at_origin = (t_span == 0);
#pragma unroll
    for (int j = 0; j < S; ++j) {
      // A strip wholly inside the row, and not holding the row's last step,
      // needs no per-step bound checks (uniform across the warp).
      if ((j + 1) * kStrip < rem && !(at_origin && j == 0))
        build_strip<true, ZERO_PAD>(p, src, boot, j, rem, false, lane);
      else
        build_strip<false, ZERO_PAD>(p, src, boot, j, rem, at_origin, lane);
    }
  }

  template <bool FULL, bool ZERO_PAD, class Src>
  __device__ __forceinline__ void build_strip(const Params &p, const Src &src, float boot, int j,
                                              int rem, bool at_origin, int lane) {
    float4 raw[kNumSlots], nx[kNumSlots];
#pragma unroll
    for (int k = 0; k < kNumSlots; ++k) raw[k] = (kUse & bit(k)) ? src.get(k, j) : f4zero();
#pragma unroll
    for (int k = 0; k < kNumSlots; ++k)
      nx[k] = (E::kBackward && (E::kNext & bit(k))) ? next4(raw[k], src.following(k, j), lane)
                                                    : f4zero();
    float4 dp = f4zero();
    if (E::kPrevD) dp = prev4(raw[kD], src.preceding_d(j), lane);
    const int o0 = j * kStrip + 4 * lane;  // offset of the lane's run in the span
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int o = o0 + i;
      StepIn s;
      s.r = f4get(raw[kR], i);
      s.v = f4get(raw[kV], i);
      s.q = f4get(raw[kQ], i);
      s.lr = f4get(raw[kLR], i);
      s.d = f4get(raw[kD], i);
      s.tau = f4get(raw[kTau], i);
      s.nv = f4get(raw[kNV], i);
      s.vn = f4get(nx[kV], i);
      s.qn = f4get(nx[kQ], i);
      s.lrn = f4get(nx[kLR], i);
      s.dp = f4get(dp, i);
      s.last = FULL ? false : (o == rem - 1);
      s.first = FULL ? false : (at_origin && o == 0);
      float a0 = 0.f, a1 = 0.f;
      P e;
      E::template coeff<TRUNC>(p, s, boot, e, a0, a1);
      if (!FULL && !ZERO_PAD && o >= rem) e = identity(P{});  // padding is the identity
      el[j][i] = e;
      aux0[j][i] = a0;
      aux1[j][i] = a1;
    }
  }

  // Lane aggregates and per-strip warp scans. Returns the span's aggregate
  // (strip 0 outermost for backward, strip S-1 outermost for forward).
  __device__ __forceinline__ P scan(int lane) {
#pragma unroll
    for (int j = 0; j < S; ++j) {
      P a = lane_aggregate(el[j], E::kBackward);
      if constexpr (E::kConstBeta) a.m = span_multiplier<4>(el[j], beta4);
      if (E::kBackward) {
        const P inc = warp_suffix_scan(a, lane);
        tot[j] = shfl_idx(inc, 0);
        const P x = shfl_down(inc, 1);
        excl[j] = (lane == 31) ? identity(P{}) : x;
      } else {
        const P inc = warp_prefix_scan(a, lane);
        tot[j] = shfl_idx(inc, 31);
        const P x = shfl_up(inc, 1);
        excl[j] = (lane == 0) ? identity(P{}) : x;
      }
    }
    P agg = identity(P{});
    if (E::kBackward) {
#pragma unroll
      for (int j = S - 1; j >= 0; --j) agg = compose(tot[j], agg);
    } else {
#pragma unroll
      for (int j = 0; j < S; ++j) agg = compose(tot[j], agg);
    }
    return agg;
  }

  // Given the value just outside the span (after it for backward, before it
  // for forward), produce every owned step's output(s).
  __device__ __forceinline__ void finish(V carry, float4 (&o0)[S], float4 (&o1)[S]) {
    V X = carry;
    V outside[S];
    if (E::kBackward) {
#pragma unroll
      for (int j = S - 1; j >= 0; --j) {
        outside[j] = X;
        X = apply(tot[j], X);
      }
    } else {
#pragma unroll
      for (int j = 0; j < S; ++j) {
        outside[j] = X;
        X = apply(tot[j], X);
      }
    }
#pragma unroll
    for (int j = 0; j < S; ++j) {
      V nb = apply(excl[j], outside[j]);  // value adjacent to the lane's run
      if (E::kBackward) {
#pragma unroll
        for (int i = 3; i >= 0; --i) {
          const V A = apply(el[j][i], nb);
          emit(j, i, A, nb, o0, o1);
          nb = A;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const V A = apply(el[j][i], nb);
          emit(j, i, A, nb, o0, o1);
          nb = A;
        }
      }
    }
  }

  __device__ __forceinline__ void emit(int j, int i, float A, float A_adj, float4 (&o0)[S],
                                       float4 (&o1)[S]) {
    f4set(o0[j], i, E::out0(A, A_adj, el[j][i], aux0[j][i], aux1[j][i]));
    if constexpr (E::kOuts > 1)
      f4set(o1[j], i, E::out1(A, A_adj, el[j][i], aux0[j][i], aux1[j][i]));
  }
  __device__ __forceinline__ void emit(int j, int i, uint32_t A, uint32_t, float4 (&o0)[S],
                                       float4 (&)[S]) {
    f4set(o0[j], i, __uint_as_float(A));
  }
};

// ---------------------------------------------------------------------------
// Warp-row tier: one warp per row, S strips (T <= 128*S).
// ---------------------------------------------------------------------------
// Rows (warps) per block of a warp-row launch (measured on GB300 at
// 4096 x 128): 8 for calls that move at most four arrays, where fewer blocks
// shorten the launch (an empty grid of 512 blocks retires in 1.2 us, of 1024
// in 1.7 us); 4 for the heavier ones, whose longer blocks spread more evenly
// over the SMs in smaller units (3, 5 and 6 rows measured slower for them).
template <class E, bool TRUNC>
constexpr int row_warps() {
  return __builtin_popcount(Strips<E, TRUNC, 1>::kUse) + E::kOuts <= 4 ? 8 : 4;
}

// One block of the warp-row tier: rows R*block .. R*block + R-1.
template <class E, bool TRUNC, int S, int R>
__device__ __forceinline__ void warp_row_body(const Params &p, int64_t block) {
  using St = Strips<E, TRUNC, S>;
  using V = typename St::V;
  const int lane = threadIdx.x & 31;
  const int64_t row = block * R + (threadIdx.x >> 5);
  const int64_t T = p.T;
  const int64_t base = row * T;
  const bool vec = p.vec != 0;
  // Start this row's inputs streaming into L2 while the previous grid in the
  // stream may still be running; the loads below come after the dependency
  // wait and find them there.
  if (vec && lane == 0 && row < p.N) {
#pragma unroll
    for (int k = 0; k < kNumSlots; ++k)
      if (St::kUse & bit(k)) prefetch_slot<E>(p, k, base, T);
  }
  pdl_wait();
  if (row >= p.N) return;  // whole warp leaves together

  const int64_t lane_off = base + 4 * lane;
  const int left = (int)(T - 4 * lane);  // T <= 512 in this tier
  float4 raw[kNumSlots][S];
#pragma unroll
  for (int k = 0; k < kNumSlots; ++k) {
#pragma unroll
    for (int j = 0; j < S; ++j) {
      if (!(St::kUse & bit(k)))
        raw[k][j] = f4zero();
      else if (vec)
        raw[k][j] = load_lane4<E>(p, k, lane_off, j, left);
      else
        raw[k][j] = load_slot4<E>(p, k, base, (int64_t)j * kStrip + 4 * lane, T, false);
    }
  }
  const float boot = (E::kUsesRowValue && p.boot) ? __ldg(p.boot + row) : 0.f;
  pdl_launch_dependents();

  float halo[kNumSlots];
#pragma unroll
  for (int k = 0; k < kNumSlots; ++k) halo[k] = 0.f;  // past the row end: never used
  const RegSource<S> src{raw, halo, 0.f, lane};
  St st;
  st.template build<true>(p, src, boot, 0, T, lane);
  st.scan(lane);
  float4 o0[S], o1[S];
  st.finish(V(0), o0, o1);
#pragma unroll
  for (int j = 0; j < S; ++j) {
    if (vec) {
      store_lane4(static_cast<float *>(p.out0), lane_off, j, left, o0[j]);
      if constexpr (E::kOuts > 1) {
        if (p.out1) store_lane4(p.out1, lane_off, j, left, o1[j]);
      }
    } else {
      const int64_t t = (int64_t)j * kStrip + 4 * lane;
      store4(static_cast<float *>(p.out0) + base, t, T, false, o0[j]);
      if constexpr (E::kOuts > 1) {
        if (p.out1) store4(p.out1 + base, t, T, false, o1[j]);
      }
    }
  }
}

template <class E, bool TRUNC, int S>
__global__ void __launch_bounds__(row_warps<E, TRUNC>() * 32) warp_row_kernel(Params p) {
  warp_row_body<E, TRUNC, S, row_warps<E, TRUNC>()>(p, blockIdx.x);
}

// ---------------------------------------------------------------------------
// Grouped warp-row launch: several independent calls on short rows (T <= 128*S)
// in one grid of kRowWarps rows per block. Call c owns blocks [first_block[c], first_block[c+1]) and runs
// the warp-row body of its estimator on them, so the group pays one launch's
// fixed cost. Calls in one group share S and whether their optional inputs are
// present.
// ---------------------------------------------------------------------------
constexpr int kMaxGroup = 16;
enum GroupKind : int {
  kGroupGae = 0,
  kGroupLambdaReturns,
  kGroupDiscountedReturns,
  kGroupVTrace,
  kGroupRetrace,
  kGroupEligibilityTraces,
  kGroupEpisodicPrefixSum,
  kGroupGaeAndReturns,
  kGroupKinds
};
struct GroupParams {
  int n;                                // calls in the group
  int kind[kMaxGroup];                  // GroupKind of each call
  int64_t first_block[kMaxGroup + 1];   // block ranges; first_block[n] = grid size
  Params p[kMaxGroup];
};

template <bool TRUNC, int S>
__global__ void __launch_bounds__(kRowWarps * 32) group_row_kernel(GroupParams gp) {
  int c = 0;  // uniform per block
  while (c + 1 < gp.n && (int64_t)blockIdx.x >= gp.first_block[c + 1]) ++c;
  const int64_t b = (int64_t)blockIdx.x - gp.first_block[c];
  const Params &p = gp.p[c];
  switch (gp.kind[c]) {
    case kGroupGae: warp_row_body<Gae, TRUNC, S, kRowWarps>(p, b); break;
    case kGroupLambdaReturns: warp_row_body<LambdaReturns, TRUNC, S, kRowWarps>(p, b); break;
    case kGroupDiscountedReturns: warp_row_body<DiscountedReturns, TRUNC, S, kRowWarps>(p, b); break;
    case kGroupVTrace: warp_row_body<VTrace, TRUNC, S, kRowWarps>(p, b); break;
    case kGroupRetrace: warp_row_body<Retrace, TRUNC, S, kRowWarps>(p, b); break;
    case kGroupEligibilityTraces: warp_row_body<EligibilityTraces, false, S, kRowWarps>(p, b); break;
    case kGroupEpisodicPrefixSum: warp_row_body<EpisodicPrefixSum, false, S, kRowWarps>(p, b); break;
    case kGroupGaeAndReturns: warp_row_body<GaeAndReturns, TRUNC, S, kRowWarps>(p, b); break;
    default: break;
  }
}

// ---------------------------------------------------------------------------
// Block-chunk tier
// ---------------------------------------------------------------------------
// Sticky device-side status: the highest code recorded wins.
__device__ __forceinline__ void set_status(WsHeader *ws, uint32_t code) {
  if (ws != nullptr) atomicMax(&ws->status, code);
}

// Bounded wait on phase 0 of the block's mbarrier. False on timeout.
__device__ __forceinline__ bool wait_bar(uint64_t *bar) {
  if (mbar_try_wait(bar, 0)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, 0)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// Decoupled look-back (warp-wide call) for the chunk whose record is
// `self`. Its predecessors in scan order are the records self - j*stride for
// j = 1..npred (nearest first). Publishes the chunk aggregate, walks the
// predecessors 32 per round until one holds an inclusive value, composes the
// aggregates in between, publishes this chunk's inclusive value and returns
// the value just outside the chunk on its scan-origin side. Every wait is
// bounded; on timeout the status word records RLCS_ERR_TIMEOUT and missing
// aggregates count as the identity, so the launch always finishes.
// `hint`: lane 0's earlier read of the nearest predecessor's inclusive word
// (0 if none was read). When it already carries this launch's inclusive
// value the look-back needs no further round trip: that word is written
// once per launch, so a matching tag read at any time is final.
template <class P, class V>
__device__ V lookback(WsHeader *ws, int64_t self, int64_t stride, int64_t npred, P agg,
                      uint32_t tag, int lane, uint64_t hint = 0) {
  WsRecord *rec = reinterpret_cast<WsRecord *>(ws + 1);
  const uint32_t tagA = (tag << 2) | kStateAgg, tagP = (tag << 2) | kStateInc;
  if (npred == 0) {  // the row's scan origin: nothing before it
    if (lane == 0) st_relaxed_gpu_u64(&rec[self].inc, tagged(tagP, vbits(apply(agg, V(0)))));
    return V(0);
  }
  const uint32_t hint_tag = __shfl_sync(kFull, (uint32_t)(hint >> 32), 0);
  if (hint_tag == tagP) {
    V Xh;
    vfrom(__shfl_sync(kFull, (uint32_t)hint, 0), Xh);
    if (lane == 0) st_relaxed_gpu_u64(&rec[self].inc, tagged(tagP, vbits(apply(agg, Xh))));
    return Xh;
  }
  if (lane == 0) {
    st_relaxed_gpu_u64(&rec[self].m, tagged(tagA, vbits(agg.m)));
    st_relaxed_gpu_u64(&rec[self].c, tagged(tagA, vbits(agg.c)));
  }
  P acc = identity(P{});
  V X = V(0);
  bool timed_out = false;
  int64_t d0 = 0;  // distance already walked
  while (true) {
    const int64_t dist = d0 + lane + 1;
    const bool valid = dist <= npred;
    const int64_t tk = self - dist * stride;
    uint64_t wm = 0, wc = 0, wi = 0;
    bool isP = false, isA = false;
    uint64_t start = 0;
    unsigned backoff = 64;
    while (true) {
      if (valid) {
        wi = ld_relaxed_gpu_u64(&rec[tk].inc);
        wm = ld_relaxed_gpu_u64(&rec[tk].m);
        wc = ld_relaxed_gpu_u64(&rec[tk].c);
        isP = (uint32_t)(wi >> 32) == tagP;
        isA = (uint32_t)(wm >> 32) == tagA && (uint32_t)(wc >> 32) == tagA;
      }
      if (__all_sync(kFull, !valid || isP || isA)) break;
      const uint64_t now = globaltimer_ns();
      if (start == 0) start = now;
      if (__any_sync(kFull, now - start > kWaitLimitNs)) {
        timed_out = true;
        break;
      }
      __nanosleep(backoff);  // back off so a waiting warp leaves issue slots to others
      if (backoff < 1024) backoff <<= 1;
    }
    const unsigned pm = __ballot_sync(kFull, valid && isP);
    const int firstP = pm ? __ffs(pm) - 1 : 32;
    P mine = identity(P{});
    if (valid && isA && lane < firstP) {
      vfrom((uint32_t)wm, mine.m);
      vfrom((uint32_t)wc, mine.c);
    }
    P win = warp_reduce_outer_first(mine);
    win = shfl_idx(win, 0);
    acc = compose(acc, win);
    if (pm) {
      V incv;
      vfrom(__shfl_sync(kFull, (uint32_t)wi, firstP), incv);
      X = apply(acc, incv);
      break;
    }
    if (timed_out || d0 + 32 >= npred) {  // only reachable after a timeout
      X = apply(acc, V(0));
      timed_out = true;
      break;
    }
    d0 += 32;
  }
  if (lane == 0) {
    if (timed_out) set_status(ws, kStatusTimeout);
    st_relaxed_gpu_u64(&rec[self].inc, tagged(tagP, vbits(apply(agg, X))));
  }
  return X;
}

// Marks the launch's block as finished; the last block of the launch resets
// the counters and moves the workspace to the next epoch, so the next call
// ignores every flag this one wrote.
// Called by one thread per block after the block's last use of the
// workspace (its epoch read and look-back are complete by then).
__device__ __forceinline__ void finish_launch(WsHeader *ws, int64_t total, uint32_t epoch) {
  const uint32_t prev = atomicAdd(&ws->done, 1u);
  if (prev == (uint32_t)(total - 1)) {
    ws->ticket = 0u;
    ws->done = 0u;
    __threadfence();
    ws->epoch = epoch + 1u;
  }
}

template <class E, bool TRUNC, int S>
__global__ void __launch_bounds__(kChunkThreads) block_chunk_kernel(Params p, ChunkShape cs) {
  using St = Strips<E, TRUNC, S>;
  using P = typename St::P;
  using V = typename St::V;
  constexpr int C = kChunkWarps * kStrip * S;  // steps per chunk
  constexpr uint32_t kUse = St::kUse;
  constexpr int kNumUsed = __builtin_popcount(kUse);

  extern __shared__ __align__(128) float smem[];  // [kNumUsed][C]
  __shared__ uint64_t bar;
  __shared__ P s_warp[kChunkWarps];
  __shared__ V s_carry[kChunkWarps];
  __shared__ int64_t s_ticket;
  __shared__ uint32_t s_epoch;
  __shared__ int s_ok;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool vec = p.vec != 0;
  const int64_t T = p.T, Q = cs.chunks_per_row;
  // L2 prefetch of the chunk this block will most likely get (tickets follow
  // block order closely; exact when Q == 1), issued before the dependency
  // wait so it overlaps the previous grid. A wrong guess only costs traffic.
  if (vec && tid == 0) {
    const int64_t g = blockIdx.x, grow = div_nonneg(g, Q), gk = g - grow * Q;
    const int64_t gq = E::kBackward ? (Q - 1 - gk) : gk;
    const int64_t gt0 = gq * C;
    const int64_t glen = (T - gt0 < C) ? (T - gt0) : C;
#pragma unroll
    for (int k = 0; k < kNumSlots; ++k)
      if (kUse & bit(k)) prefetch_l2(p.in[k] + grow * T + gt0, (uint32_t)(glen * 4));
  }
  pdl_wait();

  if (tid == 0) {
    int64_t ticket = blockIdx.x;
    uint32_t epoch = 0;
    int ok = 1;
    if (Q > 1) {
      ticket = atomicAdd(&cs.ws->ticket, 1u);
      if (ticket >= cs.total_chunks) {
        set_status(cs.ws, kStatusWorkspace);
        ok = 0;
      }
    }
    s_ticket = ticket;
    s_ok = ok;
    if (ok && vec) {
      const int64_t row = div_nonneg(ticket, Q), kk = ticket - row * Q;
      const int64_t q = E::kBackward ? (Q - 1 - kk) : kk;
      const int64_t t0 = q * C;
      const int64_t len = (T - t0 < C) ? (T - t0) : C;
      mbar_init(&bar, 1);
      fence_mbar_init();
      fence_proxy_async_shared();
      mbar_arrive_expect_tx(&bar, (uint32_t)(kNumUsed * len * 4));
      int idx = 0;
#pragma unroll
      for (int k = 0; k < kNumSlots; ++k) {
        if (kUse & bit(k)) {
          bulk_g2s(smem + idx * C, p.in[k] + row * T + t0, (uint32_t)(len * 4), &bar);
          ++idx;
        }
      }
    }
    if (ok && Q > 1) epoch = ld_relaxed_gpu(&cs.ws->epoch);  // after the copies are issued
    s_epoch = epoch;
  }
  __syncthreads();
  if (!s_ok) return;  // uniform: a corrupted workspace handed out a bad ticket

  const int64_t ticket = s_ticket;
  const int64_t row = div_nonneg(ticket, Q), kk = ticket - row * Q;
  const int64_t q = E::kBackward ? (Q - 1 - kk) : kk;
  const int64_t t0 = q * C;
  const int64_t base = row * T;
  const int span_off = warp * kStrip * S;

  if (!vec) {  // unaligned rows: stage with plain loads
    int idx = 0;
#pragma unroll
    for (int k = 0; k < kNumSlots; ++k) {
      if (kUse & bit(k)) {
        for (int e = tid; e < C; e += kChunkThreads)
          smem[idx * C + e] = (t0 + e < T) ? __ldg(p.in[k] + base + t0 + e) : 0.f;
        ++idx;
      }
    }
  }

  // Halo steps just outside the chunk (read while the bulk copy is in flight).
  float halo[kNumSlots];
#pragma unroll
  for (int k = 0; k < kNumSlots; ++k) {
    halo[k] = 0.f;
    if (E::kBackward && (E::kNext & bit(k)) && warp == kChunkWarps - 1 && t0 + C < T)
      halo[k] = __ldg(p.in[k] + base + t0 + C);
  }
  const float halo_d = (E::kPrevD && warp == 0 && t0 > 0) ? __ldg(p.in[kD] + base + t0 - 1)
                                                          : 0.f;
  const float boot = (E::kUsesRowValue && p.boot) ? __ldg(p.boot + row) : 0.f;

  if (vec) {
    if (!wait_bar(&bar)) set_status(cs.ws, kStatusTimeout);
  } else {
    __syncthreads();
  }
  pdl_launch_dependents();

  SmemSource<S> src{{}, span_off, C, halo, halo_d, lane};
  {
    int idx = 0;
#pragma unroll
    for (int k = 0; k < kNumSlots; ++k) {
      src.slot[k] = smem + idx * C;  // unused slots alias a used one; never read
      if (kUse & bit(k)) ++idx;
    }
  }
  St st;
  st.build(p, src, boot, t0 + span_off, T, lane);
  const P wagg = st.scan(lane);
  if (lane == 0) s_warp[warp] = wagg;
  __syncthreads();

  if (warp == 0) {
    const P w = (lane < kChunkWarps) ? s_warp[lane] : identity(P{});
    P inc, nb;
    P chunk_agg;
    if (E::kBackward) {
      inc = warp_suffix_scan(w, lane);
      chunk_agg = shfl_idx(inc, 0);
      const P x = shfl_down(inc, 1);
      nb = (lane >= kChunkWarps - 1) ? identity(P{}) : x;
    } else {
      inc = warp_prefix_scan(w, lane);
      chunk_agg = shfl_idx(inc, kChunkWarps - 1);
      const P x = shfl_up(inc, 1);
      nb = (lane == 0) ? identity(P{}) : x;
    }
    V X = V(0);
    if (Q > 1) {
      const uint32_t epoch = s_epoch;
      X = lookback<P, V>(cs.ws, ticket, 1, kk, chunk_agg, epoch & kTagMask, lane);
    }
    if (lane < kChunkWarps) s_carry[lane] = apply(nb, X);
  }
  __syncthreads();

  float4 o0[S], o1[S];
  st.finish(s_carry[warp], o0, o1);
#pragma unroll
  for (int j = 0; j < S; ++j) {
    const int64_t t = t0 + span_off + (int64_t)j * kStrip + 4 * lane;
    store4(static_cast<float *>(p.out0) + base, t, T, vec, o0[j]);
    if constexpr (E::kOuts > 1) {
      if (p.out1) store4(p.out1 + base, t, T, vec, o1[j]);
    }
  }
  if (Q > 1 && tid == 0) finish_launch(cs.ws, cs.total_chunks, s_epoch);
}

// ---------------------------------------------------------------------------
// Block-tile tier: one 256-thread block per row tile of 1024*S steps, inputs
// loaded straight into registers (each warp its own span of S strips, like
// the warp-row tier), warp aggregates composed in shared memory, tiles of a
// row chained by decoupled look-back. No shared-memory staging and low
// register use keep several blocks resident per SM, so one block's look-back
// wait overlaps other blocks' loads.
//
// Tile order: block b handles tile round r = b / N of row b % N (row-
// interleaved), at position q = r (forward) or Q-1-r (backward) along the
// row. A tile's predecessor in its row is block b - N: issued N blocks
// earlier, so with many rows its inclusive value is usually published before
// it is needed. Blocks are dispatched in index order, so every block a tile
// waits for has already been scheduled; the waits are bounded all the same.
// The bulk L2 prefetch of the tile is issued before the grid-dependency wait.
// ---------------------------------------------------------------------------
struct TileShape {
  WsHeader *ws;           // workspace (records indexed by block); NULL when Q == 1
  int64_t tiles_per_row;  // Q
  int64_t total_tiles;    // blocks of the whole launch (N * Q for a single call)
  int64_t rec_off;        // first workspace record of this call (0 for a single call)
};

// Tile layouts: W warps of S strips, W * 128 * S steps per tile. 1024- and
// 2048-step tiles are 8 warps of 1 or 2 strips; 4096- and 8192-step tiles
// are 16 or 32 warps of 2 strips, which keeps the per-thread state of the
// 2048-step tile
// (measured on GB300 against 8 warps of 4 strips at 2 blocks/SM: 256 x 4096
// single calls 3-28% faster, where a row is one tile and needs no
// look-back, 8 x 131072 4-10% faster; the 256 x 4096 grouped step 25.6
// against 26.5 us).
template <int S>
constexpr int tile_warps() {
  return S >= 8 ? 32 : (S >= 4 ? 16 : kChunkWarps);
}
template <int S>
constexpr int tile_strips() {
  return S >= 4 ? 2 : S;
}

// Resident blocks per SM the compiler must allow (measured on GB300): 2 for
// 16-warp tiles and 4 for 8 warps of 2 strips (64 registers), 6 for 1024-step
// tiles (40), so one block's look-back overlaps the others' loads.
template <int S, int W> struct TileMinBlocks {
  static constexpr int value = W >= 32 ? 1 : (W >= 16 ? 2 : (S >= 2 ? 4 : 6));
};
// Single calls of estimators that move at most four arrays: 8-warp 2048-step
// tiles at 5 blocks/SM (48 registers, a few bytes spilled). Measured on
// GB300 at 256 x 16384: discounted returns 14.3 against 15.5 us, eligibility
// traces 13.2 against 14.1, prefix sum 13.5 against 14.7. (The grouped
// launch keeps 4 blocks/SM: a separate launch for its light calls was slower
// overall.)
// 16-warp tiles of calls that move three arrays (discounted returns,
// eligibility traces, the prefix sum) run at 3 blocks/SM (40 registers, a
// few bytes spilled) when the grid spans more than one wave: measured at
// 4096 x 4096, 8-13% faster than at 2 blocks/SM; on one-wave grids
// (256 x 4096) 32% slower, so those keep 2. Calls that move four arrays
// were slower at 3 everywhere.
template <class E, bool TRUNC>
constexpr bool three_arrays() {
  return __builtin_popcount(Strips<E, TRUNC, 1>::kUse) + E::kOuts <= 3;
}
template <class E, bool TRUNC, int S, int W, bool MANY_WAVES = false> struct CallTileMinBlocks {
  static constexpr int value =
      (S == 2 && W == 8 && row_warps<E, TRUNC>() == 8) ? 5
      : (W == 16 && MANY_WAVES && three_arrays<E, TRUNC>()) ? 3
                                                             : TileMinBlocks<S, W>::value;
};

// Block b of one call's tiles (b counts from 0 within the call); W warps of
// S strips each.
template <class E, bool TRUNC, int S, int W>
__device__ __forceinline__ void tile_body(const Params &p, const TileShape &ts, int64_t b) {
  static_assert(W <= 32, "warp 0 scans the warps' aggregates");
  using St = Strips<E, TRUNC, S>;
  using P = typename St::P;
  using V = typename St::V;
  constexpr int C = W * kStrip * S;  // steps per tile
  constexpr uint32_t kUse = St::kUse;

  __shared__ P s_warp[W];
  __shared__ V s_carry[W];
  __shared__ uint32_t s_epoch;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool vec = p.vec != 0;
  const int64_t N = p.N, T = p.T, Q = ts.tiles_per_row;
  const int64_t r = div_nonneg(b, N), row = b - r * N;
  const int64_t q = E::kBackward ? (Q - 1 - r) : r;
  const int64_t t0 = q * C;
  const int64_t base = row * T;
  const int span_off = warp * kStrip * S;
  if (vec && tid == 0) {
    const int64_t len = (T - t0 < C) ? (T - t0) : C;
#pragma unroll
    for (int k = 0; k < kNumSlots; ++k)
      if (kUse & bit(k)) prefetch_slot<E>(p, k, base + t0, len);
  }
  pdl_wait();

  const int64_t t_span = t0 + span_off;
  const int64_t lane_off = base + t_span + 4 * lane;
  const int64_t left64 = T - t_span - 4 * lane;
  const int left = left64 > (int64_t)(1 << 30) ? (1 << 30) : (int)left64;
  float4 raw[kNumSlots][S];
#pragma unroll
  for (int k = 0; k < kNumSlots; ++k) {
#pragma unroll
    for (int j = 0; j < S; ++j) {
      if (!(kUse & bit(k)))
        raw[k][j] = f4zero();
      else if (vec)
        raw[k][j] = load_lane4<E>(p, k, lane_off, j, left);
      else
        raw[k][j] = load_slot4<E>(p, k, base, t_span + (int64_t)j * kStrip + 4 * lane, T, false);
    }
  }
  float halo[kNumSlots];
#pragma unroll
  for (int k = 0; k < kNumSlots; ++k) {
    const int64_t th = t_span + (int64_t)kStrip * S;  // first step after the span
    halo[k] = (E::kBackward && (E::kNext & bit(k)) && th < T) ? load_slot1<E>(p, k, base + th) : 0.f;
  }
  // A span wholly past the row end (the last tile of a row longer than
  // what is left) reads nothing: its halo is never used.
  const float halo_d =
      (E::kPrevD && t_span > 0 && t_span <= T) ? load_slot1<E>(p, kD, base + t_span - 1) : 0.f;
  const float boot = (E::kUsesRowValue && p.boot) ? __ldg(p.boot + row) : 0.f;
  if (tid == 0 && Q > 1) s_epoch = ld_relaxed_gpu(&ts.ws->epoch);  // after the loads issue
  pdl_launch_dependents();

  const RegSource<S> src{raw, halo, halo_d, lane};
  St st;
  st.template build<true>(p, src, boot, t_span, T, lane);
  const P wagg = st.scan(lane);
  // Warp 0 reads the nearest predecessor tile's inclusive word as soon as
  // its own scan is done, so the read overlaps the other warps' scans and the
  // block barrier; the look-back uses it if it is ready. (Measured on GB300:
  // the 256 x 16384 grouped step went from 105 to 96 us. Issued before the
  // pairs are built, the read mostly came too soon to find the value.)
  uint64_t hint = 0;
  if (warp == 0 && lane == 0 && Q > 1 && r > 0)
    hint = ld_relaxed_gpu_u64(&reinterpret_cast<WsRecord *>(ts.ws + 1)[ts.rec_off + b - N].inc);
  if (lane == 0) s_warp[warp] = wagg;
  __syncthreads();

  if (warp == 0) {
    const P w = (lane < W) ? s_warp[lane] : identity(P{});
    P inc, nb, tile_agg;
    if (E::kBackward) {
      inc = warp_suffix_scan(w, lane);
      tile_agg = shfl_idx(inc, 0);
      const P x = shfl_down(inc, 1);
      nb = (lane >= W - 1) ? identity(P{}) : x;
    } else {
      inc = warp_prefix_scan(w, lane);
      tile_agg = shfl_idx(inc, W - 1);
      const P x = shfl_up(inc, 1);
      nb = (lane == 0) ? identity(P{}) : x;
    }
    V X = V(0);
    if (Q > 1) {
      const uint32_t epoch = s_epoch;
      X = lookback<P, V>(ts.ws, ts.rec_off + b, N, r, tile_agg, epoch & kTagMask, lane, hint);
    }
    if (lane < W) s_carry[lane] = apply(nb, X);
  }
  __syncthreads();

  float4 o0[S], o1[S];
  st.finish(s_carry[warp], o0, o1);
#pragma unroll
  for (int j = 0; j < S; ++j) {
    if (vec) {
      store_lane4(static_cast<float *>(p.out0), lane_off, j, left, o0[j]);
      if constexpr (E::kOuts > 1) {
        if (p.out1) store_lane4(p.out1, lane_off, j, left, o1[j]);
      }
    } else {
      const int64_t t = t_span + (int64_t)j * kStrip + 4 * lane;
      store4(static_cast<float *>(p.out0) + base, t, T, false, o0[j]);
      if constexpr (E::kOuts > 1) {
        if (p.out1) store4(p.out1 + base, t, T, false, o1[j]);
      }
    }
  }
  if (Q > 1 && tid == 0) finish_launch(ts.ws, ts.total_tiles, s_epoch);
}

template <class E, bool TRUNC, int S, int W, bool MANY_WAVES>
__global__ void __launch_bounds__(W * 32, CallTileMinBlocks<E, TRUNC, S, W, MANY_WAVES>::value)
    block_tile_kernel(Params p, TileShape ts) {
  tile_body<E, TRUNC, S, W>(p, ts, blockIdx.x);
}

// ---------------------------------------------------------------------------
// Eight-step tiles, for light backward calls: compact GAE (bf16 values,
// uint8 masks) and float32 discounted returns. Each lane owns eight consecutive
// steps, so it reads each bf16 input with one 16-byte load (a float32 input
// with two) and a warp covers 256 steps with one shuffle scan. Needs
// T % 8 == 0 (a lane's eight steps never straddle two rows) and 16-byte
// aligned arrays.
//  * T <= C (the tile length, W * 256 steps: 1024 to 8192): a tile holds
//    R = C / T whole rows, scanned as one sequence. A row's last step is a
//    cut (multiplier 0), so nothing carries from a row into the row before
//    it, and a tile needs no look-back; when T divides 256 no row straddles
//    two warps either, and the block skips its barrier and shared scan.
//  * T > C: row tiles in row-interleaved order, chained by the decoupled
//    look-back as the register tiles are.
// Each layout comes in two register budgets: MINB = 8, 4 or 2 blocks/SM
// (4, 8 or 16 warps) without spills for grids of about one wave, 12, 6 or 3
// with a few spilled bytes for larger grids, where resident blocks hide
// latency; 32 warps (8192-step tiles, for few long rows whose grid fits in
// one block per SM) take the whole register file of an SM.
// ---------------------------------------------------------------------------
constexpr int kLane8 = 8;                   // steps per lane
constexpr int kStrip8 = 32 * kLane8;        // steps per warp

struct EightShape {
  WsHeader *ws;           // look-back workspace; NULL unless Q > 1
  int64_t rows_per_tile;  // R when whole rows share a tile (Q == 1)
  int64_t tiles_per_row;  // Q
  int warp_rows;          // 256 % T == 0: every warp holds whole rows
};

// Eight consecutive elements of slot k from element offset `off` (a multiple
// of 8, so every access is aligned), converted to float.
template <class E>
__device__ __forceinline__ void load8(const Params &p, int k, int64_t off, float (&x)[8]) {
  if (E::kBF16Slots & bit(k)) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(
        reinterpret_cast<const uint16_t *>(p.in[k]) + off));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else if (E::kU8Slots & bit(k)) {
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(
        reinterpret_cast<const uint8_t *>(p.in[k]) + off));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[i] = ((u.x >> (8 * i)) & 0xffu) ? 1.0f : 0.0f;
      x[4 + i] = ((u.y >> (8 * i)) & 0xffu) ? 1.0f : 0.0f;
    }
  } else {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p.in[k] + off));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p.in[k] + off + 4));
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

template <class E, bool TRUNC, int W, int MINB>
__global__ void __launch_bounds__(W * 32, MINB) eight_step_tile_kernel(Params p, EightShape es) {
  static_assert(E::kBackward && !E::kPrevD && E::kOuts == 1,
                "whole rows share a tile only where each row ends in a cut");
  using P = typename E::Pair;
  using V = typename ValueOf<P>::type;
  constexpr int C = W * kStrip8;
  constexpr uint32_t kUse = E::kSlots | (TRUNC ? E::kOptSlots : 0u);
  __shared__ P s_warp[W];
  __shared__ V s_carry[W];
  __shared__ uint32_t s_epoch;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t N = p.N, T = p.T, b = blockIdx.x, Q = es.tiles_per_row;
  const int off = warp * kStrip8 + lane * kLane8;  // lane's first step within the tile
  // The lane's row, its first step's position in the row, and whether it
  // holds steps at all; the tile's first element and length for the prefetch.
  int64_t row, pos, r = 0, t_first, t_len;
  bool valid;
  if (Q == 1) {
    const int64_t R = es.rows_per_tile, row0 = b * R;
    const int64_t rows = (N - row0 < R) ? (N - row0) : R;
    const int o = off < (int)(R * T) ? off : 0;  // R * T <= C
    row = row0 + o / (int)T;
    pos = o - (row - row0) * T;
    valid = off < rows * T;
    t_first = row0 * T;
    t_len = rows * T;
  } else {
    r = div_nonneg(b, N);
    row = b - r * N;
    const int64_t q = Q - 1 - r;  // backward: round 0 holds each row's last tile
    pos = q * C + off;
    valid = pos < T;
    t_first = row * T + q * C;
    t_len = (T - q * C < C) ? (T - q * C) : C;
  }
  const int64_t f0 = row * T + pos;  // element offset of the lane's first step
  if (tid == 0) {
#pragma unroll
    for (int k = 0; k < kNumSlots; ++k)
      if (kUse & bit(k)) prefetch_slot<E>(p, k, t_first, t_len);
  }
  pdl_wait();

  float x[kNumSlots][kLane8];
#pragma unroll
  for (int k = 0; k < kNumSlots; ++k) {
    if ((kUse & bit(k)) && valid) {
      load8<E>(p, k, f0, x[k]);
    } else {
#pragma unroll
      for (int i = 0; i < kLane8; ++i) x[k][i] = 0.f;
    }
  }
  const bool row_end = valid && pos + kLane8 == T;  // the lane's last step ends its row
  // successor values of the lane's last step: the next lane's first step,
  // or (lane 31) the first step after the warp's span, read directly
  float nxt[kNumSlots];
#pragma unroll
  for (int k = 0; k < kNumSlots; ++k) {
    nxt[k] = 0.f;
    if (E::kNext & bit(k)) {
      const float down = __shfl_down_sync(kFull, x[k][0], 1);
      if (lane < 31) nxt[k] = down;
      else if (valid && !row_end) nxt[k] = load_slot1<E>(p, k, f0 + kLane8);
    }
  }
  const float boot = (E::kUsesRowValue && p.boot && row_end) ? __ldg(p.boot + row) : 0.f;
  if (tid == 0 && Q > 1) s_epoch = ld_relaxed_gpu(&es.ws->epoch);  // after the loads issue
  pdl_launch_dependents();

  P e[kLane8];
#pragma unroll
  for (int i = 0; i < kLane8; ++i) {
    StepIn s;
    s.r = x[kR][i];
    s.v = x[kV][i];
    s.q = x[kQ][i];
    s.lr = x[kLR][i];
    s.d = x[kD][i];
    s.tau = x[kTau][i];
    s.nv = x[kNV][i];
    s.vn = i + 1 < kLane8 ? x[kV][i + 1] : nxt[kV];
    s.qn = i + 1 < kLane8 ? x[kQ][i + 1] : nxt[kQ];
    s.lrn = i + 1 < kLane8 ? x[kLR][i + 1] : nxt[kLR];
    s.dp = 0.f;
    s.last = row_end && i == kLane8 - 1;
    s.first = valid && pos + i == 0;
    float a0 = 0.f, a1 = 0.f;
    E::template coeff<TRUNC>(p, s, boot, e[i], a0, a1);
  }
  // Steps past a row end or the array end read zeros, so their pairs are
  // finite; they only compose behind a row's last step (a cut, multiplier
  // 0), so they never reach an output.
  P agg = e[kLane8 - 1];
#pragma unroll
  for (int i = kLane8 - 2; i >= 0; --i) agg = compose(e[i], agg);
  if constexpr (E::kConstBeta) agg.m = span_multiplier<kLane8>(e, p.beta8);
  const P inc = warp_suffix_scan(agg, lane);
  const P wtot = shfl_idx(inc, 0);
  const P down = shfl_down(inc, 1);
  const P excl = lane == 31 ? identity(P{}) : down;
  // Rows that divide a warp's 256 steps never straddle two warps: each warp
  // ends at a row end, so nothing passes between warps (uniform per launch).
  V carry = V(0);
  if (!es.warp_rows) {
    uint64_t hint = 0;  // the nearest predecessor tile's inclusive word, read early
    if (warp == 0 && lane == 0 && Q > 1 && r > 0)
      hint = ld_relaxed_gpu_u64(&reinterpret_cast<WsRecord *>(es.ws + 1)[b - N].inc);
    if (lane == 0) s_warp[warp] = wtot;
    __syncthreads();
    if (warp == 0) {
      const P w = (lane < W) ? s_warp[lane] : identity(P{});
      const P winc = warp_suffix_scan(w, lane);
      const P tile_agg = shfl_idx(winc, 0);
      const P x1 = shfl_down(winc, 1);
      const P nb = (lane >= W - 1) ? identity(P{}) : x1;
      V X = V(0);
      if (Q > 1) X = lookback<P, V>(es.ws, b, N, r, tile_agg, s_epoch & kTagMask, lane, hint);
      if (lane < W) s_carry[lane] = apply(nb, X);
    }
    __syncthreads();
    carry = s_carry[warp];
  }

  V nbv = apply(excl, carry);  // the value just after the lane's steps
  float o[kLane8];
#pragma unroll
  for (int i = kLane8 - 1; i >= 0; --i) {
    const V A = apply(e[i], nbv);
    o[i] = E::out0(A, nbv, e[i], 0.f, 0.f);
    nbv = A;
  }
  if (valid) {
    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out0) + f0);
    dst[0] = make_float4(o[0], o[1], o[2], o[3]);
    dst[1] = make_float4(o[4], o[5], o[6], o[7]);
  }
  if (Q > 1 && tid == 0) finish_launch(es.ws, N * Q, s_epoch);
}

// Grouped long-row launch: several calls' tiles in one grid, each call's
// tiles in its own row-interleaved order (block b of a call: round b / N of
// row b % N). All calls share one workspace: a call's look-back records
// start at its rec_off, and the launch's single epoch is moved on by the
// last block of the calls that chain tiles (ts.total_tiles counts those
// blocks only). Two block orders:
//  * contiguous: call c owns blocks [first_block[c], first_block[c+1]);
//  * round-major (round_rows > 0: every call has round_rows rows and the
//    same number of tiles per row): round r of call 0, round r of call 1,
//    ..., then round r+1. A tile's predecessor in its row then sits n
//    segments of round_rows blocks earlier instead of one, so it has
//    usually finished, and the look-back's early read finds its inclusive
//    value. Each segment still reads neighbouring rows of one array.
//    (Interleaving single blocks of the calls measured 1.5x slower.)
// Either way a tile waits only on lower block indices.
struct GroupTileParams {
  int n;
  int kind[kMaxGroup];
  int64_t first_block[kMaxGroup + 1];
  int64_t round_rows;  // > 0: round-major order (see above); 0: contiguous
  Params p[kMaxGroup];
  TileShape ts[kMaxGroup];
};

template <bool TRUNC, int S, int W>
__global__ void __launch_bounds__(W * 32, TileMinBlocks<S, W>::value)
    group_tile_kernel(GroupTileParams gp) {
  int c = 0;  // uniform per block
  int64_t b;
  if (gp.round_rows > 0) {
    const int64_t B = blockIdx.x, seg = div_nonneg(B, gp.round_rows);  // (round, call) segment
    const int64_t rnd = div_nonneg(seg, (int64_t)gp.n);
    c = (int)(seg - rnd * gp.n);
    b = rnd * gp.round_rows + (B - seg * gp.round_rows);
  } else {
    while (c + 1 < gp.n && (int64_t)blockIdx.x >= gp.first_block[c + 1]) ++c;
    b = (int64_t)blockIdx.x - gp.first_block[c];
  }
  const Params &p = gp.p[c];
  const TileShape &ts = gp.ts[c];
  switch (gp.kind[c]) {
    case kGroupGae: tile_body<Gae, TRUNC, S, W>(p, ts, b); break;
    case kGroupLambdaReturns: tile_body<LambdaReturns, TRUNC, S, W>(p, ts, b); break;
    case kGroupDiscountedReturns: tile_body<DiscountedReturns, TRUNC, S, W>(p, ts, b); break;
    case kGroupVTrace: tile_body<VTrace, TRUNC, S, W>(p, ts, b); break;
    case kGroupRetrace: tile_body<Retrace, TRUNC, S, W>(p, ts, b); break;
    case kGroupEligibilityTraces: tile_body<EligibilityTraces, false, S, W>(p, ts, b); break;
    case kGroupEpisodicPrefixSum: tile_body<EpisodicPrefixSum, false, S, W>(p, ts, b); break;
    case kGroupGaeAndReturns: tile_body<GaeAndReturns, TRUNC, S, W>(p, ts, b); break;
    default: break;
  }
}

// ---------------------------------------------------------------------------
// Time-major tier: inputs and outputs [T, N] (element (t, n) at t*N + n).
// Lane l of every warp owns environment n = 32*g + l of the block's group g,
// so each load or store instruction of a warp moves one 128-byte row segment
// (32 consecutive environments at one step) and no data passes through
// shared memory. A block owns one chunk of kTmChunk steps of its 32
// environments; warp w holds steps [L*w, L*(w+1)) of the chunk in registers
// (L = 8 or 16) and composes them serially, per lane, into one affine pair.
// The warps' pairs meet in shared memory, and warp 0 links the chunk to the
// chunks before it in scan order with a per-environment decoupled look-back
// (one workspace record per environment and chunk). Each warp then walks its
// steps again from its carry-in and stores the outputs.
// ---------------------------------------------------------------------------
constexpr int kTmChunk = 128;  // steps per block (one chunk of 32 environments)
constexpr int kTmEnvs = 32;    // environments per block (one per lane)
// A block of kTmChunk/L warps, each holding L steps of the chunk in registers.
template <int L>
constexpr int tm_threads() {
  return kTmChunk / L * 32;
}
// Resident blocks per SM the compiler must allow, for 8-warp blocks (16
// steps per lane; the 32-environment kernel from T = 1024 and the
// 8-environment kernel's 512-step chunks) and 16-warp blocks (8 steps per
// lane, L = 8):
//  * 2 by default, which caps the heaviest instances at 128 registers
//    (measured on GB300: Retrace at 256 x 16384 took 42.7 us uncapped and
//    31.5 us capped);
//  * 3 (80 registers) for calls that move four arrays with one output
//    (GAE, TD(lambda) returns): GAE 5-7% faster at 256 x 16384 and
//    1024 x 4096; V-trace and Retrace spilled and slowed by up to 1.6x there;
//  * for three-array calls, 4 (64 registers), or 3 for the ones that spill
//    more there (eligibility traces 24-56 bytes, the affine scan 32-56).
//    Measured against 2 (us): 8-environment chunks, discounted returns
//    128 x 16384 9.6 / 11.3, 32 x 65536 11.5 / 13.1, prefix sum 128 x 16384
//    9.3 / 11.8, 256 x 8192 10.2 / 11.9, traces at 3 128 x 16384 10.5 / 10.9
//    (10.1 at 4), 32 x 65536 11.7 / 12.8 (12.2 at 4); 32-environment chunks
//    (which held 3 blocks at 80 registers), discounted returns 1024 x 16384
//    46.8 / 50.0, 512 x 8192 16.4 / 16.9, prefix sum 1024 x 16384 47.6 /
//    51.6;
//  * at L = 8, 1 for four arrays or more, 2 for three-array calls (the prefix
//    sum used 67 registers uncapped, one 512-thread block per SM).
template <class E>
struct TmThreeArrayBlocks {
  static constexpr int value = 4;
};
template <>
struct TmThreeArrayBlocks<EligibilityTraces> {
  static constexpr int value = 3;
};
template <bool B>
struct TmThreeArrayBlocks<Affine<B>> {
  static constexpr int value = 3;
};
template <class E, bool TRUNC, int L>
constexpr int tm_min_blocks() {
  return L < 16 ? (three_arrays<E, TRUNC>() ? 2 : 1)
         : three_arrays<E, TRUNC>()
             ? TmThreeArrayBlocks<E>::value
             : (__builtin_popcount(E::kSlots | (TRUNC ? E::kOptSlots : 0u)) + E::kOuts == 4 &&
                        E::kOuts == 1
                    ? 3
                    : 2);
}

struct TmShape {
  WsHeader *ws;    // workspace header; NULL when one chunk covers T
  int64_t groups;  // G = ceil(N / 32) (ceil(N / 8) for the 8-environment chunks)
  int64_t chunks;  // chunks per environment = ceil(T / chunk length)
  int slots;       // look-back distances per warp and round, per environment (8-environment chunks: 1 or 4)
};

// One record of a chunk: its inclusive value (kStateInc), its aggregate
// pair (kStateAgg), or nothing of this epoch yet (0). The aggregate words
// are read only when the inclusive word is stale (measured on GB300:
// reading all three at once was up to 2 us slower, e.g. discounted returns
// at 256 x 16384 20.7 against 18.7 us).
template <class P, class V>
__device__ __forceinline__ uint32_t tm_read_record(const WsRecord *r, uint32_t tagA, uint32_t tagP,
                                                   P &pv) {
  const uint64_t wi = ld_relaxed_gpu_u64(&r->inc);
  if ((uint32_t)(wi >> 32) == tagP) {
    vfrom((uint32_t)wi, pv.c);
    return kStateInc;
  }
  const uint64_t wm = ld_relaxed_gpu_u64(&r->m), wc = ld_relaxed_gpu_u64(&r->c);
  if ((uint32_t)(wm >> 32) == tagA && (uint32_t)(wc >> 32) == tagA) {
    vfrom((uint32_t)wm, pv.m);
    vfrom((uint32_t)wc, pv.c);
    return kStateAgg;
  }
  return 0u;
}

template <class P, class V, int kWarps>
struct TmSlices {
  P acc[kWarps][32];         // per warp and environment: the warp's records composed, up to its stop
  uint32_t val[kWarps][32];  // the inclusive value's bits where the warp met one
  uint32_t stop[kWarps][32]; // 0: none, 1: inclusive value, 2: wait ran out, 3: scan origin
  uint32_t open[32];         // environment still walking (set by warp 0 between rounds)
  uint32_t more;
};

// Decoupled look-back of the time-major tier, one chain per environment,
// run by the whole block. A warp's lanes cover 32/kSub environments, lane l
// taking environment l % (32/kSub) and distance slot l / (32/kSub); the
// first `slots` (1..kSub) slots read. The record of environment e for this
// chunk is self + e; its predecessors in scan order are self + e - d*stride
// for d = 1..npred. Warp 0 publishes the chunk aggregate of every
// environment. Then, round by round, warp w takes the distances
// d0 + w*slots + 1 .. d0 + (w+1)*slots, one per reading slot: each lane
// reads its record, waits (bounded) if it is not yet published, and the
// slots of an environment combine nearest first (stopping at an inclusive
// value) with shuffles; warp 0 chains the warps' results in order. One L2
// round trip thus brings a window of kWarps*slots predecessors for every
// environment, and the waits on unpublished records run in parallel. (Many chunks of an environment are in flight at once when there
// are few environment groups; walking them one record per round trip was
// the time-major tier's main cost.) On a timeout the status word records
// RLCS_ERR_TIMEOUT and the missing aggregates count as the identity.
// Environments past N (env_ok false) neither publish nor wait. Every thread
// of the block calls this; `agg` is read in warp 0's lanes of slot 0, where
// the value just outside the chunk on its scan-origin side is returned and
// the chunk's inclusive value published.
template <class P, class V, int kSub, int kWarps>
__device__ V tm_lookback(WsHeader *ws, int64_t self, int64_t stride, int64_t npred, P agg,
                         uint32_t tag, int lane, int warp, bool env_ok, int slots,
                         TmSlices<P, V, kWarps> &sl) {
  static_assert(kSub == 1 || kSub == 2 || kSub == 4, "distance slots per warp");
  constexpr int kE = 32 / kSub;  // environments per warp
  const int env = lane % kE, slot = lane / kE;
  const int nsub = slots < 1 ? 1 : (slots > kSub ? kSub : slots);
  const bool owner = warp == 0 && slot == 0;  // publishes and walks for `env`
  WsRecord *mine = reinterpret_cast<WsRecord *>(ws + 1) + self + env;
  const uint32_t tagA = (tag << 2) | kStateAgg, tagP = (tag << 2) | kStateInc;
  if (npred == 0) {  // the scan origin: nothing before it
    if (owner && env_ok) st_relaxed_gpu_u64(&mine->inc, tagged(tagP, vbits(apply(agg, V(0)))));
    return V(0);
  }
  if (owner) {
    if (env_ok) {
      st_relaxed_gpu_u64(&mine->m, tagged(tagA, vbits(agg.m)));
      st_relaxed_gpu_u64(&mine->c, tagged(tagA, vbits(agg.c)));
    }
    sl.open[env] = env_ok ? 1u : 0u;
  }
  __syncthreads();
  P acc = identity(P{});
  V X = V(0);
  bool done = !(owner && env_ok), timed_out = false;
  const int window = nsub * kWarps;
  for (int64_t d0 = 0;; d0 += window) {
    P sacc = identity(P{});
    uint32_t stop = 0u, sval = 0u;
    const int64_t d = d0 + warp * nsub + slot + 1;
    if (slot < nsub && sl.open[env]) {
      if (d > npred) {  // every predecessor composed: the origin's value is 0
        stop = 3u;
      } else {
        const WsRecord *r = mine - d * stride;
        uint32_t s = tm_read_record<P, V>(r, tagA, tagP, sacc);
        if (s == 0u) {  // not yet published: wait for it (bounded)
          const uint64_t t0 = globaltimer_ns();
          unsigned backoff = 64;
          while ((s = tm_read_record<P, V>(r, tagA, tagP, sacc)) == 0u) {
            if (globaltimer_ns() - t0 > kWaitLimitNs) break;
            __nanosleep(backoff);
            if (backoff < 1024) backoff <<= 1;
          }
        }
        if (s == 0u) {
          stop = 2u;
          sacc = identity(P{});
        } else if (s == kStateInc) {
          stop = 1u;
          sval = vbits(sacc.c);
          sacc = identity(P{});
        }
      }
    }
    // the slots of each environment, nearest first: a slot that stopped
    // hides the farther ones (nsub is uniform over the block)
    // (measured on GB300, skipping it for one slot: 256 x 16384 GAE 19.9
    // against 20.5 us, 256 x 4096 V-trace 8.6 against 9.3)
    if (nsub > 1) {
#pragma unroll
      for (int off = kE; off < 32; off <<= 1) {
        const P o = shfl_down(sacc, off);
        const uint32_t ostop = __shfl_down_sync(kFull, stop, off);
        const uint32_t oval = __shfl_down_sync(kFull, sval, off);
        if (stop == 0u && slot + (off / kE) < nsub) {
          sacc = compose(sacc, o);
          stop = ostop;
          sval = oval;
        }
      }
    }
    if (slot == 0) {
      sl.acc[warp][env] = sacc;
      sl.stop[warp][env] = stop;
      sl.val[warp][env] = sval;
    }
    __syncthreads();
    if (warp == 0) {
      if (slot == 0) {
        for (int w = 0; w < kWarps && !done; ++w) {
          acc = compose(acc, sl.acc[w][env]);
          const uint32_t st = sl.stop[w][env];
          if (st == 1u) {
            V v;
            vfrom(sl.val[w][env], v);
            X = apply(acc, v);
            done = true;
          } else if (st != 0u) {  // the origin, or a wait that ran out (missing terms count as identity)
            X = apply(acc, V(0));
            done = true;
            if (st == 2u) timed_out = true;
          }
        }
        sl.open[env] = done ? 0u : 1u;
      }
      const bool more = __any_sync(kFull, !done);
      if (lane == 0) sl.more = more ? 1u : 0u;
    }
    __syncthreads();
    if (!sl.more) break;
  }
  if (owner) {
    if (timed_out) set_status(ws, kStatusTimeout);
    if (env_ok) st_relaxed_gpu_u64(&mine->inc, tagged(tagP, vbits(apply(agg, X))));
  }
  return X;
}

__device__ __forceinline__ float ldg_at(const void *base, int64_t byte_off) {
  return __ldg(reinterpret_cast<const float *>(static_cast<const char *>(base) + byte_off));
}

// L2 bulk prefetch of rows [t0, t1) of every input slot in the [T, N]
// layout. Those rows are one contiguous range per slot, read in 32- or
// 128-byte pieces by the `parts` blocks of that chunk (one per environment
// group, adjacent in launch order); block `part` prefetches the part-th
// 16-byte-aligned share, so DRAM sees long runs instead of one sector per
// row per block. A hint only: issued before the grid-dependency wait (L2 is
// the coherence point), and a share that is not 16-byte aligned is skipped.
template <class E, bool TRUNC>
__device__ __forceinline__ void tm_prefetch(const Params &p, int64_t t0, int64_t t1, int64_t part,
                                            int64_t parts) {
  constexpr uint32_t kUse = E::kSlots | (TRUNC ? E::kOptSlots : 0u);
  const int64_t lo = t0 * p.N * 4, total = (t1 - t0) * p.N * 4;
  const int64_t share = ((total + parts - 1) / parts + 15) & ~int64_t(15);
  const int64_t s0 = part * share;
  int64_t len = total - s0 < share ? total - s0 : share;
  len &= ~int64_t(15);
  if (len <= 0) return;
#pragma unroll
  for (int k = 0; k < kNumSlots; ++k) {
    if (!(kUse & bit(k))) continue;
    const char *a = reinterpret_cast<const char *>(p.in[k]) + lo + s0;
    if ((reinterpret_cast<uintptr_t>(a) & 15u) == 0) prefetch_l2(a, (uint32_t)len);
  }
}

// One warp's span of L steps for its 32 environments. b0 + j*rowb: byte
// offset of step ts+j of this lane's environment; rowb: bytes per row (4N).
// FULL: the span holds neither step 0 nor step T-1 and every lane's
// environment exists, so no step needs a bounds check or an edge flag.
template <int L>
struct TmRaw {
  float v[kNumSlots][L];   // inputs at ts .. ts+L-1
  float next[kNumSlots];   // at ts+L (backward estimators' successor values)
  float prev_d;            // done mask at ts-1 (forward estimators)
};

// Issue every load of the span (nothing here waits for one).
template <class E, bool TRUNC, bool FULL, int L>
__device__ __forceinline__ void tm_load(const Params &p, int64_t b0, int64_t rowb,
                                        int64_t ts, int64_t T, bool env_ok, TmRaw<L> &raw) {
  constexpr uint32_t kUse = E::kSlots | (TRUNC ? E::kOptSlots : 0u);
#pragma unroll
  for (int k = 0; k < kNumSlots; ++k) {
#pragma unroll
    for (int j = 0; j < L; ++j) {
      const bool ok = FULL || (env_ok && ts + j < T);
      raw.v[k][j] = ((kUse & bit(k)) && ok) ? ldg_at(p.in[k], b0 + j * rowb) : 0.f;
    }
  }
  // a span wholly past T (last chunk) reads neither neighbour
  const bool next_ok = FULL || (env_ok && ts + L < T);
#pragma unroll
  for (int k = 0; k < kNumSlots; ++k)
    raw.next[k] = (E::kBackward && (E::kNext & bit(k)) && next_ok)
                      ? ldg_at(p.in[k], b0 + L * rowb)
                      : 0.f;
  const bool prev_ok = FULL || (env_ok && ts > 0 && ts <= T);
  raw.prev_d = (E::kPrevD && prev_ok) ? ldg_at(p.in[kD], b0 - rowb) : 0.f;
}

// Build every step's pair; steps past T become the identity (never stored).
template <class E, bool TRUNC, bool FULL, int L>
__device__ __forceinline__ void tm_build(const Params &p, const TmRaw<L> &raw, int64_t ts,
                                         int64_t T, float boot, typename E::Pair (&e)[L],
                                         float (&aux0)[L], float (&aux1)[L]) {
  using P = typename E::Pair;
#pragma unroll
  for (int j = 0; j < L; ++j) {
    StepIn st;
    st.r = raw.v[kR][j];
    st.v = raw.v[kV][j];
    st.q = raw.v[kQ][j];
    st.lr = raw.v[kLR][j];
    st.d = raw.v[kD][j];
    st.tau = raw.v[kTau][j];
    st.nv = raw.v[kNV][j];
    st.vn = (j + 1 < L) ? raw.v[kV][j + 1] : raw.next[kV];
    st.qn = (j + 1 < L) ? raw.v[kQ][j + 1] : raw.next[kQ];
    st.lrn = (j + 1 < L) ? raw.v[kLR][j + 1] : raw.next[kLR];
    st.dp = (j > 0) ? raw.v[kD][j - 1] : raw.prev_d;
    st.last = FULL ? false : (ts + j == T - 1);
    st.first = FULL ? false : (ts + j == 0);
    aux0[j] = aux1[j] = 0.f;
    E::template coeff<TRUNC>(p, st, boot, e[j], aux0[j], aux1[j]);
    if (!FULL && ts + j >= T) e[j] = identity(P{});
  }
}

// Walk the span from the value adjacent to it on the scan-origin side and
// store every step's output(s).
template <class E, bool FULL, int L>
__device__ __forceinline__ void tm_emit(const Params &p, int64_t b0, int64_t rowb, int64_t ts,
                                        int64_t T, bool env_ok,
                                        typename ValueOf<typename E::Pair>::type nb,
                                        const typename E::Pair (&e)[L], const float (&aux0)[L],
                                        const float (&aux1)[L]) {
  using V = typename ValueOf<typename E::Pair>::type;
  char *out0 = static_cast<char *>(p.out0);
  char *out1 = reinterpret_cast<char *>(p.out1);
#pragma unroll
  for (int jj = 0; jj < L; ++jj) {
    const int j = E::kBackward ? L - 1 - jj : jj;
    const V A = apply(e[j], nb);
    if (FULL || (env_ok && ts + j < T)) {
      if constexpr (std::is_same<V, uint32_t>::value) {
        *reinterpret_cast<uint32_t *>(out0 + b0 + j * rowb) = A;
      } else {
        *reinterpret_cast<float *>(out0 + b0 + j * rowb) = E::out0(A, nb, e[j], aux0[j], aux1[j]);
        if constexpr (E::kOuts > 1) {
          if (out1)
            *reinterpret_cast<float *>(out1 + b0 + j * rowb) = E::out1(A, nb, e[j], aux0[j], aux1[j]);
        }
      }
    }
    nb = A;
  }
}

template <class E, bool TRUNC, int L>
__global__ void __launch_bounds__(tm_threads<L>(), tm_min_blocks<E, TRUNC, L>())
    time_major_kernel(Params p, TmShape sh) {
  static_assert((E::kBF16Slots | E::kU8Slots) == 0u, "time-major slots are 4-byte words");
  static_assert(kTmChunk % L == 0 && kTmChunk / L <= 32, "whole warps per chunk");
  using P = typename E::Pair;
  using V = typename ValueOf<P>::type;
  constexpr int kWarps = kTmChunk / L;
  __shared__ P s_agg[kWarps][kTmEnvs];
  __shared__ V s_in[kWarps][kTmEnvs];
  __shared__ TmSlices<P, V, kWarps> s_sl;
  __shared__ uint32_t s_epoch;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t N = p.N, T = p.T;
  const int64_t q = div_nonneg((int64_t)blockIdx.x, sh.groups);  // chunk position in scan order
  const int64_t g = (int64_t)blockIdx.x - q * sh.groups;
  const int64_t chunk = E::kBackward ? sh.chunks - 1 - q : q;
  const int64_t n = g * kTmEnvs + lane;
  const bool env_ok = n < N;
  const int64_t ts = chunk * kTmChunk + (int64_t)warp * L;  // this warp's first step
  const bool chained = sh.chunks > 1;
  // uniform across the warp: an interior span of a full group of environments
  const bool full = ts > 0 && ts + L < T && (g + 1) * kTmEnvs <= N;
  const int64_t rowb = N * 4;
  const int64_t b0 = (ts * N + n) * 4;  // byte offset of step ts of this lane's environment

  // The chunk's rows into L2 for calls that move four arrays or more
  // (measured on GB300, prefetch against none: GAE 1024 x 4096 16.7 / 17.8 us,
  // 4096 x 512 14.5 / 15.8, V-trace 4096 x 512 17.2 / 19.3); the three-array
  // calls ran slower with it (discounted returns 4096 x 512 13.8 / 9.9,
  // 1024 x 16384 60.4 / 50.6, 1024 x 4096 16.8 / 15.5), so they skip it.
  if constexpr (!three_arrays<E, TRUNC>()) {
    if (threadIdx.x == 0) {
      const int64_t c0 = chunk * kTmChunk, c1 = c0 + kTmChunk < T ? c0 + kTmChunk : T;
      tm_prefetch<E, TRUNC>(p, c0, c1, g, sh.groups);
    }
  }
  pdl_wait();
  TmRaw<L> raw;
  if (full)
    tm_load<E, TRUNC, true, L>(p, b0, rowb, ts, T, env_ok, raw);
  else
    tm_load<E, TRUNC, false, L>(p, b0, rowb, ts, T, env_ok, raw);
  const float boot = (E::kUsesRowValue && p.boot && env_ok) ? __ldg(p.boot + n) : 0.f;
  if (chained && threadIdx.x == 0) s_epoch = ld_relaxed_gpu(&sh.ws->epoch);
  // Besides letting the next grid launch, this instruction keeps the
  // compiler from sinking the loads above into the arithmetic below: every
  // load of the span is in flight before the first one is waited on.
  pdl_launch_dependents();
  P e[L];
  float aux0[L], aux1[L];
  if (full)
    tm_build<E, TRUNC, true, L>(p, raw, ts, T, boot, e, aux0, aux1);
  else
    tm_build<E, TRUNC, false, L>(p, raw, ts, T, boot, e, aux0, aux1);

  P agg = identity(P{});
  if (E::kBackward) {
#pragma unroll
    for (int j = L - 1; j >= 0; --j) agg = compose(e[j], agg);
  } else {
#pragma unroll
    for (int j = 0; j < L; ++j) agg = compose(e[j], agg);
  }
  if constexpr (E::kConstBeta) agg.m = span_multiplier<L>(e, const_beta_power<L>(p));
  s_agg[warp][lane] = agg;
  __syncthreads();

  // the chunk's pair (warp 0): warps in order outer-first from the scan origin side
  P cagg = identity(P{});
  if (warp == 0) {
    if (E::kBackward) {
      for (int w = kWarps - 1; w >= 0; --w) cagg = compose(s_agg[w][lane], cagg);
    } else {
      for (int w = 0; w < kWarps; ++w) cagg = compose(s_agg[w][lane], cagg);
    }
  }
  V X = V(0);
  if (chained)  // uniform over the block: every thread takes part
    // one distance per warp and round (measured on GB300 against a serial walk
    // of the same window by warp 0: 256 x 16384 GAE 20.8 against 23.3 us,
    // V-trace 28.9 against 30.8, discounted returns 18.7 against 21.1; two
    // or four distances per warp were slower)
    X = tm_lookback<P, V, 1, kWarps>(sh.ws, (q * sh.groups + g) * kTmEnvs, sh.groups * kTmEnvs, q,
                                     cagg, s_epoch & kTagMask, lane, warp, env_ok, 1, s_sl);
  if (warp == 0) {
    if (E::kBackward) {
      for (int w = kWarps - 1; w >= 0; --w) {
        s_in[w][lane] = X;
        X = apply(s_agg[w][lane], X);
      }
    } else {
      for (int w = 0; w < kWarps; ++w) {
        s_in[w][lane] = X;
        X = apply(s_agg[w][lane], X);
      }
    }
  }
  __syncthreads();

  const V nb = s_in[warp][lane];  // value adjacent to this warp's span, scan-origin side
  if (full)
    tm_emit<E, true, L>(p, b0, rowb, ts, T, env_ok, nb, e, aux0, aux1);
  else
    tm_emit<E, false, L>(p, b0, rowb, ts, T, env_ok, nb, e, aux0, aux1);
  if (chained && threadIdx.x == 0) finish_launch(sh.ws, sh.groups * sh.chunks, s_epoch);
}

// Time-major rows of few environment groups: 8 environments per block over
// a 512- or 1024-step chunk, so an environment's chain has a quarter or an
// eighth of the links of the 128-step chunks. Lane l of warp w owns
// environment 8*g + (l % 8) and the 16 steps 64*w + 16*(l / 8) .. +15 of the
// chunk; lanes 0..7 read the 8 environments' words at one step, so every
// access moves whole 32-byte sectors. A warp composes its four runs per
// environment with two shuffle rounds, the warps meet in shared memory, and
// warp 0 runs the look-back for the 8 environments (lanes 0..7).
constexpr int kTmNarrowEnvs = 8;
constexpr int kTmNarrowL = 16;                // steps per lane
// Warps per block: 8 (512-step chunks), or 16 (1024-step chunks, half the
// chain links) when the grid fits in one block per SM, where fewer links
// matter more than resident blocks.
template <int W, int L>
constexpr int tm_narrow_chunk() {
  return W * 4 * L;
}
// The 8-environment kernel: the 8-warp shape takes the budgets above; the
// 16-warp shape (grids of at most one block per SM) takes one block.
template <class E, bool TRUNC, int W, int L>
constexpr int tm_narrow_min_blocks() {
  return W >= 16 ? 1 : tm_min_blocks<E, TRUNC, L>();
}

template <class E, bool TRUNC, int W, int L>
__global__ void __launch_bounds__(W * 32, tm_narrow_min_blocks<E, TRUNC, W, L>())
    time_major_narrow_kernel(Params p, TmShape sh) {
  static_assert((E::kBF16Slots | E::kU8Slots) == 0u, "time-major slots are 4-byte words");
  using P = typename E::Pair;
  using V = typename ValueOf<P>::type;
  constexpr int kWarps = W, kE = kTmNarrowEnvs;
  __shared__ P s_agg[kWarps][kE];
  __shared__ V s_in[kWarps][kE];
  __shared__ TmSlices<P, V, kWarps> s_sl;
  __shared__ uint32_t s_epoch;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ev = lane & (kE - 1), run = lane >> 3;  // environment in the block, run in the warp
  const int64_t N = p.N, T = p.T;
  const int64_t q = div_nonneg((int64_t)blockIdx.x, sh.groups);  // chunk position in scan order
  const int64_t g = (int64_t)blockIdx.x - q * sh.groups;
  const int64_t chunk = E::kBackward ? sh.chunks - 1 - q : q;
  const int64_t n = g * kE + ev;
  const bool env_ok = n < N;
  const int64_t tw = chunk * tm_narrow_chunk<W, L>() + (int64_t)warp * 4 * L;  // the warp's first step
  const int64_t ts = tw + (int64_t)run * L;                            // this lane's first step
  const bool chained = sh.chunks > 1;
  // uniform across the warp: all four runs interior and the group full
  const bool full = tw > 0 && tw + 4 * L < T && (g + 1) * kE <= N;
  const int64_t rowb = N * 4;
  const int64_t b0 = (ts * N + n) * 4;  // byte offset of step ts of this lane's environment

  // the chunk's rows into L2 (measured on GB300, prefetch against none:
  // GAE 8 x 131072 10.3 / 11.2 us, 64 x 16384 7.2 / 8.3, 256 x 4096 6.6 /
  // 7.6; discounted returns 8 x 131072 9.4 / 10.3; 256 x 16384 unchanged)
  if (threadIdx.x == 0) {
    const int64_t c0 = chunk * tm_narrow_chunk<W, L>();
    const int64_t c1 = c0 + tm_narrow_chunk<W, L>() < T ? c0 + tm_narrow_chunk<W, L>() : T;
    tm_prefetch<E, TRUNC>(p, c0, c1, g, sh.groups);
  }
  pdl_wait();
  TmRaw<L> raw;
  if (full)
    tm_load<E, TRUNC, true, L>(p, b0, rowb, ts, T, env_ok, raw);
  else
    tm_load<E, TRUNC, false, L>(p, b0, rowb, ts, T, env_ok, raw);
  const float boot = (E::kUsesRowValue && p.boot && env_ok) ? __ldg(p.boot + n) : 0.f;
  if (chained && threadIdx.x == 0) s_epoch = ld_relaxed_gpu(&sh.ws->epoch);
  pdl_launch_dependents();  // also keeps the loads above ahead of the arithmetic
  P e[L];
  float aux0[L], aux1[L];
  if (full)
    tm_build<E, TRUNC, true, L>(p, raw, ts, T, boot, e, aux0, aux1);
  else
    tm_build<E, TRUNC, false, L>(p, raw, ts, T, boot, e, aux0, aux1);

  P agg = identity(P{});
  if (E::kBackward) {
#pragma unroll
    for (int j = L - 1; j >= 0; --j) agg = compose(e[j], agg);
  } else {
#pragma unroll
    for (int j = 0; j < L; ++j) agg = compose(e[j], agg);
  }
  if constexpr (E::kConstBeta) agg.m = span_multiplier<L>(e, const_beta_power<L>(p));
  // the warp's four runs of each environment (lanes ev, ev+8, ev+16, ev+24)
  P inc = agg, excl, wagg;
  if (E::kBackward) {
#pragma unroll
    for (int off = 8; off < 32; off <<= 1) {
      const P o = shfl_down(inc, off);
      if (lane + off < 32) inc = compose(inc, o);
    }
    wagg = shfl_idx(inc, ev);
    const P x = shfl_down(inc, 8);
    excl = (run == 3) ? identity(P{}) : x;
  } else {
#pragma unroll
    for (int off = 8; off < 32; off <<= 1) {
      const P o = shfl_up(inc, off);
      if (lane >= off) inc = compose(inc, o);
    }
    wagg = shfl_idx(inc, 24 + ev);
    const P x = shfl_up(inc, 8);
    excl = (run == 0) ? identity(P{}) : x;
  }
  if (run == 0) s_agg[warp][ev] = wagg;
  __syncthreads();

  // the chunk's pair (warp 0, lanes 0..7): warps outer-first from the scan origin side
  P cagg = identity(P{});
  if (warp == 0 && lane < kE) {
    if (E::kBackward) {
      for (int w = kWarps - 1; w >= 0; --w) cagg = compose(s_agg[w][lane], cagg);
    } else {
      for (int w = 0; w < kWarps; ++w) cagg = compose(s_agg[w][lane], cagg);
    }
  }
  V X = V(0);
  if (chained)  // uniform over the block: every thread takes part
    X = tm_lookback<P, V, 32 / kE, kWarps>(sh.ws, (q * sh.groups + g) * kE, sh.groups * kE, q,
                                           cagg, s_epoch & kTagMask, lane, warp, env_ok,
                                           sh.slots, s_sl);
  if (warp == 0 && lane < kE) {
    if (E::kBackward) {
      for (int w = kWarps - 1; w >= 0; --w) {
        s_in[w][lane] = X;
        X = apply(s_agg[w][lane], X);
      }
    } else {
      for (int w = 0; w < kWarps; ++w) {
        s_in[w][lane] = X;
        X = apply(s_agg[w][lane], X);
      }
    }
  }
  __syncthreads();

  const V nb = apply(excl, s_in[warp][ev]);  // value adjacent to this lane's run, origin side
  if (full)
    tm_emit<E, true, L>(p, b0, rowb, ts, T, env_ok, nb, e, aux0, aux1);
  else
    tm_emit<E, false, L>(p, b0, rowb, ts, T, env_ok, nb, e, aux0, aux1);
  if (chained && threadIdx.x == 0) finish_launch(sh.ws, sh.groups * sh.chunks, s_epoch);
}

// Short time-major rows (T <= 128): one chunk, no look-back, and 16
// environments per block so that the grid has twice the blocks of the
// 32-environment shape. Lane l of warp w owns environment 16*g + (l % 16)
// and the 8 steps 16*w + 8*(l / 16) .. +7; the two halves of a warp combine
// with one shuffle, the 8 warps of the block in shared memory. Each warp
// access reads two 64-byte row segments.
constexpr int kTmShortEnvs = 16;
constexpr int kTmShortWarps = 8;
constexpr int kTmShortSteps = 8;  // per lane
constexpr int kTmShortT = kTmShortWarps * 2 * kTmShortSteps;  // 128

template <class E, bool TRUNC>
__global__ void __launch_bounds__(kTmShortWarps * 32) time_major_short_kernel(Params p) {
  static_assert((E::kBF16Slots | E::kU8Slots) == 0u, "time-major slots are 4-byte words");
  using P = typename E::Pair;
  using V = typename ValueOf<P>::type;
  constexpr int L = kTmShortSteps;
  __shared__ P s_agg[kTmShortWarps][kTmShortEnvs];
  __shared__ V s_in[kTmShortWarps][kTmShortEnvs];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int el = lane % kTmShortEnvs, half = lane / kTmShortEnvs;
  const int64_t N = p.N, T = p.T;
  const int64_t g = blockIdx.x;
  const int64_t n = g * kTmShortEnvs + el;
  const bool env_ok = n < N;
  const int64_t ts = (int64_t)warp * 2 * L + half * L;  // this lane's first step
  const bool full = ts > 0 && ts + L < T && (g + 1) * kTmShortEnvs <= N;
  const int64_t rowb = N * 4;
  const int64_t b0 = (ts * N + n) * 4;  // byte offset of step ts of this lane's environment

  // all T rows into L2, a share per block (measured on GB300 at 4096 x 128:
  // GAE 2.67 against 3.31 us without, V-trace 3.86 / 4.61, discounted
  // returns 2.74 / 3.27)
  if (threadIdx.x == 0) tm_prefetch<E, TRUNC>(p, 0, T, g, (int64_t)gridDim.x);
  pdl_wait();
  TmRaw<L> raw;
  if (full)
    tm_load<E, TRUNC, true, L>(p, b0, rowb, ts, T, env_ok, raw);
  else
    tm_load<E, TRUNC, false, L>(p, b0, rowb, ts, T, env_ok, raw);
  const float boot = (E::kUsesRowValue && p.boot && env_ok) ? __ldg(p.boot + n) : 0.f;
  pdl_launch_dependents();  // also keeps the loads above ahead of the arithmetic
  P e[L];
  float aux0[L], aux1[L];
  if (full)
    tm_build<E, TRUNC, true, L>(p, raw, ts, T, boot, e, aux0, aux1);
  else
    tm_build<E, TRUNC, false, L>(p, raw, ts, T, boot, e, aux0, aux1);

  P agg = identity(P{});
  if (E::kBackward) {
#pragma unroll
    for (int j = L - 1; j >= 0; --j) agg = compose(e[j], agg);
  } else {
#pragma unroll
    for (int j = 0; j < L; ++j) agg = compose(e[j], agg);
  }
  if constexpr (E::kConstBeta) agg.m = span_multiplier<L>(e, const_beta_power<L>(p));
  // the other half of the warp (same environment, the neighbouring 8 steps)
  P other;
  other.m = __shfl_xor_sync(kFull, agg.m, kTmShortEnvs);
  other.c = __shfl_xor_sync(kFull, agg.c, kTmShortEnvs);
  // warp pair: outer = the half nearer the scan origin
  const P first = half == 0 ? agg : other, second = half == 0 ? other : agg;
  const P wagg = E::kBackward ? compose(first, second) : compose(second, first);
  if (half == 0) s_agg[warp][el] = wagg;
  __syncthreads();

  if (warp == 0 && half == 0) {
    V X = V(0);  // one chunk: nothing outside it
    if (E::kBackward) {
      for (int w = kTmShortWarps - 1; w >= 0; --w) {
        s_in[w][el] = X;
        X = apply(s_agg[w][el], X);
      }
    } else {
      for (int w = 0; w < kTmShortWarps; ++w) {
        s_in[w][el] = X;
        X = apply(s_agg[w][el], X);
      }
    }
  }
  __syncthreads();

  // value adjacent to this lane's 8 steps on the scan-origin side
  const V Xw = s_in[warp][el];
  const bool outer = E::kBackward ? (half == 1) : (half == 0);  // nearer the origin
  const V nb = outer ? Xw : apply(other, Xw);
  if (full)
    tm_emit<E, true, L>(p, b0, rowb, ts, T, env_ok, nb, e, aux0, aux1);
  else
    tm_emit<E, false, L>(p, b0, rowb, ts, T, env_ok, nb, e, aux0, aux1);
}

}  // namespace rlcs
