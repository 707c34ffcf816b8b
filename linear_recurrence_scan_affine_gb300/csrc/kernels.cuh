// The two launch shapes of the scan, templated on an estimator functor.
//
// Data layout on chip ("strip-major"): a warp walks its span of a row in
// strips of 128 steps; in strip j lane l owns the four consecutive steps
// 128*j + 4*l .. +3, so each warp-wide float4 access covers 512 contiguous
// bytes. Per strip: each lane composes its four pairs (lane-serial
// sub-scan), a 5-round shuffle scan composes the lanes, and the strips of a
// warp are chained by their totals.
//
//  * warp_row_kernel    one warp per row (T <= 128*S): inputs go straight
//                       to registers with 128-bit loads; no shared memory.
//  * block_chunk_kernel one 256-thread block per row chunk of 1024*S steps:
//                       the chunk's inputs are staged into shared memory by
//                       cp.async.bulk (1-D TMA) completing on an mbarrier;
//                       warp aggregates are composed in shared memory; the
//                       chunks of one row are chained in a single pass by
//                       decoupled look-back through the workspace
//                       (ticket-ordered chunks, epoch-tagged flags, bounded
//                       waits).
#pragma once

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

// One environment's column of a time-major tile in shared memory (one strip).
struct ColumnSource {
  const float *col[kNumSlots];  // per slot: this warp's column, 128 steps
  float halo_next[kNumSlots];   // first step after the tile (scan order)
  float halo_prev_d;            // done mask before the tile
  int lane;
  __device__ __forceinline__ float4 get(int k, int) const {
    return *reinterpret_cast<const float4 *>(col[k] + 4 * lane);
  }
  __device__ __forceinline__ float following(int k, int) const { return halo_next[k]; }
  __device__ __forceinline__ float preceding_d(int) const { return halo_prev_d; }
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
      const P a = lane_aggregate(el[j], E::kBackward);
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
template <class E, bool TRUNC, int S>
__global__ void __launch_bounds__(kRowWarps * 32) warp_row_kernel(Params p) {
  using St = Strips<E, TRUNC, S>;
  using V = typename St::V;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5);
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
template <class P, class V>
__device__ V lookback(WsHeader *ws, int64_t self, int64_t stride, int64_t npred, P agg,
                      uint32_t tag, int lane) {
  WsRecord *rec = reinterpret_cast<WsRecord *>(ws + 1);
  const uint32_t tagA = (tag << 2) | kStateAgg, tagP = (tag << 2) | kStateInc;
  if (npred == 0) {  // the row's scan origin: nothing before it
    if (lane == 0) st_relaxed_gpu_u64(&rec[self].inc, tagged(tagP, vbits(apply(agg, V(0)))));
    return V(0);
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
    const int64_t g = blockIdx.x, grow = g / Q, gk = g - grow * Q;
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
      const int64_t row = ticket / Q, kk = ticket - row * Q;
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
  const int64_t row = ticket / Q, kk = ticket - row * Q;
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
  int64_t total_tiles;    // N * Q = grid size
};

// Resident blocks per SM the compiler must allow (measured on GB300):
// 4096-step tiles keep more state per thread and are used when the whole
// grid fits in about one wave (2 per SM); 2048-step tiles are capped at 64
// registers (4 per SM) and 1024-step tiles at 40 (6 per SM), so one block's
// look-back overlaps the others' loads.
template <int S> struct TileMinBlocks { static constexpr int value = S >= 4 ? 2 : (S == 2 ? 4 : 6); };

template <class E, bool TRUNC, int S>
__global__ void __launch_bounds__(kChunkThreads, TileMinBlocks<S>::value)
    block_tile_kernel(Params p, TileShape ts) {
  using St = Strips<E, TRUNC, S>;
  using P = typename St::P;
  using V = typename St::V;
  constexpr int C = kChunkWarps * kStrip * S;  // steps per tile
  constexpr uint32_t kUse = St::kUse;

  __shared__ P s_warp[kChunkWarps];
  __shared__ V s_carry[kChunkWarps];
  __shared__ uint32_t s_epoch;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool vec = p.vec != 0;
  const int64_t N = p.N, T = p.T, Q = ts.tiles_per_row;
  const int64_t b = blockIdx.x;
  const int64_t r = b / N, row = b - r * N;
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
  const float halo_d = (E::kPrevD && t_span > 0) ? load_slot1<E>(p, kD, base + t_span - 1) : 0.f;
  const float boot = (E::kUsesRowValue && p.boot) ? __ldg(p.boot + row) : 0.f;
  if (tid == 0 && Q > 1) s_epoch = ld_relaxed_gpu(&ts.ws->epoch);  // after the loads issue
  pdl_launch_dependents();

  const RegSource<S> src{raw, halo, halo_d, lane};
  St st;
  st.template build<true>(p, src, boot, t_span, T, lane);
  const P wagg = st.scan(lane);
  if (lane == 0) s_warp[warp] = wagg;
  __syncthreads();

  if (warp == 0) {
    const P w = (lane < kChunkWarps) ? s_warp[lane] : identity(P{});
    P inc, nb, tile_agg;
    if (E::kBackward) {
      inc = warp_suffix_scan(w, lane);
      tile_agg = shfl_idx(inc, 0);
      const P x = shfl_down(inc, 1);
      nb = (lane >= kChunkWarps - 1) ? identity(P{}) : x;
    } else {
      inc = warp_prefix_scan(w, lane);
      tile_agg = shfl_idx(inc, kChunkWarps - 1);
      const P x = shfl_up(inc, 1);
      nb = (lane == 0) ? identity(P{}) : x;
    }
    V X = V(0);
    if (Q > 1) {
      const uint32_t epoch = s_epoch;
      X = lookback<P, V>(ts.ws, b, N, r, tile_agg, epoch & kTagMask, lane);
    }
    if (lane < kChunkWarps) s_carry[lane] = apply(nb, X);
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

// ---------------------------------------------------------------------------
// Time-major tier: inputs and outputs [T, N] (element (t, n) at t*N + n).
// A block owns kTmEnvs environments (kTmEnvsPerWarp per warp) and walks T in tiles of
// kStrip steps, in scan order, carrying each environment's value from tile
// to tile: no look-back. Per tile, rows are loaded with coalesced accesses
// (kTmEnvs consecutive environments per row) into an env-major shared tile
// padded to kTmPitch floats, so the row writes and each warp's float4 reads
// of its environment's column are both bank-conflict-free; the warp then runs
// the strip engine on its column (lane l owns steps 4l..4l+3, exactly as in
// the warp-row tier), writes its outputs into an output tile of the same
// layout, and the block stores those rows coalesced.
// ---------------------------------------------------------------------------
#ifndef RLCS_TM_ENVS_PER_WARP
#define RLCS_TM_ENVS_PER_WARP 1
#endif
constexpr int kTmWarps = 8;
constexpr int kTmEnvsPerWarp = RLCS_TM_ENVS_PER_WARP;  // columns each warp scans, in turn
constexpr int kTmEnvs = kTmWarps * kTmEnvsPerWarp;     // environments per block
constexpr int kTmThreads = kTmWarps * 32;
constexpr int kTmPitch = kStrip + 4;                   // floats per environment column
constexpr int kTmRowsPerLoad = 32 / kTmEnvs;           // rows one warp instruction covers
constexpr int kTmRowsPerPass = kTmWarps * kTmRowsPerLoad;
constexpr int kTmPasses = kStrip / kTmRowsPerPass;
static_assert(kTmEnvs <= 32 && 32 % kTmEnvs == 0, "a warp covers whole row segments");

template <class E, bool TRUNC>
constexpr int tm_tiles() {  // shared tiles: used input slots + outputs
  return __builtin_popcount(Strips<E, TRUNC, 1>::kUse) + E::kOuts;
}

template <class E, bool TRUNC>
__global__ void __launch_bounds__(kTmThreads) time_major_kernel(Params p) {
  using St = Strips<E, TRUNC, 1>;
  using V = typename St::V;
  constexpr uint32_t kUse = St::kUse;
  constexpr int kNumUsed = __builtin_popcount(kUse);
  extern __shared__ __align__(16) float tm_smem[];  // [kNumUsed + kOuts][kTmEnvs][kTmPitch]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t N = p.N, T = p.T;
  const int64_t env0 = (int64_t)blockIdx.x * kTmEnvs;
  // loader mapping: one warp instruction = kTmRowsPerLoad rows x kTmEnvs environments
  const int ld_env = lane % kTmEnvs, ld_row = lane / kTmEnvs;
  const bool ld_ok = env0 + ld_env < N;
  const int64_t tiles = (T + kStrip - 1) / kStrip;

  auto tile_of = [&](int idx) { return tm_smem + (size_t)idx * kTmEnvs * kTmPitch; };

  pdl_wait();
  V carry[kTmEnvsPerWarp];
  float boot[kTmEnvsPerWarp];
  float halo_next[kTmEnvsPerWarp][kNumSlots];
  float halo_prev_d[kTmEnvsPerWarp];
#pragma unroll
  for (int q = 0; q < kTmEnvsPerWarp; ++q) {
    const int64_t env = env0 + warp * kTmEnvsPerWarp + q;
    boot[q] = (E::kUsesRowValue && p.boot && env < N) ? __ldg(p.boot + env) : 0.f;
    carry[q] = V(0);
    halo_prev_d[q] = 0.f;
#pragma unroll
    for (int k = 0; k < kNumSlots; ++k) halo_next[q][k] = 0.f;
  }

  for (int64_t i = 0; i < tiles; ++i) {
    const int64_t tt = E::kBackward ? (tiles - 1 - i) : i;
    const int64_t t0 = tt * kStrip;
    __syncthreads();  // the previous tile's shared reads are done
    // coalesced row loads into the env-major tiles
    {
      int idx = 0;
#pragma unroll
      for (int k = 0; k < kNumSlots; ++k) {
        if (!(kUse & bit(k))) continue;
        float *tile = tile_of(idx);
        float v[kTmPasses];
#pragma unroll
        for (int q = 0; q < kTmPasses; ++q) {
          const int r = q * kTmRowsPerPass + warp * kTmRowsPerLoad + ld_row;
          const int64_t t = t0 + r;
          v[q] = (t < T && ld_ok) ? load_slot1<E>(p, k, t * N + env0 + ld_env) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kTmPasses; ++q) {
          const int r = q * kTmRowsPerPass + warp * kTmRowsPerLoad + ld_row;
          tile[ld_env * kTmPitch + r] = v[q];
        }
        ++idx;
      }
    }
    if (i == 0) pdl_launch_dependents();
    __syncthreads();

#pragma unroll 1
    for (int q = 0; q < kTmEnvsPerWarp; ++q) {
      const int e = warp * kTmEnvsPerWarp + q;  // this warp's column
      ColumnSource src;
      {
        int idx = 0;
#pragma unroll
        for (int k = 0; k < kNumSlots; ++k) {
          src.col[k] = tile_of(idx) + e * kTmPitch;  // unused slots alias a used one
          if (kUse & bit(k)) ++idx;
        }
      }
#pragma unroll
      for (int k = 0; k < kNumSlots; ++k) src.halo_next[k] = halo_next[q][k];
      src.halo_prev_d = halo_prev_d[q];
      src.lane = lane;
      St st;
      st.template build<true>(p, src, boot[q], t0, T, lane);
      const auto agg = st.scan(lane);
      float4 o0[1], o1[1];
      st.finish(carry[q], o0, o1);
      carry[q] = apply(agg, carry[q]);
      // values just outside the next tile in scan order
#pragma unroll
      for (int k = 0; k < kNumSlots; ++k)
        if (E::kBackward && (E::kNext & bit(k))) halo_next[q][k] = src.col[k][0];
      if (E::kPrevD) halo_prev_d[q] = src.col[kD][kStrip - 1];
      *reinterpret_cast<float4 *>(tile_of(kNumUsed) + e * kTmPitch + 4 * lane) = o0[0];
      if constexpr (E::kOuts > 1)
        *reinterpret_cast<float4 *>(tile_of(kNumUsed + 1) + e * kTmPitch + 4 * lane) = o1[0];
    }
    __syncthreads();

    // coalesced row stores
#pragma unroll
    for (int o = 0; o < E::kOuts; ++o) {
      float *dst = (o == 0) ? static_cast<float *>(p.out0) : p.out1;
      if (dst == nullptr) continue;
      const float *tile = tile_of(kNumUsed + o);
#pragma unroll
      for (int q = 0; q < kTmPasses; ++q) {
        const int r = q * kTmRowsPerPass + warp * kTmRowsPerLoad + ld_row;
        const int64_t t = t0 + r;
        if (t < T && ld_ok) dst[t * N + env0 + ld_env] = tile[ld_env * kTmPitch + r];
      }
    }
  }
}

}  // namespace rlcs
