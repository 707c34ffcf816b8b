// C ABI entry points: argument validation, launch-shape planning and the
// workspace/status helpers declared in include/rlcs.h, and the test and
// tuning hooks declared in include/rlcs_internal.h.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "launch.cuh"

namespace rlcs {
namespace {

constexpr int64_t kRowMaxT = 512;       // warp-row shape: T <= 4 strips
constexpr int64_t kMinChunk = 1024;     // smallest block chunk (S = 1)
constexpr int kMaxDevices = 64;

std::atomic<int> g_override_shape{RLCS_SHAPE_AUTO};
std::atomic<int64_t> g_override_chunk{0};
std::atomic<int> g_sm_count[kMaxDevices];

// Set while a time-major (_tm) entry point runs its row-major counterpart's
// validation and launch; run() reads it. Thread-local, so concurrent callers
// on other threads are unaffected.
thread_local bool t_time_major = false;
struct TimeMajorScope {
  TimeMajorScope() { t_time_major = true; }
  ~TimeMajorScope() { t_time_major = false; }
};

struct Buf {
  const void *p;
  size_t bytes;
};
bool overlaps(const Buf &a, const Buf &b) {
  if (!a.p || !b.p) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Set while rlcs_run_group passes its calls through their namesake entry
// points: run() validates each call as usual, then records it here instead
// of launching it.
struct GroupEntry {
  Params p;
  int kind;
  int S;         // strips per warp (short rows) or tile length / 1024 (long rows)
  bool trunc;
  bool long_row;  // T > kRowMaxT: block tiles, planned with the whole group
  Buf reads[kNumSlots + 1];  // input planes and the bootstrap array
  Buf writes[2];
};
struct GroupCollect {
  int n = 0;
  GroupEntry e[kMaxGroup];
};
thread_local GroupCollect *t_group = nullptr;

int group_kind(cudaError_t (*launch)(const Params &, const Plan &, WsHeader *, cudaStream_t)) {
  if (launch == launch_gae) return kGroupGae;
  if (launch == launch_lambda_returns) return kGroupLambdaReturns;
  if (launch == launch_discounted_returns) return kGroupDiscountedReturns;
  if (launch == launch_vtrace) return kGroupVTrace;
  if (launch == launch_retrace) return kGroupRetrace;
  if (launch == launch_eligibility_traces) return kGroupEligibilityTraces;
  if (launch == launch_episodic_prefix_sum) return kGroupEpisodicPrefixSum;
  if (launch == launch_gae_and_returns) return kGroupGaeAndReturns;
  return -1;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
  int v = g_sm_count[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 152;
    g_sm_count[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Tile/chunk length for rows longer than the warp-row limit (measured on
// GB300): the shortest tile that holds a whole row up to 4096 steps, so such
// rows need no look-back; for longer rows 4096 steps while the grid fits in
// about one wave of two blocks per SM, where fewer and larger tiles shorten
// the chain of look-backs, and 2048 steps for larger grids, where more
// resident blocks overlap better (256 x 8192: 2048-step tiles 1-7% faster).
int64_t pick_chunk(int64_t N, int64_t T) {
  if (T <= 1024) return 1024;
  if (T <= 2048) return 2048;
  if (T <= 4096 || N * ceil_div(T, 4096) <= 2 * (int64_t)sm_count()) return 4096;
  return 2048;
}

// Tile length of a long-row call in a group: the single-call rule applied
// to the rows of all the group's long calls together (they share the GPU in
// one grid), unless a block-tile override names one.
int64_t group_chunk(int64_t rows, int64_t T) {
  const int ov = g_override_shape.load(std::memory_order_relaxed);
  const int64_t forced = g_override_chunk.load(std::memory_order_relaxed);
  if (ov == RLCS_SHAPE_BLOCK_TILE && forced != 0) return forced;
  return pick_chunk(rows, T);
}

// Look-back records a group's long calls need: sum over calls whose rows
// span several tiles of N * tiles per row. `Ns`, `Ts`: the long calls only.
int64_t group_records(const int64_t *Ns, const int64_t *Ts, int n) {
  int64_t rows = 0, recs = 0;
  for (int i = 0; i < n; ++i) rows += Ns[i];
  for (int i = 0; i < n; ++i) {
    const int64_t Q = ceil_div(Ts[i], group_chunk(rows, Ts[i]));
    if (Q > 1) recs += Ns[i] * Q;
  }
  return recs;
}

// Choose the launch shape for an [N, T] call.
rlcs_status plan_call(int64_t N, int64_t T, bool trunc, Plan &plan, bool time_major = false) {
  plan = Plan{};
  plan.trunc = trunc;
  plan.pdl = true;
  if (time_major) {  // a block per 32 environments and kTmChunk steps, or per 8 (few environments)
    plan.shape = kShapeTimeMajor;
    plan.S = 1;
    plan.Q = ceil_div(T, kTmChunk);
    // 8-environment chunks of 16 warps when their grid fits in one block per
    // SM (measured on GB300, GAE: 8 x 131072 11.1 against 14.1 us with 8
    // warps, 64 x 16384 8.2 against 9.7, 256 x 4096 7.6 against 8.2; with a
    // larger grid 256 x 16384 24.4 against 19.5)
    plan.tm_wide = ceil_div(N, kTmNarrowEnvs) * ceil_div(T, tm_narrow_chunk<16, kTmNarrowL>()) <=
                   (int64_t)sm_count();
    return RLCS_OK;
  }
  const int ov = g_override_shape.load(std::memory_order_relaxed);
  if (ov == RLCS_SHAPE_WARP_ROW || (ov == RLCS_SHAPE_AUTO && T <= kRowMaxT)) {
    if (T > kRowMaxT) return RLCS_ERR_INVALID_ARG;
    plan.shape = RLCS_SHAPE_WARP_ROW;
    plan.S = T <= 128 ? 1 : (T <= 256 ? 2 : 4);
    plan.Q = 1;
    return RLCS_OK;
  }
  plan.shape = (ov == RLCS_SHAPE_BLOCK_CHUNK) ? RLCS_SHAPE_BLOCK_CHUNK : RLCS_SHAPE_BLOCK_TILE;
  int64_t chunk = g_override_chunk.load(std::memory_order_relaxed);
  if (ov == RLCS_SHAPE_AUTO || chunk == 0) {
    chunk = pick_chunk(N, T);
    // Single calls whose rows are long and few enough that 8192-step tiles
    // (32 warps of 2 strips) fill at most one block per SM: half the chain
    // links of 4096-step tiles. Measured on GB300 (V-trace / Retrace / GAE,
    // us): 8 x 131072 8.36 / 8.55 / 6.96 against 9.37 / 9.41 / 8.06;
    // 64 x 16384 7.28 / 7.04 / 5.57 against 7.75 / 7.57 / 6.11. (Grouped
    // calls keep 4096 at most.)
    if (ov == RLCS_SHAPE_AUTO && T > 8192 && N * ceil_div(T, 8192) <= (int64_t)sm_count())
      chunk = 8192;
  }
  plan.S = (int)(chunk / kMinChunk);
  plan.Q = ceil_div(T, chunk);
  plan.many_waves = N * plan.Q > 2 * (int64_t)sm_count();
  return RLCS_OK;
}

size_t ws_bytes_for(int64_t N, int64_t Q) {
  return sizeof(WsHeader) + sizeof(WsRecord) * (size_t)N * (size_t)Q;
}

// Time-major records: one per environment (N rounded up to whole 32-lane
// groups) and chunk of kTmChunk steps.
size_t ws_bytes_tm(int64_t N, int64_t T) {
  return ws_bytes_for(ceil_div(N, kTmEnvs) * kTmEnvs, ceil_div(T, kTmChunk));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


// Shared tail of every entry point.
// `opt`: the estimator's optional inputs are present (the truncation pair,
// or the affine scan's reset mask already placed in p.in).
// `esize`: bytes per element of each input slot (NULL: all float32).
// `time_major`: arrays are [T, N] (element (t, n) at t*N + n).
template <class Launch>
rlcs_status run(Params &p, const float *trunc, const float *next_values, void *const *outs,
                int n_outs, void *ws, size_t ws_bytes, cudaStream_t stream, Launch launch,
                bool opt, const int *esize = nullptr, bool time_major = false) {
  const int64_t N = p.N, T = p.T;
  if (N <= 0 || T <= 0) return RLCS_ERR_INVALID_ARG;
  if (N > (int64_t)(INT64_MAX / 4) / T) return RLCS_ERR_INVALID_ARG;
  if ((trunc == nullptr) != (next_values == nullptr)) return RLCS_ERR_INVALID_ARG;
  p.in[kTau] = trunc;
  p.in[kNV] = next_values;
  const size_t plane = (size_t)N * (size_t)T * 4u;
  bool vec = (T % 4) == 0;
  for (int k = 0; k < kNumSlots; ++k)
    if (p.in[k] && !aligned16(p.in[k])) vec = false;
  for (int o = 0; o < n_outs; ++o) {
    if (!outs[o]) continue;
    if (!aligned16(outs[o])) vec = false;
    const Buf ob{outs[o], plane};
    for (int k = 0; k < kNumSlots; ++k) {
      const size_t in_plane = (size_t)N * (size_t)T * (size_t)(esize ? esize[k] : 4);
      if (overlaps(ob, Buf{p.in[k], in_plane})) return RLCS_ERR_INVALID_ARG;
    }
    if (overlaps(ob, Buf{p.boot, (size_t)N * 4u})) return RLCS_ERR_INVALID_ARG;
    for (int o2 = o + 1; o2 < n_outs; ++o2)
      if (overlaps(ob, Buf{outs[o2], plane})) return RLCS_ERR_INVALID_ARG;
  }
  p.vec = vec ? 1 : 0;

  if (t_group != nullptr) {  // record a grouped call instead of launching it
    const int kind = group_kind(launch);
    if (kind < 0 || time_major || t_time_major || esize != nullptr) return RLCS_ERR_INVALID_ARG;
    if (t_group->n >= kMaxGroup) return RLCS_ERR_INVALID_ARG;
    GroupEntry &g = t_group->e[t_group->n++];
    g.p = p;
    g.kind = kind;
    g.long_row = T > kRowMaxT;
    g.S = g.long_row ? 0 : (T <= 128 ? 1 : (T <= 256 ? 2 : 4));  // long rows: set later
    g.trunc = opt;
    for (int k = 0; k < kNumSlots; ++k) g.reads[k] = Buf{p.in[k], plane};
    g.reads[kNumSlots] = Buf{p.boot, (size_t)N * 4u};
    for (int o = 0; o < 2; ++o) g.writes[o] = Buf{o < n_outs ? outs[o] : nullptr, plane};
    return RLCS_OK;
  }

  Plan plan;
  const rlcs_status st = plan_call(N, T, opt, plan, time_major || t_time_major);
  if (st != RLCS_OK) return st;
  // Light calls in rows of whole 8-step groups take the eight-step tiles
  // unless a shape is forced: compact GAE (the only call with element
  // sizes) and float32 discounted returns without truncation. Measured on
  // GB300 against the four-step shapes, discounted returns: 12.4 against
  // 14.1 us at 256 x 16384, 34.6 against 39.5 at 4096 x 4096, 16.0 against
  // 18.1 at 65536 x 128, 3.58 against 3.73 at 256 x 4096, 2.47 against 2.53
  // at 4096 x 128. Slower there: eligibility traces and the prefix sum
  // (forward; 4096 x 128 2.30 against 2.08 us, 256 x 16384 13.2 against
  // 12.8), GAE, TD(lambda) returns and Retrace in float32 (4096 x 128 2.64
  // against 2.57, 256 x 16384 14.7 against 14.3 for GAE).
  // The tile length follows the register tiles' rule: 1024 steps (4 warps)
  // for rows up to 1024 steps, measured against 2048 (us, compact GAE /
  // discounted returns): 1024 x 1024 3.28 / 3.37 against 3.46 / 3.51,
  // 16384 x 512 17.0 / 16.7 against 18.0 / 17.4, 4096 x 128 2.44 / 2.36
  // against 2.40 / 2.45, 256 x 1024 2.40 / 2.21 against 2.30 / 2.14.
  const bool eight = esize != nullptr || (!opt && launch == launch_discounted_returns);
  if (eight && p.vec && T % 8 == 0 && !time_major && !t_time_major &&
      g_override_shape.load(std::memory_order_relaxed) == RLCS_SHAPE_AUTO) {
    const int64_t tile = T <= 1024                                            ? 1024
                         : (T > 8192 && N * ceil_div(T, 8192) <= (int64_t)sm_count()) ? 8192
                         : pick_chunk(N, T) >= 4096                                 ? 4096
                                                                                    : 2048;
    plan.shape = kShapeEight;
    plan.S = (int)(tile / kMinChunk);  // 1: 4 warps, 2: 8, 4: 16, 8: 32
    plan.Q = T <= tile ? 1 : ceil_div(T, tile);
    plan.rows_per_tile = T <= tile ? tile / T : 0;
    const int64_t blocks = plan.Q > 1 ? N * plan.Q : ceil_div(N, plan.rows_per_tile);
    // one wave: 8 blocks of 4 warps, 4 of 8, 2 of 16 or 1 of 32 per SM
    plan.many_waves =
        blocks > (tile == 8192 ? 1 : tile == 4096 ? 2 : (tile == 2048 ? 4 : 8)) * (int64_t)sm_count();
  }
  WsHeader *wsh = nullptr;
  if (plan.shape != RLCS_SHAPE_WARP_ROW) {
    if (N * plan.Q >= (int64_t)INT32_MAX) return RLCS_ERR_INVALID_ARG;  // grid x limit
    if (plan.Q > 1) {
      const size_t need =
          plan.shape == kShapeTimeMajor ? ws_bytes_tm(N, T) : ws_bytes_for(N, plan.Q);
      if (!ws || ws_bytes < need || !aligned16(ws)) return RLCS_ERR_WORKSPACE;
    }
    if (ws && ws_bytes >= sizeof(WsHeader) && aligned16(ws)) wsh = static_cast<WsHeader *>(ws);
    for (int k = 0; k < kNumSlots; ++k) {
      const size_t in_plane = (size_t)N * (size_t)T * (size_t)(esize ? esize[k] : 4);
      if (overlaps(Buf{ws, ws_bytes}, Buf{p.in[k], in_plane})) return RLCS_ERR_INVALID_ARG;
    }
  }
  const cudaError_t err = launch(p, plan, wsh, stream);
  if (err != cudaSuccess) {
    cudaGetLastError();  // clear the non-sticky launch error
    return RLCS_ERR_CUDA;
  }
  return RLCS_OK;
}

// Powers of beta, the multiplier between cuts of the estimators that have
// one constant multiplier (discounted returns: gamma; GAE, TD(lambda) returns
// and eligibility traces: gamma*lambda), raised in double and rounded once.
void set_beta(Params &p, double beta) {
  const double b4 = (beta * beta) * (beta * beta), b8 = b4 * b4;
  p.beta4 = (float)b4;
  p.beta8 = (float)b8;
  p.beta16 = (float)(b8 * b8);
}

Params base_params(int64_t N, int64_t T, const float *boot) {
  Params p;
  std::memset(&p, 0, sizeof(p));
  p.N = N;
  p.T = T;
  p.boot = boot;
  return p;
}

}  // namespace
}  // namespace rlcs

using namespace rlcs;

extern "C" {

size_t rlcs_workspace_bytes(int64_t N, int64_t T) {
  if (N <= 0 || T <= 0) return 0;
  return ws_bytes_for(N, ceil_div(T, kMinChunk));
}

size_t rlcs_workspace_bytes_tm(int64_t N, int64_t T) {
  if (N <= 0 || T <= 0) return 0;
  return ws_bytes_tm(N, T);
}

rlcs_status rlcs_workspace_init(void *workspace, size_t bytes, rlcs_stream_t stream) {
  if (!workspace || bytes == 0) return RLCS_ERR_INVALID_ARG;
  if (cudaMemsetAsync(workspace, 0, bytes, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return RLCS_ERR_CUDA;
  }
  return RLCS_OK;
}

rlcs_status rlcs_check_status(void *workspace, rlcs_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return RLCS_ERR_CUDA;
  }
  if (!workspace) return RLCS_OK;
  uint32_t code = 0;
  WsHeader *h = static_cast<WsHeader *>(workspace);
  if (cudaMemcpy(&code, &h->status, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return RLCS_ERR_CUDA;
  }
  if (code == 0) return RLCS_OK;
  if (cudaMemset(&h->status, 0, sizeof(code)) != cudaSuccess) {
    cudaGetLastError();
    return RLCS_ERR_CUDA;
  }
  return static_cast<rlcs_status>(code);
}

const char *rlcs_status_string(rlcs_status status) {
  switch (status) {
    case RLCS_OK: return "RLCS_OK";
    case RLCS_ERR_INVALID_ARG: return "RLCS_ERR_INVALID_ARG: bad size, NULL pointer, aliasing or half a truncation pair";
    case RLCS_ERR_MISALIGNED: return "RLCS_ERR_MISALIGNED";
    case RLCS_ERR_WORKSPACE: return "RLCS_ERR_WORKSPACE: workspace missing, too small or not initialised";
    case RLCS_ERR_CUDA: return "RLCS_ERR_CUDA: a CUDA call or kernel launch failed";
    case RLCS_ERR_TIMEOUT: return "RLCS_ERR_TIMEOUT: a device-side bounded wait ran out";
  }
  return "unknown rlcs_status";
}

rlcs_status rlcs_set_shape_override(rlcs_shape shape, int64_t chunk) {
  if (shape != RLCS_SHAPE_AUTO && shape != RLCS_SHAPE_WARP_ROW &&
      shape != RLCS_SHAPE_BLOCK_CHUNK && shape != RLCS_SHAPE_BLOCK_TILE)
    return RLCS_ERR_INVALID_ARG;
  const bool block = shape == RLCS_SHAPE_BLOCK_CHUNK || shape == RLCS_SHAPE_BLOCK_TILE;
  const bool tile8192 = shape == RLCS_SHAPE_BLOCK_TILE && chunk == 8192;  // register tiles only
  if (block && !(chunk == 0 || chunk == 1024 || chunk == 2048 || chunk == 4096 || tile8192))
    return RLCS_ERR_INVALID_ARG;
  g_override_chunk.store(block ? chunk : 0);
  g_override_shape.store(shape);
  return RLCS_OK;
}

rlcs_status rlcs_internal_plan(int64_t N, int64_t T, int time_major, rlcs_plan_info *info) {
  if (!info || N <= 0 || T <= 0) return RLCS_ERR_INVALID_ARG;
  if (g_override_shape.load(std::memory_order_relaxed) != RLCS_SHAPE_AUTO)
    return RLCS_ERR_INVALID_ARG;  // the automatic plan only
  Plan plan;
  const rlcs_status st = plan_call(N, T, false, plan, time_major != 0);
  if (st != RLCS_OK) return st;
  std::memset(info, 0, sizeof(*info));
  info->shape = plan.shape;
  info->sms = sm_count();
  info->tiles_per_row = plan.Q;
  info->many_waves = plan.many_waves ? 1 : 0;
  if (plan.shape == RLCS_SHAPE_WARP_ROW) {
    info->tile = kStrip * plan.S;
    info->warps = 1;
    info->strips = plan.S;
  } else if (plan.shape == kShapeTimeMajor) {
    if (tm_narrow(N, T)) {
      const int W = plan.tm_wide ? 16 : 8;
      info->tile = (int64_t)W * 4 * kTmNarrowL;
      info->warps = W;
      info->strips = kTmNarrowL;
      info->envs = kTmNarrowEnvs;
      info->tiles_per_row = ceil_div(T, info->tile);
      info->lookback_slots = tm_window_slots(ceil_div(N, kTmNarrowEnvs), info->tiles_per_row);
    } else {
      const int L = tm_lane_steps(T);
      info->tile = kTmChunk;
      info->warps = kTmChunk / L;
      info->strips = L;
      info->envs = kTmEnvs;
      info->lookback_slots = 1;
    }
  } else {  // block tiles (the automatic long-row shape)
    info->tile = kMinChunk * plan.S;
    info->warps = plan.S == 1   ? tile_warps<1>()
                  : plan.S == 2 ? tile_warps<2>()
                  : plan.S == 4 ? tile_warps<4>()
                                : tile_warps<8>();
    info->strips = plan.S == 1   ? tile_strips<1>()
                   : plan.S == 2 ? tile_strips<2>()
                   : plan.S == 4 ? tile_strips<4>()
                                 : tile_strips<8>();
  }
  return RLCS_OK;
}

rlcs_status rlcs_gae(const float *rewards, const float *values, const float *terminateds,
                     const float *truncateds, const float *next_values,
                     const float *bootstrap_value, float *advantages, int64_t N, int64_t T,
                     double gamma, double lambda, void *workspace, size_t workspace_bytes,
                     rlcs_stream_t stream) {
  if (!rewards || !values || !terminateds || !advantages) return RLCS_ERR_INVALID_ARG;
  Params p = base_params(N, T, bootstrap_value);
  p.in[kR] = rewards;
  p.in[kV] = values;
  p.in[kD] = terminateds;
  p.out0 = advantages;
  p.gamma = (float)gamma;
  p.lambda = (float)lambda;
  set_beta(p, gamma * lambda);
  void *outs[1] = {advantages};
  return run(p, truncateds, next_values, outs, 1, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), launch_gae, truncateds != nullptr);
}

rlcs_status rlcs_lambda_returns(const float *rewards, const float *values,
                                const float *terminateds, const float *truncateds,
                                const float *next_values, const float *bootstrap_value,
                                float *returns, int64_t N, int64_t T, double gamma, double lambda,
                                void *workspace, size_t workspace_bytes, rlcs_stream_t stream) {
  if (!rewards || !values || !terminateds || !returns) return RLCS_ERR_INVALID_ARG;
  Params p = base_params(N, T, bootstrap_value);
  p.in[kR] = rewards;
  p.in[kV] = values;
  p.in[kD] = terminateds;
  p.out0 = returns;
  p.gamma = (float)gamma;
  p.lambda = (float)lambda;
  set_beta(p, gamma * lambda);
  void *outs[1] = {returns};
  return run(p, truncateds, next_values, outs, 1, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), launch_lambda_returns, truncateds != nullptr);
}

rlcs_status rlcs_discounted_returns(const float *rewards, const float *terminateds,
                                    const float *truncateds, const float *next_values,
                                    const float *bootstrap_value, float *returns, int64_t N,
                                    int64_t T, double gamma, void *workspace,
                                    size_t workspace_bytes, rlcs_stream_t stream) {
  if (!rewards || !terminateds || !returns) return RLCS_ERR_INVALID_ARG;
  Params p = base_params(N, T, bootstrap_value);
  p.in[kR] = rewards;
  p.in[kD] = terminateds;
  p.out0 = returns;
  p.gamma = (float)gamma;
  set_beta(p, gamma);
  void *outs[1] = {returns};
  return run(p, truncateds, next_values, outs, 1, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), launch_discounted_returns, truncateds != nullptr);
}

rlcs_status rlcs_vtrace(const float *rewards, const float *values, const float *log_rhos,
                        const float *terminateds, const float *truncateds,
                        const float *next_values, const float *bootstrap_value, float *vs,
                        float *pg_advantages, int64_t N, int64_t T, double gamma, double lambda,
                        double rho_bar, double c_bar, void *workspace, size_t workspace_bytes,
                        rlcs_stream_t stream) {
  if (!rewards || !values || !log_rhos || !terminateds || !vs) return RLCS_ERR_INVALID_ARG;
  Params p = base_params(N, T, bootstrap_value);
  p.in[kR] = rewards;
  p.in[kV] = values;
  p.in[kLR] = log_rhos;
  p.in[kD] = terminateds;
  p.out0 = vs;
  p.out1 = pg_advantages;
  p.gamma = (float)gamma;
  p.lambda = (float)lambda;
  p.rho_bar = (float)rho_bar;
  p.c_bar = (float)c_bar;
  void *outs[2] = {vs, pg_advantages};
  return run(p, truncateds, next_values, outs, 2, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), launch_vtrace, truncateds != nullptr);
}

rlcs_status rlcs_retrace(const float *rewards, const float *values, const float *q_values,
                         const float *log_rhos, const float *terminateds,
                         const float *truncateds, const float *next_values,
                         const float *bootstrap_value, float *q_ret, int64_t N, int64_t T,
                         double gamma, double lambda, double c_bar, void *workspace,
                         size_t workspace_bytes, rlcs_stream_t stream) {
  if (!rewards || !values || !q_values || !log_rhos || !terminateds || !q_ret)
    return RLCS_ERR_INVALID_ARG;
  Params p = base_params(N, T, bootstrap_value);
  p.in[kR] = rewards;
  p.in[kV] = values;
  p.in[kQ] = q_values;
  p.in[kLR] = log_rhos;
  p.in[kD] = terminateds;
  p.out0 = q_ret;
  p.gamma = (float)gamma;
  p.lambda = (float)lambda;
  p.c_bar = (float)c_bar;
  void *outs[1] = {q_ret};
  return run(p, truncateds, next_values, outs, 1, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), launch_retrace, truncateds != nullptr);
}

rlcs_status rlcs_eligibility_traces(const float *x, const float *dones, float *traces, int64_t N,
                                    int64_t T, double gamma, double lambda, void *workspace,
                                    size_t workspace_bytes, rlcs_stream_t stream) {
  if (!x || !dones || !traces) return RLCS_ERR_INVALID_ARG;
  Params p = base_params(N, T, nullptr);
  p.in[kR] = x;
  p.in[kD] = dones;
  p.out0 = traces;
  p.gamma = (float)gamma;
  p.lambda = (float)lambda;
  set_beta(p, gamma * lambda);
  void *outs[1] = {traces};
  return run(p, nullptr, nullptr, outs, 1, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), launch_eligibility_traces, false);
}

rlcs_status rlcs_episodic_prefix_sum(const int32_t *x, const float *dones, int32_t *out,
                                     int64_t N, int64_t T, void *workspace,
                                     size_t workspace_bytes, rlcs_stream_t stream) {
  if (!x || !dones || !out) return RLCS_ERR_INVALID_ARG;
  Params p = base_params(N, T, nullptr);
  p.in[kR] = reinterpret_cast<const float *>(x);  // raw int32 bits travel in slot R
  p.in[kD] = dones;
  p.out0 = out;
  void *outs[1] = {out};
  return run(p, nullptr, nullptr, outs, 1, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), launch_episodic_prefix_sum, false);
}

}  // extern "C"

extern "C" rlcs_status rlcs_gae_and_returns(const float *rewards, const float *values,
                                            const float *terminateds, const float *truncateds,
                                            const float *next_values,
                                            const float *bootstrap_value, float *advantages,
                                            float *returns, int64_t N, int64_t T, double gamma,
                                            double lambda, void *workspace,
                                            size_t workspace_bytes, rlcs_stream_t stream) {
  if (!rewards || !values || !terminateds || !advantages || !returns) return RLCS_ERR_INVALID_ARG;
  Params p = base_params(N, T, bootstrap_value);
  p.in[kR] = rewards;
  p.in[kV] = values;
  p.in[kD] = terminateds;
  p.out0 = advantages;
  p.out1 = returns;
  p.gamma = (float)gamma;
  p.lambda = (float)lambda;
  set_beta(p, gamma * lambda);
  void *outs[2] = {advantages, returns};
  return run(p, truncateds, next_values, outs, 2, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), launch_gae_and_returns,
             truncateds != nullptr);
}

extern "C" rlcs_status rlcs_gae_compact(const uint16_t *rewards, const uint16_t *values,
                                        const uint8_t *terminateds, const uint8_t *truncateds,
                                        const uint16_t *next_values,
                                        const float *bootstrap_value, float *advantages,
                                        int64_t N, int64_t T, double gamma, double lambda,
                                        void *workspace, size_t workspace_bytes,
                                        rlcs_stream_t stream) {
  if (!rewards || !values || !terminateds || !advantages) return RLCS_ERR_INVALID_ARG;
  Params p = base_params(N, T, bootstrap_value);
  p.in[kR] = reinterpret_cast<const float *>(rewards);
  p.in[kV] = reinterpret_cast<const float *>(values);
  p.in[kD] = reinterpret_cast<const float *>(terminateds);
  p.out0 = advantages;
  p.gamma = (float)gamma;
  p.lambda = (float)lambda;
  set_beta(p, gamma * lambda);
  void *outs[1] = {advantages};
  static const int esize[kNumSlots] = {2, 2, 4, 4, 1, 1, 2};  // R V Q LR D Tau NV
  return run(p, reinterpret_cast<const float *>(truncateds),
             reinterpret_cast<const float *>(next_values), outs, 1, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream), launch_gae_compact, truncateds != nullptr,
             esize);
}

extern "C" rlcs_status rlcs_affine_scan(const float *a, const float *b, const float *reset,
                                        const float *x_init, float *x, int64_t N, int64_t T,
                                        int reverse, void *workspace, size_t workspace_bytes,
                                        rlcs_stream_t stream) {
  if (!a || !b || !x) return RLCS_ERR_INVALID_ARG;
  Params p = base_params(N, T, x_init);
  p.in[kR] = b;
  p.in[kQ] = a;
  p.in[kD] = reset;
  p.out0 = x;
  void *outs[1] = {x};
  return run(p, nullptr, nullptr, outs, 1, workspace, workspace_bytes,
             reinterpret_cast<cudaStream_t>(stream),
             reverse ? launch_affine_backward : launch_affine_forward, reset != nullptr);
}

// ---------------------------------------------------------------------------
// Time-major [T, N] entry points: the row-major validation and functors,
// launched in the time-major shape.
// ---------------------------------------------------------------------------
extern "C" {

rlcs_status rlcs_gae_tm(const float *rewards, const float *values, const float *terminateds,
                        const float *truncateds, const float *next_values,
                        const float *bootstrap_value, float *advantages, int64_t N, int64_t T,
                        double gamma, double lambda, void *workspace, size_t workspace_bytes,
                        rlcs_stream_t stream) {
  TimeMajorScope tm;
  return rlcs_gae(rewards, values, terminateds, truncateds, next_values, bootstrap_value,
                  advantages, N, T, gamma, lambda, workspace, workspace_bytes, stream);
}

rlcs_status rlcs_lambda_returns_tm(const float *rewards, const float *values,
                                   const float *terminateds, const float *truncateds,
                                   const float *next_values, const float *bootstrap_value,
                                   float *returns, int64_t N, int64_t T, double gamma,
                                   double lambda, void *workspace, size_t workspace_bytes,
                                   rlcs_stream_t stream) {
  TimeMajorScope tm;
  return rlcs_lambda_returns(rewards, values, terminateds, truncateds, next_values,
                             bootstrap_value, returns, N, T, gamma, lambda, workspace,
                             workspace_bytes, stream);
}

rlcs_status rlcs_discounted_returns_tm(const float *rewards, const float *terminateds,
                                       const float *truncateds, const float *next_values,
                                       const float *bootstrap_value, float *returns, int64_t N,
                                       int64_t T, double gamma, void *workspace,
                                       size_t workspace_bytes, rlcs_stream_t stream) {
  TimeMajorScope tm;
  return rlcs_discounted_returns(rewards, terminateds, truncateds, next_values, bootstrap_value,
                                 returns, N, T, gamma, workspace, workspace_bytes, stream);
}

rlcs_status rlcs_vtrace_tm(const float *rewards, const float *values, const float *log_rhos,
                           const float *terminateds, const float *truncateds,
                           const float *next_values, const float *bootstrap_value, float *vs,
                           float *pg_advantages, int64_t N, int64_t T, double gamma,
                           double lambda, double rho_bar, double c_bar, void *workspace,
                           size_t workspace_bytes, rlcs_stream_t stream) {
  TimeMajorScope tm;
  return rlcs_vtrace(rewards, values, log_rhos, terminateds, truncateds, next_values,
                     bootstrap_value, vs, pg_advantages, N, T, gamma, lambda, rho_bar, c_bar,
                     workspace, workspace_bytes, stream);
}

rlcs_status rlcs_retrace_tm(const float *rewards, const float *values, const float *q_values,
                            const float *log_rhos, const float *terminateds,
                            const float *truncateds, const float *next_values,
                            const float *bootstrap_value, float *q_ret, int64_t N, int64_t T,
                            double gamma, double lambda, double c_bar, void *workspace,
                            size_t workspace_bytes, rlcs_stream_t stream) {
  TimeMajorScope tm;
  return rlcs_retrace(rewards, values, q_values, log_rhos, terminateds, truncateds, next_values,
                      bootstrap_value, q_ret, N, T, gamma, lambda, c_bar, workspace,
                      workspace_bytes, stream);
}

rlcs_status rlcs_eligibility_traces_tm(const float *x, const float *dones, float *traces,
                                       int64_t N, int64_t T, double gamma, double lambda,
                                       void *workspace, size_t workspace_bytes,
                                       rlcs_stream_t stream) {
  TimeMajorScope tm;
  return rlcs_eligibility_traces(x, dones, traces, N, T, gamma, lambda, workspace,
                                 workspace_bytes, stream);
}

rlcs_status rlcs_episodic_prefix_sum_tm(const int32_t *x, const float *dones, int32_t *out,
                                        int64_t N, int64_t T, void *workspace,
                                        size_t workspace_bytes, rlcs_stream_t stream) {
  TimeMajorScope tm;
  return rlcs_episodic_prefix_sum(x, dones, out, N, T, workspace, workspace_bytes, stream);
}

rlcs_status rlcs_gae_and_returns_tm(const float *rewards, const float *values,
                                    const float *terminateds, const float *truncateds,
                                    const float *next_values, const float *bootstrap_value,
                                    float *advantages, float *returns, int64_t N, int64_t T,
                                    double gamma, double lambda, void *workspace,
                                    size_t workspace_bytes, rlcs_stream_t stream) {
  TimeMajorScope tm;
  return rlcs_gae_and_returns(rewards, values, terminateds, truncateds, next_values,
                              bootstrap_value, advantages, returns, N, T, gamma, lambda,
                              workspace, workspace_bytes, stream);
}

rlcs_status rlcs_affine_scan_tm(const float *a, const float *b, const float *reset,
                                const float *x_init, float *x, int64_t N, int64_t T, int reverse,
                                void *workspace, size_t workspace_bytes, rlcs_stream_t stream) {
  TimeMajorScope tm;
  return rlcs_affine_scan(a, b, reset, x_init, x, N, T, reverse, workspace, workspace_bytes,
                          stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Grouped calls: one launch per class (short rows by strips and optional inputs,
// long rows by tile length and optional inputs).
// ---------------------------------------------------------------------------
namespace rlcs {
namespace {

// Pass one call through its namesake entry point (validation and recording).
rlcs_status group_one(const rlcs_call &c, rlcs_stream_t stream) {
  switch (c.estimator) {
    case RLCS_EST_GAE:
      return rlcs_gae(static_cast<const float *>(c.rewards), c.values, c.terminateds,
                      c.truncateds, c.next_values, c.bootstrap_value,
                      static_cast<float *>(c.out), c.N, c.T, c.gamma, c.lambda, nullptr, 0,
                      stream);
    case RLCS_EST_LAMBDA_RETURNS:
      return rlcs_lambda_returns(static_cast<const float *>(c.rewards), c.values,
                                 c.terminateds, c.truncateds, c.next_values, c.bootstrap_value,
                                 static_cast<float *>(c.out), c.N, c.T, c.gamma, c.lambda,
                                 nullptr, 0, stream);
    case RLCS_EST_DISCOUNTED_RETURNS:
      return rlcs_discounted_returns(static_cast<const float *>(c.rewards), c.terminateds,
                                     c.truncateds, c.next_values, c.bootstrap_value,
                                     static_cast<float *>(c.out), c.N, c.T, c.gamma, nullptr, 0,
                                     stream);
    case RLCS_EST_VTRACE:
      return rlcs_vtrace(static_cast<const float *>(c.rewards), c.values, c.log_rhos,
                         c.terminateds, c.truncateds, c.next_values, c.bootstrap_value,
                         static_cast<float *>(c.out), c.out2, c.N, c.T, c.gamma, c.lambda,
                         c.rho_bar, c.c_bar, nullptr, 0, stream);
    case RLCS_EST_RETRACE:
      return rlcs_retrace(static_cast<const float *>(c.rewards), c.values, c.q_values,
                          c.log_rhos, c.terminateds, c.truncateds, c.next_values,
                          c.bootstrap_value, static_cast<float *>(c.out), c.N, c.T, c.gamma,
                          c.lambda, c.c_bar, nullptr, 0, stream);
    case RLCS_EST_ELIGIBILITY_TRACES:
      return rlcs_eligibility_traces(static_cast<const float *>(c.rewards), c.terminateds,
                                     static_cast<float *>(c.out), c.N, c.T, c.gamma, c.lambda,
                                     nullptr, 0, stream);
    case RLCS_EST_EPISODIC_PREFIX_SUM:
      return rlcs_episodic_prefix_sum(static_cast<const int32_t *>(c.rewards), c.terminateds,
                                      static_cast<int32_t *>(c.out), c.N, c.T, nullptr, 0,
                                      stream);
    case RLCS_EST_GAE_AND_RETURNS:
      return rlcs_gae_and_returns(static_cast<const float *>(c.rewards), c.values,
                                  c.terminateds, c.truncateds, c.next_values, c.bootstrap_value,
                                  static_cast<float *>(c.out), c.out2, c.N, c.T, c.gamma,
                                  c.lambda, nullptr, 0, stream);
  }
  return RLCS_ERR_INVALID_ARG;
}

struct GroupScope {
  explicit GroupScope(GroupCollect *g) { t_group = g; }
  ~GroupScope() { t_group = nullptr; }
};

}  // namespace
}  // namespace rlcs

extern "C" size_t rlcs_group_workspace_bytes(const rlcs_call *calls, int n_calls) {
  if (calls == nullptr || n_calls <= 0 || n_calls > RLCS_MAX_GROUP) return 0;
  int64_t Ns[kMaxGroup], Ts[kMaxGroup];
  int n = 0;
  for (int i = 0; i < n_calls; ++i)
    if (calls[i].N > 0 && calls[i].T > kRowMaxT) {
      Ns[n] = calls[i].N;
      Ts[n] = calls[i].T;
      ++n;
    }
  const int64_t recs = group_records(Ns, Ts, n);
  return recs > 0 ? ws_bytes_for(recs, 1) : 0;
}

extern "C" rlcs_status rlcs_run_group(const rlcs_call *calls, int n_calls, void *workspace,
                                      size_t workspace_bytes, rlcs_stream_t stream) {
  if (n_calls < 0 || n_calls > RLCS_MAX_GROUP || (n_calls > 0 && calls == nullptr))
    return RLCS_ERR_INVALID_ARG;
  if (n_calls == 0) return RLCS_OK;
  GroupCollect col;
  {
    GroupScope scope(&col);
    for (int i = 0; i < n_calls; ++i) {
      if (calls[i].reserved != 0) return RLCS_ERR_INVALID_ARG;
      const rlcs_status st = group_one(calls[i], stream);
      if (st != RLCS_OK) return st;
    }
  }
  // calls run concurrently: no call may write what another reads or writes
  for (int i = 0; i < col.n; ++i)
    for (int w = 0; w < 2; ++w) {
      const Buf &out = col.e[i].writes[w];
      if (!out.p) continue;
      for (int j = 0; j < col.n; ++j) {
        if (j == i) continue;
        for (const Buf &b : col.e[j].reads)
          if (overlaps(out, b)) return RLCS_ERR_INVALID_ARG;
        for (const Buf &b : col.e[j].writes)
          if (overlaps(out, b)) return RLCS_ERR_INVALID_ARG;
      }
    }
  // long rows: tile lengths from the whole group, then the workspace
  int64_t long_rows = 0;
  for (int i = 0; i < col.n; ++i)
    if (col.e[i].long_row) long_rows += col.e[i].p.N;
  int64_t Q[kMaxGroup] = {}, recs = 0;
  for (int i = 0; i < col.n; ++i) {
    GroupEntry &g = col.e[i];
    if (!g.long_row) continue;
    const int64_t chunk = group_chunk(long_rows, g.p.T);
    g.S = (int)(chunk / kMinChunk);
    Q[i] = ceil_div(g.p.T, chunk);
    if (Q[i] > 1) recs += g.p.N * Q[i];
  }
  WsHeader *wsh = nullptr;
  if (recs > 0) {
    if (!workspace || workspace_bytes < ws_bytes_for(recs, 1) || !aligned16(workspace))
      return RLCS_ERR_WORKSPACE;
    const Buf wb{workspace, workspace_bytes};
    for (int i = 0; i < col.n; ++i) {
      for (const Buf &b : col.e[i].reads)
        if (overlaps(wb, b)) return RLCS_ERR_INVALID_ARG;
      for (const Buf &b : col.e[i].writes)
        if (overlaps(wb, b)) return RLCS_ERR_INVALID_ARG;
    }
    wsh = static_cast<WsHeader *>(workspace);
  }
  // one launch per class, calls in their given order within it
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  bool done[kMaxGroup] = {};
  int64_t rec_off = 0;
  for (int i = 0; i < col.n; ++i) {
    if (done[i]) continue;
    const GroupEntry &lead = col.e[i];
    auto same_class = [&](const GroupEntry &g) {
      return g.long_row == lead.long_row && g.S == lead.S && g.trunc == lead.trunc;
    };
    cudaError_t err;
    if (!lead.long_row) {
      GroupParams gp;
      std::memset(&gp, 0, sizeof(gp));
      int64_t blocks = 0;
      for (int j = i; j < col.n; ++j) {
        if (done[j] || !same_class(col.e[j])) continue;
        done[j] = true;
        gp.kind[gp.n] = col.e[j].kind;
        gp.p[gp.n] = col.e[j].p;
        gp.first_block[gp.n] = blocks;
        blocks += ceil_div(col.e[j].p.N, kRowWarps);
        ++gp.n;
      }
      gp.first_block[gp.n] = blocks;
      if (blocks >= (int64_t)INT32_MAX) return RLCS_ERR_INVALID_ARG;
      err = launch_group(gp, lead.S, lead.trunc, s);
    } else {
      GroupTileParams gp;
      std::memset(&gp, 0, sizeof(gp));
      int64_t blocks = 0, chained = 0;
      for (int j = i; j < col.n; ++j) {
        if (done[j] || !same_class(col.e[j])) continue;
        done[j] = true;
        const int64_t tiles = col.e[j].p.N * Q[j];
        gp.kind[gp.n] = col.e[j].kind;
        gp.p[gp.n] = col.e[j].p;
        gp.ts[gp.n] = TileShape{Q[j] > 1 ? wsh : nullptr, Q[j], 0, Q[j] > 1 ? rec_off : 0};
        gp.first_block[gp.n] = blocks;
        blocks += tiles;
        if (Q[j] > 1) {
          rec_off += tiles;
          chained += tiles;
        }
        ++gp.n;
      }
      gp.first_block[gp.n] = blocks;
      for (int c = 0; c < gp.n; ++c) gp.ts[c].total_tiles = chained;  // finish_launch count
      // round-major block order when every call has the same rows and tiles
      // per row (see GroupTileParams)
      bool uniform = gp.n > 1;
      for (int c = 1; c < gp.n && uniform; ++c)
        uniform = gp.p[c].N == gp.p[0].N && gp.ts[c].tiles_per_row == gp.ts[0].tiles_per_row;
      gp.round_rows = (uniform && gp.ts[0].tiles_per_row > 1) ? gp.p[0].N : 0;
      if (blocks >= (int64_t)INT32_MAX) return RLCS_ERR_INVALID_ARG;
      err = launch_group_tiles(gp, lead.S, lead.trunc, s);
    }
    if (err != cudaSuccess) {
      cudaGetLastError();
      return RLCS_ERR_CUDA;
    }
  }
  return RLCS_OK;
}

// ---------------------------------------------------------------------------
// GAE for callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc: a plugin inside a host
// program that owns every device allocation, or a real-time loop that
// forbids allocating after start-up. They cannot provide the workspace that
// long rows need, so here the look-back scratch lives in a fixed array of
// device memory that belongs to this library: a 64-byte header plus 65536
// chunk records of 32 bytes (about 2 MiB), held on every GPU that loads the
// library until the process exits.
// ---------------------------------------------------------------------------
namespace rlcs {
namespace {

constexpr int64_t kNoAllocRecords = 65536;
constexpr size_t kNoAllocBytes = sizeof(WsHeader) + sizeof(WsRecord) * kNoAllocRecords;

// Device memory. In host code this name is only a stand-in for the symbol;
// the array's device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];  // device address of the array, per device

// Once per device, with that device current: look up the array's device
// address and zero it. The header's ticket and done counters must start at
// zero; every call leaves them at zero again when it finishes.
rlcs_status noalloc_scratch(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return RLCS_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return RLCS_ERR_CUDA;
    }
    if (cudaMemset(p, 0, kNoAllocBytes) != cudaSuccess ||
        cudaStreamSynchronize(nullptr) != cudaSuccess) {
      cudaGetLastError();
      return RLCS_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return RLCS_OK;
}

}  // namespace
}  // namespace rlcs

extern "C" rlcs_status rlcs_gae_noalloc(const float *rewards, const float *values,
                                        const float *terminateds, const float *truncateds,
                                        const float *next_values, const float *bootstrap_value,
                                        float *advantages, int64_t N, int64_t T, double gamma,
                                        double lambda, rlcs_stream_t stream) {
  if (!rewards || !values || !terminateds || !advantages || N <= 0 || T <= 0)
    return RLCS_ERR_INVALID_ARG;
  if (rlcs_workspace_bytes(N, T) > kNoAllocBytes) return RLCS_ERR_WORKSPACE;
  void *scratch = nullptr;
  const rlcs_status st = noalloc_scratch(&scratch);
  if (st != RLCS_OK) return st;
  return rlcs_gae(rewards, values, terminateds, truncateds, next_values, bootstrap_value,
                  advantages, N, T, gamma, lambda, scratch, kNoAllocBytes, stream);
}

// Status and repair of the scratch array. Reading the status needs the
// stream's work done; the zeroing covers the whole array, records included:
// a header-only reset would restart the epoch at 0, whose tag the records of
// the earliest calls still carry.
extern "C" rlcs_status rlcs_gae_noalloc_recover(rlcs_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void *scratch = nullptr;
  const rlcs_status st = noalloc_scratch(&scratch);
  if (st != RLCS_OK) return st;
  if (cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return RLCS_ERR_CUDA;
  }
  uint32_t code = 0;
  const WsHeader *h = static_cast<const WsHeader *>(scratch);
  if (cudaMemcpy(&code, &h->status, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemsetAsync(scratch, 0, kNoAllocBytes, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return RLCS_ERR_CUDA;
  }
  return static_cast<rlcs_status>(code);
}

extern "C" rlcs_status rlcs_internal_noalloc_scratch(void **device_ptr, size_t *bytes) {
  if (!device_ptr || !bytes) return RLCS_ERR_INVALID_ARG;
  const rlcs_status st = noalloc_scratch(device_ptr);
  if (st != RLCS_OK) return st;
  *bytes = kNoAllocBytes;
  return RLCS_OK;
}
