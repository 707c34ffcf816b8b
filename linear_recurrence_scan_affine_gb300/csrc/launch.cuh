// Host-side launch of one estimator in the shape the planner chose.
#pragma once

#include <mutex>

#include "kernels.cuh"
#include "rlcs_internal.h"

namespace rlcs {

// Internal launch shapes (not rlcs_shape values): time-major [T, N] inputs,
// and tiles of eight steps per lane for light calls.
constexpr int kShapeTimeMajor = RLCS_PLAN_TIME_MAJOR;
constexpr int kShapeEight = RLCS_PLAN_TIME_MAJOR + 1;

// Steps per lane of the time-major chunk kernel (measured on GB300): 16
// warps of 8 steps for short rows, where more warps per chunk finish it
// sooner; 8 warps of 16 steps from T = 1024, where more bytes in flight per
// lane pay.
inline int tm_lane_steps(int64_t T) { return T >= 1024 ? 16 : 8; }

// Time-major calls with few environments take 8 environments per block over
// 512- or 1024-step chunks (a quarter or an eighth of the chain links of the
// 32-environment shape; the planner picks 1024 when that grid fits in one
// block per SM). Measured on GB300 (us, 8 against 32 environments per
// block): GAE 8 x 131072 8.1 against 29.8, 64 x 16384 6.9 against 11.9,
// 256 x 16384 19.4 against 20.9; with 4 blocks per SM for the three-array
// calls, discounted returns 256 x 16384 16.5 against 18.7 and 200 x 20000
// 16.7 against 19.9, prefix sum 16.1 against 19.3 and 16.7 against 20.9.
// From N = 512 the narrow shape was 0-17% slower (1024 x 4096 GAE 18.8
// against 16.6).
inline bool tm_narrow(int64_t N, int64_t T) { return N <= 256 && T >= 2048; }

// Look-back distances per warp and round for the 8-environment chunks: 4
// (all 32 lanes read, a window of 4 x warps predecessors per L2 round trip)
// when few environment groups have long chains, so that many chunks of one
// environment are in flight at once; else 1 (lanes 0..7). Measured on GB300
// (GAE and discounted returns, us, 4 against 1): 8 x 131072 8.1 / 10.3 and
// 7.3 / 9.3; 32 x 65536 13.5 / 14.2 and 12.9 / 14.6; 64 x 16384 6.9 / 7.1
// and 6.3 / 6.5; with 32 groups, 256 x 16384 GAE 20.0 / 19.4 and
// 256 x 4096 6.6 / 6.6.
inline int tm_window_slots(int64_t groups, int64_t chunks) {
  return groups <= 16 && chunks >= 16 ? 4 : 1;
}

struct Plan {
  int shape;       // RLCS_SHAPE_WARP_ROW, RLCS_SHAPE_BLOCK_CHUNK or RLCS_SHAPE_BLOCK_TILE
  int S;           // strips per warp: 1, 2 or 4
  int64_t Q;       // chunks per row (block-chunk shape)
  bool trunc;      // the estimator's optional inputs are present (truncation,
                   // or the affine scan's reset mask)
  bool pdl;        // launch with programmatic stream serialization
  bool many_waves;  // block tiles: the grid exceeds one wave of 2 blocks per SM
  int64_t rows_per_tile;  // eight-step tiles holding whole rows (Q == 1)
  bool tm_wide;           // time-major, few environments: 16-warp chunks
};

// Raise Kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device (the attribute is per device and per function).
// Set even below 48 KiB: without it, static plus dynamic shared memory must
// fit in 48 KiB together.
template <auto Kernel>
inline cudaError_t allow_dynamic_smem(size_t bytes) {
  static std::mutex mu;
  static uint64_t done = 0;  // bit d: set on device d (devices 0..63; others every call)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t b = dev < 64 ? (uint64_t{1} << dev) : 0;
  std::lock_guard<std::mutex> lock(mu);
  if (b & done) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done |= b;
  return e;
}

template <class K, class... Args>
inline cudaError_t launch_ex(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <class E, bool TRUNC, int S>
inline cudaError_t launch_shape(const Params &p, const Plan &plan, WsHeader *ws, cudaStream_t s) {
  if (plan.shape == kShapeEight) {
    // the estimators the planner routes here (compact GAE, discounted returns)
    if constexpr ((E::kBF16Slots | E::kU8Slots) != 0u ||
                  (std::is_same<E, DiscountedReturns>::value && !TRUNC)) {
      const EightShape es{plan.Q > 1 ? ws : nullptr, plan.rows_per_tile, plan.Q,
                            (plan.Q == 1 && kStrip8 % p.T == 0) ? 1 : 0};
      const int64_t blocks =
          plan.Q > 1 ? p.N * plan.Q : (p.N + plan.rows_per_tile - 1) / plan.rows_per_tile;
      const dim3 grid((unsigned)blocks);
      if (plan.S == 1) {  // 1024-step tiles: 4 warps
        if (plan.many_waves)
          return launch_ex(eight_step_tile_kernel<E, TRUNC, 4, 12>, grid, dim3(128), 0, s,
                           plan.pdl, p, es);
        return launch_ex(eight_step_tile_kernel<E, TRUNC, 4, 8>, grid, dim3(128), 0, s, plan.pdl,
                         p, es);
      }
      if (plan.S == 8)  // 8192-step tiles: 32 warps, one block per SM
        return launch_ex(eight_step_tile_kernel<E, TRUNC, 32, 1>, grid, dim3(1024), 0, s, plan.pdl,
                         p, es);
      if (plan.S == 4) {  // 4096-step tiles: 16 warps
        if (plan.many_waves)
          return launch_ex(eight_step_tile_kernel<E, TRUNC, 16, 3>, grid, dim3(512), 0, s, plan.pdl,
                           p, es);
        return launch_ex(eight_step_tile_kernel<E, TRUNC, 16, 2>, grid, dim3(512), 0, s, plan.pdl, p,
                         es);
      }
      if (plan.many_waves)
        return launch_ex(eight_step_tile_kernel<E, TRUNC, 8, 6>, grid, dim3(256), 0, s, plan.pdl, p,
                         es);
      return launch_ex(eight_step_tile_kernel<E, TRUNC, 8, 4>, grid, dim3(256), 0, s, plan.pdl, p,
                       es);
    } else {
      return cudaErrorInvalidValue;  // the planner sends no other estimator here
    }
  }
  if (plan.shape == kShapeTimeMajor) {
    if constexpr ((E::kBF16Slots | E::kU8Slots) != 0u) {
      return cudaErrorInvalidValue;  // no time-major entry takes compact inputs
    } else {
      // one chunk: 16 environments per block, twice the grid; measured
      // faster for calls that move at most four arrays, slower for the
      // heavier ones (V-trace, Retrace, the fused pair), as for the warp rows
      if (p.T <= kTmShortT && row_warps<E, TRUNC>() == 8) {
        const dim3 grid((unsigned)((p.N + kTmShortEnvs - 1) / kTmShortEnvs));
        return launch_ex(time_major_short_kernel<E, TRUNC>, grid, dim3(kTmShortWarps * 32), 0, s,
                         plan.pdl, p);
      }
      if (tm_narrow(p.N, p.T)) {
        const int64_t g8 = (p.N + kTmNarrowEnvs - 1) / kTmNarrowEnvs;
        constexpr int L = kTmNarrowL;
        if (plan.tm_wide) {
          constexpr int64_t chunk = tm_narrow_chunk<16, L>();
          const int64_t q8 = (p.T + chunk - 1) / chunk;
          const TmShape sh8{q8 > 1 ? ws : nullptr, g8, q8, tm_window_slots(g8, q8)};
          return launch_ex(time_major_narrow_kernel<E, TRUNC, 16, L>, dim3((unsigned)(g8 * q8)),
                           dim3(16 * 32), 0, s, plan.pdl, p, sh8);
        }
        constexpr int64_t chunk = tm_narrow_chunk<8, L>();
        const int64_t q8 = (p.T + chunk - 1) / chunk;
        const TmShape sh8{q8 > 1 ? ws : nullptr, g8, q8, tm_window_slots(g8, q8)};
        return launch_ex(time_major_narrow_kernel<E, TRUNC, 8, L>, dim3((unsigned)(g8 * q8)),
                         dim3(8 * 32), 0, s, plan.pdl, p, sh8);
      }

      const int64_t groups = (p.N + kTmEnvs - 1) / kTmEnvs;
      const TmShape sh{plan.Q > 1 ? ws : nullptr, groups, plan.Q, 1};
      const dim3 grid((unsigned)(groups * plan.Q));
      if (tm_lane_steps(p.T) == 16)
        return launch_ex(time_major_kernel<E, TRUNC, 16>, grid, dim3(tm_threads<16>()), 0, s,
                         plan.pdl, p, sh);
      return launch_ex(time_major_kernel<E, TRUNC, 8>, grid, dim3(tm_threads<8>()), 0, s,
                       plan.pdl, p, sh);
    }
  }
  if (plan.shape == RLCS_SHAPE_WARP_ROW) {
    constexpr int R = row_warps<E, TRUNC>();
    const dim3 grid((unsigned)((p.N + R - 1) / R));
    return launch_ex(warp_row_kernel<E, TRUNC, S>, grid, dim3(R * 32), 0, s, plan.pdl, p);
  }
  // register tiles: plan.S * 1024 steps as tile_warps warps of tile_strips strips
  constexpr int TS = tile_strips<S>(), TW = tile_warps<S>();
  constexpr bool kTwoTileKernels = TW == 16 && three_arrays<E, TRUNC>();
  const bool tiles = (E::kBF16Slots | E::kU8Slots) != 0u || plan.shape == RLCS_SHAPE_BLOCK_TILE;
  if (tiles) {  // compact inputs are never staged through shared memory
    TileShape ts{plan.Q > 1 ? ws : nullptr, plan.Q, p.N * plan.Q, 0};
    const dim3 grid((unsigned)(p.N * plan.Q)), block(TW * 32);
    if constexpr (kTwoTileKernels) {
      if (plan.many_waves)
        return launch_ex(block_tile_kernel<E, TRUNC, TS, TW, true>, grid, block, 0, s, plan.pdl,
                         p, ts);
    }
    return launch_ex(block_tile_kernel<E, TRUNC, TS, TW, false>, grid, block, 0, s, plan.pdl, p,
                     ts);
  }
  if constexpr ((E::kBF16Slots | E::kU8Slots) == 0u && S <= 4) {
    constexpr uint32_t kUse = Strips<E, TRUNC, S>::kUse;
    constexpr size_t smem = (size_t)__builtin_popcount(kUse) * kChunkWarps * kStrip * S * 4;
    if (const cudaError_t e = allow_dynamic_smem<block_chunk_kernel<E, TRUNC, S>>(smem)) return e;
    ChunkShape cs{ws, plan.Q, p.N * plan.Q};
    return launch_ex(block_chunk_kernel<E, TRUNC, S>, dim3((unsigned)(p.N * plan.Q)),
                     dim3(kChunkThreads), smem, s, plan.pdl, p, cs);
  }
  return cudaErrorInvalidValue;  // not reached: compact inputs always take tiles
}

template <class E, bool TRUNC>
inline cudaError_t launch_trunc(const Params &p, const Plan &plan, WsHeader *ws, cudaStream_t s) {
  switch (plan.S) {
    case 1: return launch_shape<E, TRUNC, 1>(p, plan, ws, s);
    case 2: return launch_shape<E, TRUNC, 2>(p, plan, ws, s);
    case 4: return launch_shape<E, TRUNC, 4>(p, plan, ws, s);
    case 8: return launch_shape<E, TRUNC, 8>(p, plan, ws, s);
    default: return cudaErrorInvalidValue;
  }
}

template <class E>
inline cudaError_t launch_estimator(const Params &p, const Plan &plan, WsHeader *ws,
                                    cudaStream_t s) {
  if constexpr (E::kOptSlots != 0u) {
    if (plan.trunc) return launch_trunc<E, true>(p, plan, ws, s);
  }
  return launch_trunc<E, false>(p, plan, ws, s);
}

// One launcher per estimator, each in its own translation unit.
cudaError_t launch_gae(const Params &, const Plan &, WsHeader *, cudaStream_t);
cudaError_t launch_lambda_returns(const Params &, const Plan &, WsHeader *, cudaStream_t);
cudaError_t launch_discounted_returns(const Params &, const Plan &, WsHeader *, cudaStream_t);
cudaError_t launch_vtrace(const Params &, const Plan &, WsHeader *, cudaStream_t);
cudaError_t launch_retrace(const Params &, const Plan &, WsHeader *, cudaStream_t);
cudaError_t launch_eligibility_traces(const Params &, const Plan &, WsHeader *, cudaStream_t);
cudaError_t launch_episodic_prefix_sum(const Params &, const Plan &, WsHeader *, cudaStream_t);
cudaError_t launch_gae_and_returns(const Params &, const Plan &, WsHeader *, cudaStream_t);
cudaError_t launch_gae_compact(const Params &, const Plan &, WsHeader *, cudaStream_t);
cudaError_t launch_affine_forward(const Params &, const Plan &, WsHeader *, cudaStream_t);
cudaError_t launch_affine_backward(const Params &, const Plan &, WsHeader *, cudaStream_t);
// One launch of grouped warp-row calls sharing S and the optional-input flag.
cudaError_t launch_group(const GroupParams &gp, int S, bool trunc, cudaStream_t s);
// One launch of grouped long-row calls (block tiles) sharing S and the flag.
cudaError_t launch_group_tiles(const GroupTileParams &gp, int S, bool trunc, cudaStream_t s);

}  // namespace rlcs
