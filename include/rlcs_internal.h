/*
 * rlcs_internal.h — test and tuning hooks of librlcs.so, outside the
 * supported C ABI in rlcs.h.
 *
 * These functions are exported so that the test suite and the benchmark can
 * pin a launch shape, measure what a bare launch costs, and reach the
 * library-owned scratch array of rlcs_gae_noalloc to inject a fault from the
 * host. They are not part of the estimator interface: no estimator result
 * depends on them, their behaviour may change between versions, and
 * rlcs_set_shape_override changes process-global state without any locking
 * against concurrent calls.
 */
#ifndef RLCS_INTERNAL_H_
#define RLCS_INTERNAL_H_

#include "rlcs.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Diagnostic, not an estimator: the warp-row shape's launch and data
 * movement with no scan, for measuring what a launch of a given size costs
 * before any estimator work. Reads n_inputs [N,T] float32 arrays (1..7,
 * 16-byte aligned, T % 4 == 0) and writes their elementwise sum to `out`,
 * with the same L2 prefetch and programmatic dependent launch as the
 * estimators; with `empty` nonzero the same grid only waits and exits.
 * Asynchronous on `stream`; RLCS_ERR_INVALID_ARG for bad arguments. */
rlcs_status rlcs_diag_stream_copy(const float *const *inputs, int n_inputs, float *out,
                                  int64_t N, int64_t T, int empty, rlcs_stream_t stream);

/* Launch-shape selection, exposed for testing and tuning. The library picks
 * a shape from (N, T) and the SM count:
 *   RLCS_SHAPE_WARP_ROW    one warp per row, inputs in registers (T <= 512);
 *   RLCS_SHAPE_BLOCK_TILE  one 256-thread block per row tile, inputs loaded
 *                          into registers, tiles of a row chained by
 *                          decoupled look-back through the workspace;
 *   RLCS_SHAPE_BLOCK_CHUNK one 256-thread block per row chunk, the chunk
 *                          staged into shared memory by bulk copy (TMA),
 *                          chunks chained by decoupled look-back.
 * Setting an override forces a shape and, for the two block shapes, a tile
 * or chunk length of 1024, 2048 or 4096 steps, or 8192 for the register
 * tiles (0 lets the library choose),
 * for every later call in this process until reset with RLCS_SHAPE_AUTO.
 * Not thread-safe with concurrent calls. Returns RLCS_ERR_INVALID_ARG for an
 * unknown shape or length. */
typedef enum {
  RLCS_SHAPE_AUTO = 0,
  RLCS_SHAPE_WARP_ROW = 1,
  RLCS_SHAPE_BLOCK_CHUNK = 2,
  RLCS_SHAPE_BLOCK_TILE = 3
} rlcs_shape;
rlcs_status rlcs_set_shape_override(rlcs_shape shape, int64_t chunk);

/* The launch plan the library chooses for an [N, T] call (time_major
 * nonzero: a [T, N] call) with no shape override in force, computed by the
 * same planner the entry points use and without launching anything, so the
 * planner can be tested on a machine without a GPU (the SM count is then
 * taken as 152, GB300's). It describes the estimators' common plan: compact
 * GAE and float32 discounted returns without truncation take tiles of eight
 * steps per lane instead where T % 8 == 0 and the arrays are 16-byte
 * aligned, which this query does not report. Fields:
 *   shape          an rlcs_shape, or RLCS_PLAN_TIME_MAJOR;
 *   sms            the SM count the plan was made for;
 *   tile           steps per warp row (128 * strips), row tile or chunk
 *                  (time-major: 128 steps of 32 environments);
 *   tiles_per_row  tiles (chunks) per row, chained by look-back when > 1;
 *   warps          warps per block (warp rows: 1 per row);
 *   strips         128-step strips per warp (time-major: steps per lane);
 *   many_waves     block tiles: the grid exceeds one wave of 2 blocks per
 *                  SM, so three-array calls take the 3-blocks/SM kernel;
 *   envs           time-major: environments per block (32, or 8 for at
 *                  most 256 environments and T >= 2048);
 *   lookback_slots time-major: predecessors each warp reads per environment
 *                  and look-back round (1; 4 for the 8-environment chunks
 *                  when there are at most 16 environment groups and at
 *                  least 16 chunks per environment, so a round covers
 *                  4 x warps predecessors).
 * RLCS_ERR_INVALID_ARG for N <= 0, T <= 0 or a NULL `info`. */
#define RLCS_PLAN_TIME_MAJOR 100
typedef struct {
  int shape;
  int sms;
  int64_t tile;
  int64_t tiles_per_row;
  int warps;
  int strips;
  int many_waves;
  int envs;
  int lookback_slots;
} rlcs_plan_info;
rlcs_status rlcs_internal_plan(int64_t N, int64_t T, int time_major, rlcs_plan_info *info);

/* The device address and size of rlcs_gae_noalloc's scratch array on the
 * current device (performing that entry point's one-time set-up there if no
 * call has yet). Tests use it to corrupt the array's header from the host
 * and check that rlcs_gae_noalloc_recover reports and repairs the damage.
 * RLCS_ERR_INVALID_ARG for NULL arguments, RLCS_ERR_CUDA if the set-up
 * fails. */
rlcs_status rlcs_internal_noalloc_scratch(void **device_ptr, size_t *bytes);

#ifdef __cplusplus
}
#endif

#endif /* RLCS_INTERNAL_H_ */
