// Kernel instantiations and launchers for grouped calls (warp rows and block tiles).
#include "launch.cuh"

namespace rlcs {

template <bool TRUNC>
static cudaError_t launch_group_s(const GroupParams &gp, int S, cudaStream_t s) {
  const dim3 grid((unsigned)gp.first_block[gp.n]), block(kRowWarps * 32);
  switch (S) {
    case 1: return launch_ex(group_row_kernel<TRUNC, 1>, grid, block, 0, s, true, gp);
    case 2: return launch_ex(group_row_kernel<TRUNC, 2>, grid, block, 0, s, true, gp);
    case 4: return launch_ex(group_row_kernel<TRUNC, 4>, grid, block, 0, s, true, gp);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_group(const GroupParams &gp, int S, bool trunc, cudaStream_t s) {
  return trunc ? launch_group_s<true>(gp, S, s) : launch_group_s<false>(gp, S, s);
}

// S: tile length / 1024, laid out as tile_warps<S>() warps of tile_strips<S>() strips
template <bool TRUNC, int S>
static cudaError_t launch_group_tiles_w(const GroupTileParams &gp, cudaStream_t s) {
  constexpr int TS = tile_strips<S>(), TW = tile_warps<S>();
  const dim3 grid((unsigned)gp.first_block[gp.n]), block(TW * 32);
  return launch_ex(group_tile_kernel<TRUNC, TS, TW>, grid, block, 0, s, true, gp);
}

template <bool TRUNC>
static cudaError_t launch_group_tiles_s(const GroupTileParams &gp, int S, cudaStream_t s) {
  switch (S) {
    case 1: return launch_group_tiles_w<TRUNC, 1>(gp, s);
    case 2: return launch_group_tiles_w<TRUNC, 2>(gp, s);
    case 4: return launch_group_tiles_w<TRUNC, 4>(gp, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_group_tiles(const GroupTileParams &gp, int S, bool trunc, cudaStream_t s) {
  return trunc ? launch_group_tiles_s<true>(gp, S, s) : launch_group_tiles_s<false>(gp, S, s);
}

}  // namespace rlcs
