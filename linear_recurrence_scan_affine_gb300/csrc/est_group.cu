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

template <bool TRUNC>
static cudaError_t launch_group_tiles_s(const GroupTileParams &gp, int S, cudaStream_t s) {
  const dim3 grid((unsigned)gp.first_block[gp.n]), block(kChunkThreads);
  switch (S) {
    case 1: return launch_ex(group_tile_kernel<TRUNC, 1>, grid, block, 0, s, true, gp);
    case 2: return launch_ex(group_tile_kernel<TRUNC, 2>, grid, block, 0, s, true, gp);
    case 4: return launch_ex(group_tile_kernel<TRUNC, 4>, grid, block, 0, s, true, gp);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_group_tiles(const GroupTileParams &gp, int S, bool trunc, cudaStream_t s) {
  return trunc ? launch_group_tiles_s<true>(gp, S, s) : launch_group_tiles_s<false>(gp, S, s);
}

}  // namespace rlcs
