// Kernel instantiations and launcher for GAE on compact (bf16 / uint8) inputs.
#include "launch.cuh"

namespace rlcs {
cudaError_t launch_gae_compact(const Params &p, const Plan &plan, WsHeader *ws, cudaStream_t s) {
  return launch_estimator<GaeCompact>(p, plan, ws, s);
}
}  // namespace rlcs
