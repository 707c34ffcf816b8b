// Kernel instantiations and launcher for one estimator (EpisodicPrefixSum).
#include "launch.cuh"

namespace rlcs {
cudaError_t launch_episodic_prefix_sum(const Params &p, const Plan &plan, WsHeader *ws, cudaStream_t s) {
  return launch_estimator<EpisodicPrefixSum>(p, plan, ws, s);
}
}  // namespace rlcs
