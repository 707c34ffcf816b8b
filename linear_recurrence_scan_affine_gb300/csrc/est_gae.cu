// Kernel instantiations and launcher for one estimator (Gae).
#include "launch.cuh"

namespace rlcs {
cudaError_t launch_gae(const Params &p, const Plan &plan, WsHeader *ws, cudaStream_t s) {
  return launch_estimator<Gae>(p, plan, ws, s);
}
}  // namespace rlcs
