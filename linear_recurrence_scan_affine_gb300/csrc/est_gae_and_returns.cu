// Kernel instantiations and launcher for fused GAE + TD(lambda) returns.
#include "launch.cuh"

namespace rlcs {
cudaError_t launch_gae_and_returns(const Params &p, const Plan &plan, WsHeader *ws, cudaStream_t s) {
  return launch_estimator<GaeAndReturns>(p, plan, ws, s);
}
}  // namespace rlcs
