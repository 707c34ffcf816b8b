// Kernel instantiations and launcher for one estimator (DiscountedReturns).
#include "launch.cuh"

namespace rlcs {
cudaError_t launch_discounted_returns(const Params &p, const Plan &plan, WsHeader *ws, cudaStream_t s) {
  return launch_estimator<DiscountedReturns>(p, plan, ws, s);
}
}  // namespace rlcs
