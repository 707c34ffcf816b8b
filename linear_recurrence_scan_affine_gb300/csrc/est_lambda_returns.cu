// Kernel instantiations and launcher for one estimator (LambdaReturns).
#include "launch.cuh"

namespace rlcs {
cudaError_t launch_lambda_returns(const Params &p, const Plan &plan, WsHeader *ws, cudaStream_t s) {
  return launch_estimator<LambdaReturns>(p, plan, ws, s);
}
}  // namespace rlcs
