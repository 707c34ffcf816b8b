// Kernel instantiations and launcher for one estimator (EligibilityTraces).
#include "launch.cuh"

namespace rlcs {
cudaError_t launch_eligibility_traces(const Params &p, const Plan &plan, WsHeader *ws, cudaStream_t s) {
  return launch_estimator<EligibilityTraces>(p, plan, ws, s);
}
}  // namespace rlcs
