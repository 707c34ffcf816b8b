// Kernel instantiations and launcher for one estimator (Retrace).
#include "launch.cuh"

namespace rlcs {
cudaError_t launch_retrace(const Params &p, const Plan &plan, WsHeader *ws, cudaStream_t s) {
  return launch_estimator<Retrace>(p, plan, ws, s);
}
}  // namespace rlcs
