// Kernel instantiations and launcher for one estimator (VTrace).
#include "launch.cuh"

namespace rlcs {
cudaError_t launch_vtrace(const Params &p, const Plan &plan, WsHeader *ws, cudaStream_t s) {
  return launch_estimator<VTrace>(p, plan, ws, s);
}
}  // namespace rlcs
