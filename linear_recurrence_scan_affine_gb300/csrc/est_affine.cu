// Kernel instantiations and launchers for the generic affine scan.
#include "launch.cuh"

namespace rlcs {
cudaError_t launch_affine_forward(const Params &p, const Plan &plan, WsHeader *ws, cudaStream_t s) {
  return launch_estimator<Affine<false>>(p, plan, ws, s);
}
cudaError_t launch_affine_backward(const Params &p, const Plan &plan, WsHeader *ws, cudaStream_t s) {
  return launch_estimator<Affine<true>>(p, plan, ws, s);
}
}  // namespace rlcs
