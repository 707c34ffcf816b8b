// Diagnostic reference kernel: the warp-row tier's launch shape and data
// movement with no scan. Each warp reads its row of every input array (one
// 128-bit load per lane per 128 steps) and writes their sum, with the same L2
// bulk prefetch ahead of the grid-dependency wait and the same programmatic
// dependent launch. `empty` launches the same grid that only waits and exits.
// Timing it beside an estimator separates the per-launch floor from the
// estimator's own work.
#include "launch.cuh"

namespace rlcs {
namespace {

constexpr int kMaxDiagIn = 7;
struct DiagParams {
  const float *in[kMaxDiagIn];
  float *out;
  int n_in;
  int64_t N, T;
  int empty;
};

// NIN inputs, every load of a lane issued before any is used (as an
// estimator issues its loads).
template <int NIN>
__global__ void __launch_bounds__(kRowWarps * 32) diag_stream_copy_kernel(DiagParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kRowWarps + (threadIdx.x >> 5);
  const int64_t base = row * p.T;
  if (lane == 0 && row < p.N && !p.empty) {
#pragma unroll
    for (int k = 0; k < NIN; ++k) prefetch_l2(p.in[k] + base, (uint32_t)(p.T * 4));
  }
  pdl_wait();
  if (row >= p.N || p.empty) {
    pdl_launch_dependents();
    return;
  }
  bool triggered = false;
  for (int64_t t = 4 * lane; t < p.T; t += kStrip) {
    float4 x[NIN];
#pragma unroll
    for (int k = 0; k < NIN; ++k) x[k] = __ldg(reinterpret_cast<const float4 *>(p.in[k] + base + t));
    if (!triggered) {
      pdl_launch_dependents();
      triggered = true;
    }
    float4 acc = x[0];
#pragma unroll
    for (int k = 1; k < NIN; ++k) {
      acc.x += x[k].x; acc.y += x[k].y; acc.z += x[k].z; acc.w += x[k].w;
    }
    *reinterpret_cast<float4 *>(p.out + base + t) = acc;
  }
  if (!triggered) pdl_launch_dependents();
}

template <int NIN>
cudaError_t launch_diag(const DiagParams &p, cudaStream_t s) {
  const dim3 grid((unsigned)((p.N + kRowWarps - 1) / kRowWarps));
  return launch_ex(diag_stream_copy_kernel<NIN>, grid, dim3(kRowWarps * 32), 0, s, true, p);
}

}  // namespace
}  // namespace rlcs

using namespace rlcs;

extern "C" rlcs_status rlcs_diag_stream_copy(const float *const *inputs, int n_inputs, float *out,
                                             int64_t N, int64_t T, int empty,
                                             rlcs_stream_t stream) {
  if (!inputs || n_inputs < 1 || n_inputs > kMaxDiagIn || !out || N <= 0 || T <= 0 ||
      T % 4 != 0 || T > (int64_t)1 << 30)
    return RLCS_ERR_INVALID_ARG;
  DiagParams p{};
  for (int k = 0; k < n_inputs; ++k) {
    if (!inputs[k] || (reinterpret_cast<uintptr_t>(inputs[k]) & 15u)) return RLCS_ERR_INVALID_ARG;
    p.in[k] = inputs[k];
  }
  if (reinterpret_cast<uintptr_t>(out) & 15u) return RLCS_ERR_INVALID_ARG;
  p.out = out;
  p.n_in = n_inputs;
  p.N = N;
  p.T = T;
  p.empty = empty;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err = cudaErrorInvalidValue;
  switch (n_inputs) {
    case 1: err = launch_diag<1>(p, s); break;
    case 2: err = launch_diag<2>(p, s); break;
    case 3: err = launch_diag<3>(p, s); break;
    case 4: err = launch_diag<4>(p, s); break;
    case 5: err = launch_diag<5>(p, s); break;
    case 6: err = launch_diag<6>(p, s); break;
    case 7: err = launch_diag<7>(p, s); break;
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return RLCS_ERR_CUDA;
  }
  return RLCS_OK;
}
