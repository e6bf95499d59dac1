// Kernel instances for the bf16 entry point.
#include "gemv_launch.cuh"

namespace gemv {
cudaError_t launch_bf16(const gemv_plan_t &p, const Args &a, float *ws, cudaStream_t s) {
  return launch<OpBF16>(p, a, ws, s);
}
}  // namespace gemv
