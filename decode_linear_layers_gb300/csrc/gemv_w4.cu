// Kernel instances for the w4 entry point.
#include "gemv_launch.cuh"

namespace gemv {
cudaError_t launch_w4(const gemv_plan_t &p, const Args &a, float *ws, cudaStream_t s) {
  return launch<OpW4>(p, a, ws, s);
}
}  // namespace gemv
