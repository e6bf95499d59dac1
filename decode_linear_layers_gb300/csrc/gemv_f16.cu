// Kernel instances for the f16 entry point.
#include "gemv_launch.cuh"

namespace gemv {
cudaError_t launch_f16(const gemv_plan_t &p, const Args &a, float *ws, cudaStream_t s) {
  return launch<OpF16>(p, a, ws, s);
}
}  // namespace gemv
