// Kernel instances for the f32 entry point.
#include "gemv_launch.cuh"

namespace gemv {
cudaError_t launch_f32(const gemv_plan_t &p, const Args &a, float *ws, cudaStream_t s) {
  return launch<OpF32>(p, a, ws, s);
}
}  // namespace gemv
