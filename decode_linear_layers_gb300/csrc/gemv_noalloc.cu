// gemv_bf16_splitk_noalloc: the bf16 split-K GEMV with its scratch memory in a
// fixed device array instead of the stream-ordered pool.
//
// Who needs this: code that must not allocate device memory while it runs, for
// example a caller whose memory is fully reserved up front by its own allocator,
// a real-time or safety-checked loop where an allocation could block or fail at a
// bad moment, or a host that forbids the CUDA allocator altogether.  The regular
// split-K path takes its partial sums from cudaMallocAsync; this entry point takes
// them from g_splitk_scratch below, a file-scope device array that exists for as
// long as the library is loaded, on every GPU that loads it.
//
// Rules that come with one shared array:
//   * Every call uses the same array, so calls whose kernels overlap in time on
//     the GPU (different streams, or different host threads on one stream without
//     ordering) race on it and give wrong results.  Order them on one stream.
//   * The array keeps whatever the last call wrote.  Nothing here needs it to start
//     at zero: the first kernel writes every partial sum that the second one reads.
//   * Requests whose partial sums need more than GEMV_NOALLOC_SCRATCH_BYTES are
//     rejected with GEMV_ERR_UNSUPPORTED before anything is launched.
//   * The first call on each device looks up the array's device address with
//     cudaGetSymbolAddress (with that device current) and keeps it; make that first
//     call before capturing a stream into a CUDA graph.  The kept address belongs to
//     the device's primary context: after cudaDeviceReset it is stale, so this entry
//     point must not be used on a device that was reset in the same process.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/gemv.h"
#include "gemv_launch.cuh"
#include "gemv_plan.h"

namespace {

constexpr int64_t kScratchFloats = GEMV_NOALLOC_SCRATCH_BYTES / 4;
static __device__ __align__(256) float g_splitk_scratch[kScratchFloats];

constexpr int kMaxDev = 256;
std::mutex g_mu;
float *g_scratch_ptr[kMaxDev] = {};
int g_sms[kMaxDev] = {};

// Device address of the scratch array and SM count on the current device.
gemv_status_t device_setup(float **ptr, int *sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) { gemv::record_cuda_error((int)e); return GEMV_ERR_CUDA; }
  if (dev < 0 || dev >= kMaxDev) return GEMV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_splitk_scratch);
    if (e != cudaSuccess) { gemv::record_cuda_error((int)e); return GEMV_ERR_CUDA; }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) { gemv::record_cuda_error((int)e); return GEMV_ERR_CUDA; }
    g_scratch_ptr[dev] = static_cast<float *>(p);
    g_sms[dev] = n;
  }
  *ptr = g_scratch_ptr[dev];
  *sms = g_sms[dev];
  return GEMV_SUCCESS;
}

bool overlap(const void *p, int64_t n, const void *q, int64_t m) {
  if (p == nullptr || q == nullptr || n <= 0 || m <= 0) return false;
  const uintptr_t a0 = (uintptr_t)p, b0 = (uintptr_t)q;
  return a0 < b0 + (uintptr_t)m && b0 < a0 + (uintptr_t)n;
}

}  // namespace

extern "C" gemv_status_t gemv_bf16_splitk_noalloc(const uint16_t *A, const uint16_t *x,
                                                  const uint16_t *bias, uint16_t *y, int64_t M,
                                                  int64_t K, int B, gemv_stream_t stream) {
  if (M < 0 || K < 0 || B < 0) return GEMV_ERR_INVALID_VALUE;
  if (B > GEMV_MAX_BATCH) return GEMV_ERR_UNSUPPORTED;
  if (M == 0 || B == 0) return GEMV_SUCCESS;
  int64_t mk, bk, bm;
  if (__builtin_mul_overflow(M, K, &mk) || __builtin_mul_overflow(mk, (int64_t)2, &mk) ||
      __builtin_mul_overflow((int64_t)B, K, &bk) || __builtin_mul_overflow(bk, (int64_t)2, &bk) ||
      __builtin_mul_overflow((int64_t)B, M, &bm) || __builtin_mul_overflow(bm, (int64_t)2, &bm))
    return GEMV_ERR_INVALID_VALUE;
  if (y == nullptr || A == nullptr || x == nullptr) return GEMV_ERR_INVALID_VALUE;
  if (((uintptr_t)A | (uintptr_t)x | (uintptr_t)y | (uintptr_t)bias) & 1) return GEMV_ERR_INVALID_VALUE;
  if (overlap(y, bm, A, mk) || overlap(y, bm, x, bk) || overlap(y, bm, bias, M * 2))
    return GEMV_ERR_INVALID_VALUE;

  float *scratch = nullptr;
  int sms = 0;
  gemv_status_t st = device_setup(&scratch, &sms);
  if (st != GEMV_SUCCESS) return st;

  // The split-K plan of the regular dispatcher; only split-K uses scratch.
  const bool al16 = ((uintptr_t)A % 16 == 0) && ((uintptr_t)x % 16 == 0);
  gemv_plan_t p;
  st = gemv::plan(GEMV_DTYPE_BF16, M, K, B, al16, sms, GEMV_KERNEL_SPLIT_K, 0, &p);
  if (st != GEMV_SUCCESS) return st;
  if (p.kernel != GEMV_KERNEL_SPLIT_K) return GEMV_ERR_UNSUPPORTED;  // unaligned rows or K too short
  if (p.workspace_bytes > GEMV_NOALLOC_SCRATCH_BYTES) return GEMV_ERR_UNSUPPORTED;

  gemv::Args a;
  a.A = A;
  a.x = x;
  a.bias = bias;
  a.scale = nullptr;
  a.y = y;
  a.M = M;
  a.K = K;
  a.B = B;
  a.pdl = gemv::launch_overlap();
  cudaError_t e = gemv::launch_bf16(p, a, scratch, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    gemv::record_cuda_error((int)e);
    return GEMV_ERR_CUDA;
  }
  gemv::count_launches(2);
  return GEMV_SUCCESS;
}
