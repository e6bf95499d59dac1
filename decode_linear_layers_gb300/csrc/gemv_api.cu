// C-ABI entry points of libgemv: argument checks, dispatch, launch.
//
// The closest interface on the source pages is lesson 3's C launch function
// (A, x, bias, y, M, N, stream) in "GEMV and row-level parallelism", which
// returns nothing and checks nothing; this boundary keeps its shape (plain device
// pointers, sizes, a stream) and adds B, status codes, host-side validation
// (the NPU MatMul post, section 3.1: parameter and shape checks before any
// kernel) and the per-shape kernel choice of gemv_plan.cpp.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/gemv.h"
#include "gemv_launch.cuh"
#include "gemv_plan.h"

namespace {

thread_local int t_last_cuda_error = 0;
thread_local gemv_plan_t t_last_plan = {};
thread_local bool t_have_plan = false;
// gemv_set_launch_overlap; programmatic dependent launches by default (they change
// no result: every kernel waits for its predecessor before touching memory)
thread_local int t_overlap = GEMV_OVERLAP_LAUNCH;

std::atomic<uint64_t> g_launches{0};
int g_force_kernel = GEMV_KERNEL_AUTO;  // test-only override (not thread-safe)
int g_force_param = 0;

constexpr int kMaxDevices = 256;
std::atomic<int> g_sm_count[kMaxDevices];

// test-only: make a tensor-core launch skip one MMA so its bounded wait runs out
int g_test_stall = 0;
int64_t g_test_timeout_ns = 0;
constexpr int64_t kDefaultTimeoutNs = 2000000000;  // 2 s

// Device status word of the kernels with bounded waits (one per device: a
// __device__ variable is instantiated in every context).
__device__ int g_device_status;
std::atomic<int *> g_status_ptr[kMaxDevices];
std::mutex g_status_mu;

gemv_status_t cuda_fail(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return GEMV_ERR_CUDA;
}

bool mul_ok(int64_t a, int64_t b, int64_t *out) { return !__builtin_mul_overflow(a, b, out); }

// [p, p + n) and [q, q + m) share a byte.
bool overlaps(const void *p, int64_t n, const void *q, int64_t m) {
  if (p == nullptr || q == nullptr || n <= 0 || m <= 0) return false;
  const uintptr_t a0 = (uintptr_t)p, a1 = a0 + (uintptr_t)n;
  const uintptr_t b0 = (uintptr_t)q, b1 = b0 + (uintptr_t)m;
  return a0 < b1 && b0 < a1;
}

bool aligned(const void *p, int bytes) { return ((uintptr_t)p % (uintptr_t)bytes) == 0; }

gemv_status_t sm_count(int *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev >= 0 && dev < kMaxDevices) {
    int v = g_sm_count[dev].load(std::memory_order_relaxed);
    if (v > 0) {
      *out = v;
      return GEMV_SUCCESS;
    }
  }
  int v = 0;
  e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(v, std::memory_order_relaxed);
  *out = v;
  return GEMV_SUCCESS;
}

gemv_status_t status_word(int **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return GEMV_ERR_UNSUPPORTED;
  int *p = g_status_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lk(g_status_mu);
    p = g_status_ptr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      void *q = nullptr;
      e = cudaGetSymbolAddress(&q, g_device_status);
      if (e != cudaSuccess) return cuda_fail(e);
      p = static_cast<int *>(q);
      g_status_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return GEMV_SUCCESS;
}

typedef cudaError_t (*launch_fn)(const gemv_plan_t &, const gemv::Args &, float *, cudaStream_t);

// M counts the rows of A.  swiglu: y has M / 2 entries per vector (M even).
gemv_status_t run(int dtype, const void *A, const float *scale, const void *x, const void *bias,
                  const void *residual, void *y, int64_t M, int64_t K, int B, int act, bool swiglu,
                  gemv_stream_t stream_in) {
  if (M < 0 || K < 0 || B < 0) return GEMV_ERR_INVALID_VALUE;
  if (dtype < GEMV_DTYPE_F32 || dtype > GEMV_DTYPE_W4) return GEMV_ERR_INVALID_VALUE;
  if (act != GEMV_ACT_NONE && act != GEMV_ACT_SILU) return GEMV_ERR_INVALID_VALUE;
  const bool w4 = dtype == GEMV_DTYPE_W4;
  if (w4 && K % GEMV_W4_GROUP != 0) return GEMV_ERR_INVALID_VALUE;
  const bool half16 = dtype == GEMV_DTYPE_F16 || dtype == GEMV_DTYPE_BF16;
  if (B > GEMV_MAX_BATCH && !(half16 && B <= GEMV_MAX_BATCH_TC)) return GEMV_ERR_UNSUPPORTED;
  if (M == 0 || B == 0) return GEMV_SUCCESS;
  const int sa = gemv::elem_bytes_a(dtype), sx = gemv::elem_bytes_x(dtype);
  const int sy = sx;
  const int64_t ym = swiglu ? M / 2 : M;  // outputs per vector
  int64_t a_bytes, x_bytes, y_bytes, mk, bk, bm;
  if (!mul_ok(M, K, &mk) || !mul_ok(mk, sa, &a_bytes)) return GEMV_ERR_INVALID_VALUE;
  if (w4) a_bytes /= 2;  // two int4 per byte
  // scale entries: one per row (int8), one per group of a row (int4)
  const int64_t s_count = w4 ? M * (K / GEMV_W4_GROUP) : M;
  if (!mul_ok(B, K, &bk) || !mul_ok(bk, sx, &x_bytes)) return GEMV_ERR_INVALID_VALUE;
  if (!mul_ok(B, ym, &bm) || !mul_ok(bm, sy, &y_bytes)) return GEMV_ERR_INVALID_VALUE;
  if (y == nullptr) return GEMV_ERR_INVALID_VALUE;
  if (K > 0 && (A == nullptr || x == nullptr)) return GEMV_ERR_INVALID_VALUE;
  if (dtype == GEMV_DTYPE_W8 && scale == nullptr) return GEMV_ERR_INVALID_VALUE;
  if (w4 && K > 0 && scale == nullptr) return GEMV_ERR_INVALID_VALUE;
  if (!aligned(A, sa) || !aligned(x, sx) || !aligned(y, sy) || !aligned(bias, sx) ||
      !aligned(scale, 4) || !aligned(residual, sy))
    return GEMV_ERR_INVALID_VALUE;
  if (overlaps(y, y_bytes, A, a_bytes) || overlaps(y, y_bytes, x, x_bytes) ||
      overlaps(y, y_bytes, bias, M * sx) || overlaps(y, y_bytes, scale, s_count * 4))
    return GEMV_ERR_INVALID_VALUE;
  // the residual may be y itself (in-place y += A x), but not a shifted view of it
  if (residual != nullptr && residual != y && overlaps(y, y_bytes, residual, y_bytes))
    return GEMV_ERR_INVALID_VALUE;

  int sms = 0;
  gemv_status_t st = sm_count(&sms);
  if (st != GEMV_SUCCESS) return st;
  const bool al16 = aligned(A, 16) && aligned(x, 16);
  gemv_plan_t p;
  if (swiglu) {
    // one vector: the streaming kernel walks gate/up row pairs; more: the batched
    // kernels carry each pair as two of their rows (the variant the dispatcher picks,
    // or the one a test forced)
    const int want = B == 1 ? GEMV_KERNEL_STREAM : GEMV_KERNEL_BATCHED;
    const int param = B > 1 && g_force_kernel == GEMV_KERNEL_BATCHED ? g_force_param : 0;
    st = gemv::plan(dtype, M, K, B, al16, sms, want, param, &p);
    if (st != GEMV_SUCCESS) return st;
    // (a K-split plan sums slices in a second pass, which knows no row pairs)
    if (p.kernel != want || p.splits > 1) return GEMV_ERR_UNSUPPORTED;
  } else {
    st = gemv::plan(dtype, M, K, B, al16, sms, g_force_kernel, g_force_param, &p);
    if (st != GEMV_SUCCESS) return st;
  }

  gemv::Args args;
  args.A = A;
  args.x = x;
  args.bias = bias;
  args.scale = w4 ? nullptr : scale;  // int4 scales are per group, applied per chunk
  args.gscale = w4 ? scale : nullptr;
  args.gshift = w4 ? 7 : 0;          // log2(GEMV_W4_GROUP)
  args.y = y;
  args.M = M;
  args.K = K;
  args.B = B;
  args.residual = residual;
  args.act = act;
  args.half = swiglu ? M / 2 : 0;
  args.pdl = t_overlap;
  if (p.kernel == GEMV_KERNEL_TC) {
    st = status_word(&args.status);
    if (st != GEMV_SUCCESS) return st;
    args.timeout_ns = g_test_stall && g_test_timeout_ns > 0 ? g_test_timeout_ns : kDefaultTimeoutNs;
    args.test_stall = g_test_stall;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream_in);

  launch_fn fn = dtype == GEMV_DTYPE_F32    ? gemv::launch_f32
                 : dtype == GEMV_DTYPE_F16  ? gemv::launch_f16
                 : dtype == GEMV_DTYPE_BF16 ? gemv::launch_bf16
                 : dtype == GEMV_DTYPE_W8   ? gemv::launch_w8
                                            : gemv::launch_w4;
  float *ws = nullptr;
  if (p.workspace_bytes > 0) {  // split-K partial sums: SPLIT_K, TC or BATCHED over K slices
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void **>(&ws), (size_t)p.workspace_bytes, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  cudaError_t e = fn(p, args, ws, s);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (ws != nullptr) {
    cudaError_t e2 = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = e2;
  }
  if (e != cudaSuccess) return cuda_fail(e);
  const bool two = p.kernel == GEMV_KERNEL_SPLIT_K || (p.kernel == GEMV_KERNEL_TC && p.splits > 1) ||
                   (p.kernel == GEMV_KERNEL_BATCHED && p.splits > 1);
  g_launches.fetch_add(two ? 2 : 1, std::memory_order_relaxed);
  t_last_plan = p;
  t_have_plan = true;
  return GEMV_SUCCESS;
}

}  // namespace

namespace gemv {
// The tensor maps of the tcgen05 kernel.  cuTensorMapEncodeTiled is a driver
// function: it is fetched once through the runtime, so the library needs no
// link-time dependency on the driver library.
bool tc_tensor_maps(int dtype, const void *A, const void *x, int64_t M, int64_t K, int B, int N, void *map_a,
                    void *map_x) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      fn = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }();
  if (encode == nullptr || M <= 0 || K <= 0 || B <= 0) return false;
  const CUtensorMapDataType t = dtype == GEMV_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint32_t es[2] = {1, 1};
  auto one = [&](void *map, const void *base, int64_t rows, cuuint32_t box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTcPlanTileK, box_rows};
    return encode(static_cast<CUtensorMap *>(map), t, 2, const_cast<void *>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  return one(map_a, A, M, (cuuint32_t)kTcPlanTileM) && one(map_x, x, B, (cuuint32_t)N);
}

// For other entry points of the library (gemv_noalloc.cu): keep the per-thread
// CUDA error and the launch counter in one place.
void record_cuda_error(int e) { t_last_cuda_error = e; }
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
int launch_overlap() { return t_overlap; }
}  // namespace gemv

extern "C" {

gemv_status_t gemv_f32(const float *A, const float *x, const float *bias, float *y, int64_t M,
                       int64_t K, int B, gemv_stream_t stream) {
  return run(GEMV_DTYPE_F32, A, nullptr, x, bias, nullptr, y, M, K, B, GEMV_ACT_NONE, false, stream);
}

gemv_status_t gemv_f16(const uint16_t *A, const uint16_t *x, const uint16_t *bias, uint16_t *y,
                       int64_t M, int64_t K, int B, gemv_stream_t stream) {
  return run(GEMV_DTYPE_F16, A, nullptr, x, bias, nullptr, y, M, K, B, GEMV_ACT_NONE, false, stream);
}

gemv_status_t gemv_bf16(const uint16_t *A, const uint16_t *x, const uint16_t *bias, uint16_t *y,
                        int64_t M, int64_t K, int B, gemv_stream_t stream) {
  return run(GEMV_DTYPE_BF16, A, nullptr, x, bias, nullptr, y, M, K, B, GEMV_ACT_NONE, false, stream);
}

gemv_status_t gemv_w8(const int8_t *A, const float *row_scale, const uint16_t *x,
                      const uint16_t *bias, uint16_t *y, int64_t M, int64_t K, int B,
                      gemv_stream_t stream) {
  return run(GEMV_DTYPE_W8, A, row_scale, x, bias, nullptr, y, M, K, B, GEMV_ACT_NONE, false, stream);
}

gemv_status_t gemv_w4(const uint8_t *A, const float *group_scale, const uint16_t *x,
                      const uint16_t *bias, uint16_t *y, int64_t M, int64_t K, int B,
                      gemv_stream_t stream) {
  return run(GEMV_DTYPE_W4, A, group_scale, x, bias, nullptr, y, M, K, B, GEMV_ACT_NONE, false, stream);
}

gemv_status_t gemv_ex(gemv_dtype_t dtype, const void *A, const float *row_scale, const void *x,
                      const void *bias, const void *residual, void *y, int64_t M, int64_t K, int B,
                      gemv_activation_t act, gemv_stream_t stream) {
  if (dtype != GEMV_DTYPE_W8 && dtype != GEMV_DTYPE_W4 && row_scale != nullptr) return GEMV_ERR_INVALID_VALUE;
  return run((int)dtype, A, row_scale, x, bias, residual, y, M, K, B, (int)act, false, stream);
}

gemv_status_t gemv_swiglu(gemv_dtype_t dtype, const void *A, const float *row_scale, const void *x,
                          const void *bias, void *y, int64_t I, int64_t K, int B,
                          gemv_stream_t stream) {
  if (I < 0) return GEMV_ERR_INVALID_VALUE;
  if (dtype != GEMV_DTYPE_W8 && dtype != GEMV_DTYPE_W4 && row_scale != nullptr) return GEMV_ERR_INVALID_VALUE;
  int64_t m2;
  if (!mul_ok(I, 2, &m2)) return GEMV_ERR_INVALID_VALUE;
  return run((int)dtype, A, row_scale, x, bias, nullptr, y, m2, K, B, GEMV_ACT_NONE, true, stream);
}

gemv_status_t gemv_host(gemv_dtype_t dtype, const void *h_A, const float *h_scale, const void *h_x,
                        const void *h_bias, void *h_y, void *d_A, float *d_scale, void *d_x, void *d_bias,
                        void *d_y, int64_t M, int64_t K, int B, gemv_stream_t stream) {
  const int dt = (int)dtype;
  if (dt < GEMV_DTYPE_F32 || dt > GEMV_DTYPE_W4 || M < 0 || K < 0 || B < 0) return GEMV_ERR_INVALID_VALUE;
  const bool w4 = dt == GEMV_DTYPE_W4, scaled = dt == GEMV_DTYPE_W8 || w4;
  const bool half16 = dt == GEMV_DTYPE_F16 || dt == GEMV_DTYPE_BF16;
  if (w4 && K % GEMV_W4_GROUP != 0) return GEMV_ERR_INVALID_VALUE;
  if (B > GEMV_MAX_BATCH && !(half16 && B <= GEMV_MAX_BATCH_TC)) return GEMV_ERR_UNSUPPORTED;
  if (M == 0 || B == 0) return GEMV_SUCCESS;
  if (h_y == nullptr || d_y == nullptr) return GEMV_ERR_INVALID_VALUE;
  if (K > 0 && (h_x == nullptr || d_x == nullptr)) return GEMV_ERR_INVALID_VALUE;
  if ((h_A != nullptr && d_A == nullptr) || (h_scale != nullptr && d_scale == nullptr) ||
      (h_bias != nullptr && d_bias == nullptr))
    return GEMV_ERR_INVALID_VALUE;
  if (!scaled && (h_scale != nullptr || d_scale != nullptr)) return GEMV_ERR_INVALID_VALUE;
  const int sa = gemv::elem_bytes_a(dt), sx = gemv::elem_bytes_x(dt);
  int64_t mk, a_bytes, bk, x_bytes, bm, y_bytes, b_bytes;
  if (!mul_ok(M, K, &mk) || !mul_ok(mk, sa, &a_bytes)) return GEMV_ERR_INVALID_VALUE;
  if (w4) a_bytes /= 2;
  const int64_t s_bytes = scaled ? (w4 ? M * (K / GEMV_W4_GROUP) : M) * 4 : 0;
  if (!mul_ok(B, K, &bk) || !mul_ok(bk, sx, &x_bytes)) return GEMV_ERR_INVALID_VALUE;
  if (!mul_ok(B, M, &bm) || !mul_ok(bm, sx, &y_bytes) || !mul_ok(M, sx, &b_bytes)) return GEMV_ERR_INVALID_VALUE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // inputs host -> device, one copy per buffer, in stream order before the GEMV
  auto h2d = [&](void *dst, const void *src, int64_t n) -> cudaError_t {
    if (src == nullptr || n == 0) return cudaSuccess;
    return cudaMemcpyAsync(dst, src, (size_t)n, cudaMemcpyHostToDevice, s);
  };
  cudaError_t e = h2d(d_A, h_A, K > 0 ? a_bytes : 0);
  if (e == cudaSuccess) e = h2d(d_scale, h_scale, K > 0 ? s_bytes : 0);
  if (e == cudaSuccess) e = h2d(d_x, h_x, x_bytes);
  if (e == cudaSuccess) e = h2d(d_bias, h_bias, b_bytes);
  if (e != cudaSuccess) return cuda_fail(e);
  const gemv_status_t st = run(dt, d_A, d_scale, d_x, h_bias != nullptr || d_bias != nullptr ? d_bias : nullptr,
                               nullptr, d_y, M, K, B, GEMV_ACT_NONE, false, stream);
  if (st != GEMV_SUCCESS) return st;
  e = cudaMemcpyAsync(h_y, d_y, (size_t)y_bytes, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return GEMV_SUCCESS;
}

gemv_status_t gemv_set_launch_overlap(int mode) {
  if (mode != GEMV_OVERLAP_OFF && mode != GEMV_OVERLAP_LAUNCH && mode != GEMV_OVERLAP_WEIGHTS)
    return GEMV_ERR_INVALID_VALUE;
  t_overlap = mode;
  return GEMV_SUCCESS;
}

const char *gemv_status_string(gemv_status_t s) {
  switch (s) {
    case GEMV_SUCCESS: return "GEMV_SUCCESS";
    case GEMV_ERR_INVALID_VALUE: return "GEMV_ERR_INVALID_VALUE";
    case GEMV_ERR_UNSUPPORTED: return "GEMV_ERR_UNSUPPORTED";
    case GEMV_ERR_CUDA: return "GEMV_ERR_CUDA";
    case GEMV_ERR_DEVICE_TIMEOUT: return "GEMV_ERR_DEVICE_TIMEOUT";
    default: return "GEMV_ERR_UNKNOWN";
  }
}

int gemv_last_cuda_error(void) { return t_last_cuda_error; }

uint64_t gemv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

gemv_status_t gemv_test_force_kernel(int kernel, int param) {
  if (kernel < GEMV_KERNEL_AUTO || kernel > GEMV_KERNEL_TC || param < 0)
    return GEMV_ERR_INVALID_VALUE;
  g_force_kernel = kernel;
  g_force_param = kernel == GEMV_KERNEL_AUTO ? 0 : param;
  return GEMV_SUCCESS;
}

gemv_status_t gemv_get_device_status(gemv_stream_t stream, int *bits) {
  if (bits != nullptr) *bits = 0;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  int *p = nullptr;
  gemv_status_t st = status_word(&p);
  if (st != GEMV_SUCCESS) return st;
  int v = 0;
  e = cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (v == 0) return GEMV_SUCCESS;
  e = cudaMemset(p, 0, sizeof v);
  if (e != cudaSuccess) return cuda_fail(e);
  if (bits != nullptr) *bits = v;
  return GEMV_ERR_DEVICE_TIMEOUT;
}

gemv_status_t gemv_test_stall(int stall, int64_t timeout_ns) {
  g_test_stall = stall != 0;
  g_test_timeout_ns = stall != 0 ? timeout_ns : 0;
  return GEMV_SUCCESS;
}

gemv_status_t gemv_test_last_plan(gemv_plan_t *plan) {
  if (plan == nullptr || !t_have_plan) return GEMV_ERR_INVALID_VALUE;
  *plan = t_last_plan;
  return GEMV_SUCCESS;
}

}  // extern "C"
