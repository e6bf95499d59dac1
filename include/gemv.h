/*
 * libgemv — dense matrix-vector products for LLM decode on NVIDIA GB300 (sm_103a).
 *
 * Every entry point computes, for b in [0, B) and m in [0, M):
 *
 *     y[b][m] = s_m * sum_{k=0}^{K-1} A[m][k] * x[b][k]  (+ bias[m])
 *
 * with the sum accumulated in fp32 and the result rounded once (round to nearest
 * even) to the output type.  s_m is the per-row weight scale of gemv_w8 and is 1
 * for the other entry points.
 *
 * Where the operation is defined:
 *   - "16-sgemv" CUDA study notes, problem definition: y[m] = sum_k A[m][k] x[k],
 *     A is M x K row-major, one dot product per output row;
 *   - lesson 3 "GEMV and row-level parallelism", section 1 (y = A x + bias) and
 *     section 3 (bias may be absent: a NULL bias adds nothing);
 *   - the GEMM/GEMV arithmetic-intensity glossary page: decode batches of M = 1
 *     and M = 16 activation rows against one weight, fp32 accumulation for 16-bit
 *     storage types;
 *   - the NPU MatMul operator post, section 1.2: quantised MatMul with int8
 *     weights, 16-bit activations, an fp32 accumulator and a write-back to the
 *     target dtype; section 4.2: a per-channel (here per-row) weight scale.
 *
 * Layout (all row-major, contiguous, no leading-dimension arguments):
 *   A    M x K     row m starts at A + m*K
 *   x    B x K     vector b starts at x + b*K
 *   y    B x M     output row b starts at y + b*M
 *   bias M         may be NULL
 *   row_scale M    gemv_w8 only, fp32, required
 * 16-bit floating point values are passed as their IEEE binary16 / bfloat16 bit
 * patterns (uint16_t).
 *
 * Ownership and memory: every pointer is caller-owned DEVICE memory on the
 * current CUDA device.  A, x, bias and row_scale are only read; y is only written
 * and must not overlap any input (checked on the host).  The library keeps no
 * pointer after the call returns.  Only the CUDA-core split-K paths (few long rows,
 * or x[0..B) too large to stage whole) use scratch memory: they take it from the
 * stream-ordered pool (cudaMallocAsync / cudaFreeAsync on the caller's stream), so
 * nothing is allocated or freed synchronously.  The tensor-core kernel sums its K
 * slices in the shared memory of one thread-block cluster and needs none.
 *
 * Execution: asynchronous on `stream` (NULL = the legacy default stream).  The
 * call validates its arguments, picks a kernel from (dtype, M, K, B, alignment)
 * and enqueues one kernel (two on the split-K path).  It never synchronises the
 * host with the device.  Results are bitwise identical from call to call for the
 * same arguments on the same device.
 *
 * Errors: the return value.  GEMV_ERR_INVALID_VALUE for negative sizes, NULL
 * pointers where data is needed, pointers not aligned to their element size,
 * sizes whose byte counts overflow int64, or y overlapping an input;
 * GEMV_ERR_UNSUPPORTED for B > 16 (B > 256 for fp16/bf16, whose 17..256 vectors run
 * on the tensor cores); GEMV_ERR_CUDA when a CUDA call fails (the
 * cudaError_t is kept per thread, see gemv_last_cuda_error).  Nothing is enqueued
 * when an argument check fails.
 *
 * Degenerate sizes: M == 0 or B == 0 does nothing and returns GEMV_SUCCESS.
 * K == 0 is the empty sum: y = bias (or 0), and A and x may then be NULL.
 */
#ifndef LIBGEMV_GEMV_H
#define LIBGEMV_GEMV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as the CUDA runtime's cudaStream_t. */
struct CUstream_st;
typedef struct CUstream_st *gemv_stream_t;

typedef enum gemv_status {
  GEMV_SUCCESS = 0,
  GEMV_ERR_INVALID_VALUE = 1,
  GEMV_ERR_UNSUPPORTED = 2,
  GEMV_ERR_CUDA = 3,
  GEMV_ERR_DEVICE_TIMEOUT = 4 /* gemv_get_device_status: a kernel's bounded wait ran out */
} gemv_status_t;

/* Storage kinds, as used by gemv_plan_for. */
typedef enum gemv_dtype {
  GEMV_DTYPE_F32 = 0,  /* A, x, bias, y: fp32 */
  GEMV_DTYPE_F16 = 1,  /* A, x, bias, y: IEEE binary16 */
  GEMV_DTYPE_BF16 = 2, /* A, x, bias, y: bfloat16 */
  GEMV_DTYPE_W8 = 3,   /* A: int8 + fp32 row scale; x, bias, y: bfloat16 */
  GEMV_DTYPE_W4 = 4    /* A: int4, two per byte, + fp32 scale per group of
                          GEMV_W4_GROUP elements; x, bias, y: bfloat16 */
} gemv_dtype_t;

/* Elements of a row that share one int4 scale. */
#define GEMV_W4_GROUP 128

/* Maximum number of decode vectors per call of the CUDA-core GEMV kernels. */
#define GEMV_MAX_BATCH 16
/* fp16/bf16 only: up to this many vectors (B > GEMV_MAX_BATCH runs as a small-N
 * GEMM on the tensor cores; the other storage types return GEMV_ERR_UNSUPPORTED). */
#define GEMV_MAX_BATCH_TC 256

/* fp32: A M x K, x B x K, y B x M.  The "16-sgemv" notes' SGEMV plus the lesson's bias. */
gemv_status_t gemv_f32(const float *A, const float *x, const float *bias, float *y,
                       int64_t M, int64_t K, int B, gemv_stream_t stream);

/* fp16 storage, fp32 accumulation, fp16 output (arithmetic-intensity page's fp16 x @ w). */
gemv_status_t gemv_f16(const uint16_t *A, const uint16_t *x, const uint16_t *bias,
                       uint16_t *y, int64_t M, int64_t K, int B, gemv_stream_t stream);

/* bf16 storage, fp32 accumulation, bf16 output: the arithmetic-intensity glossary
 * page's 16-bit weights and activations with an fp32 accumulator (its dtype notes),
 * written back once to the storage type (NPU MatMul post, section 1.2). */
gemv_status_t gemv_bf16(const uint16_t *A, const uint16_t *x, const uint16_t *bias,
                        uint16_t *y, int64_t M, int64_t K, int B, gemv_stream_t stream);

/* Weight-only int8: A int8 M x K with row_scale[m] (fp32); x, bias, y bf16.
 * y[b][m] = row_scale[m] * sum_k A[m][k] x[b][k] + bias[m]; the int8 values are
 * widened to fp32 in registers (NPU MatMul post, sections 1.2 and 5.2). */
gemv_status_t gemv_w8(const int8_t *A, const float *row_scale, const uint16_t *x,
                      const uint16_t *bias, uint16_t *y, int64_t M, int64_t K, int B,
                      gemv_stream_t stream);

/* Weight-only int4 (NPU MatMul post, section 5.2: int4 halves the weight bytes of
 * int8 again; scales, fp32 accumulation).  A holds M x K int4 values as M x K/2
 * bytes, row-major; element k of row m is the low nibble of byte m*K/2 + k/2 for
 * even k and the high nibble for odd k, symmetric two's complement in [-8, 7].
 * group_scale is M x K/GEMV_W4_GROUP fp32: one scale per group of GEMV_W4_GROUP
 * consecutive elements of a row.  x, bias, y are bf16.
 *     y[b][m] = sum_k group_scale[m][k / GEMV_W4_GROUP] * A[m][k] * x[b][k] + bias[m]
 * Each 16-byte chunk (32 weights, inside one group) is summed in fp32 and scaled
 * once.  K must be a multiple of GEMV_W4_GROUP (GEMV_ERR_INVALID_VALUE otherwise);
 * group_scale is required when M * K > 0.  B >= 2, and B == 1 with 16 or more rows
 * per SM (below 65536 rows), run in the batched cp.async ring kernel, whose ring
 * slots carry each chunk's group scale; the other shapes run in the streaming,
 * warp-per-row, block-per-row or split-K kernels. */
gemv_status_t gemv_w4(const uint8_t *A, const float *group_scale, const uint16_t *x,
                      const uint16_t *bias, uint16_t *y, int64_t M, int64_t K, int B,
                      gemv_stream_t stream);

/* bf16 GEMV that allocates nothing.  The source pages have no counterpart: this is
 * a service for callers that cannot allocate device memory while they run (memory
 * reserved up front by their own allocator, real-time loops where an allocation
 * could block or fail, hosts that forbid the CUDA allocator).  Same arguments and
 * result as gemv_bf16, computed on the split-K path, whose partial sums live in a
 * fixed device array of GEMV_NOALLOC_SCRATCH_BYTES inside the library (held on
 * every GPU that loads the library until the process exits) instead of the
 * stream-ordered pool.
 *   - GEMV_ERR_UNSUPPORTED when the partial sums (splits x B x M x 4 bytes) would
 *     not fit in that array, or when the split-K path cannot run (rows not 16-byte
 *     aligned, fewer than two 16-byte chunks per row); nothing is launched then.
 *   - All calls share the one array: calls whose kernels overlap on the GPU race
 *     and give wrong results; order them on one stream.
 *   - The first call on each device looks up the array's address (cudaGetSymbolAddress
 *     with that device current); make it before any stream capture.  The address is
 *     kept for the life of the process: do not use this entry point on a device after
 *     cudaDeviceReset there (the reset discards the context the address belongs to). */
#define GEMV_NOALLOC_SCRATCH_BYTES (4 * 1024 * 1024)
gemv_status_t gemv_bf16_splitk_noalloc(const uint16_t *A, const uint16_t *x, const uint16_t *bias,
                                       uint16_t *y, int64_t M, int64_t K, int B,
                                       gemv_stream_t stream);

/* ------------------------------------------------------- fused epilogues */

/* Activation applied after the bias (NPU MatMul post, section 5.1: fuse the bias,
 * the activation and the residual into the MatMul rather than running separate
 * passes over y). */
typedef enum gemv_activation {
  GEMV_ACT_NONE = 0,
  GEMV_ACT_SILU = 1 /* silu(v) = v / (1 + e^-v), fp32 */
} gemv_activation_t;

/* y[b][m] = act(s_m * sum_k A[m][k] x[b][k] + bias[m]) + residual[b][m]
 * Any storage type (`dtype`); row_scale only (and required) for GEMV_DTYPE_W8
 * (M scales) and GEMV_DTYPE_W4 (the M x K/GEMV_W4_GROUP group scales), NULL
 * otherwise.  residual is B x M in y's type, may be NULL, and may be y itself
 * (in place: y += act(A x + bias)); it must not otherwise overlap y.  The kernel
 * choice, layouts and errors are those of the plain entry points. */
gemv_status_t gemv_ex(gemv_dtype_t dtype, const void *A, const float *row_scale, const void *x,
                      const void *bias, const void *residual, void *y, int64_t M, int64_t K, int B,
                      gemv_activation_t act, gemv_stream_t stream);

/* SwiGLU over a concatenated gate/up projection: A is 2I x K, rows 0..I-1 the gate
 * and rows I..2I-1 the up projection (bias and row_scale, when given, have 2I
 * entries in the same order); y is B x I:
 *     y[b][m] = silu(g) * u,  g = s_m A[m] x[b] + bias[m],
 *                             u = s_{m+I} A[m+I] x[b] + bias[m+I].
 * One launch; the gate and up sums of an output meet in registers, so the 2I
 * intermediate values never reach memory.  Needs 16-byte aligned rows with at least
 * one 16-byte chunk per lane of a warp, and for B > 1 x[0..B) small enough to stage
 * in shared memory whole (one K slice); otherwise GEMV_ERR_UNSUPPORTED and nothing is
 * launched. */
gemv_status_t gemv_swiglu(gemv_dtype_t dtype, const void *A, const float *row_scale, const void *x,
                          const void *bias, void *y, int64_t I, int64_t K, int B,
                          gemv_stream_t stream);

/* End to end on host buffers: the GEMV of gemv_f32 .. gemv_w4 (chosen by dtype) with
 * its operands in host memory.  On `stream` it copies each host input into the
 * caller's device buffer of the same size (one cudaMemcpyAsync per buffer), runs the
 * GEMV on the device buffers, and copies y back into h_y.
 *   h_A / d_A      A: M x K elements (int4: M x K / 2 bytes).  h_A == NULL skips the
 *                  copy (weights already resident in d_A).
 *   h_scale / d_scale  int8: M fp32 row scales; int4: M x K / GEMV_W4_GROUP fp32
 *                  group scales; NULL for the other types.  h_scale == NULL skips
 *                  the copy (scales resident in d_scale).
 *   h_x / d_x      x: B x K (required when K > 0).
 *   h_bias / d_bias  bias: M entries, or both NULL.
 *   h_y / d_y      y: B x M (required).
 * Ownership: all buffers are the caller's; the library allocates nothing beyond what
 * the device GEMV needs.  Host buffers should be pinned: with pageable memory the
 * copies synchronise the host.  The call returns after enqueueing; h_y holds y once
 * `stream` has drained.  Errors: bad sizes, a device buffer missing for a host buffer
 * given, or a missing x or y are GEMV_ERR_INVALID_VALUE and B beyond the type's limit
 * GEMV_ERR_UNSUPPORTED, all before any copy; a failed copy is GEMV_ERR_CUDA; the
 * device GEMV's own checks (alignment, overlap, shapes its kernels cannot run) come
 * after the input copies are enqueued, and then y is not copied back. */
gemv_status_t gemv_host(gemv_dtype_t dtype, const void *h_A, const float *h_scale, const void *h_x,
                        const void *h_bias, void *h_y, void *d_A, float *d_scale, void *d_x, void *d_bias,
                        void *d_y, int64_t M, int64_t K, int B, gemv_stream_t stream);

/* Launch overlap for the calling thread's later calls (initially GEMV_OVERLAP_LAUNCH).
 * Programmatic dependent launch: a GEMV's kernels may be scheduled while the kernel
 * before them on the stream is finishing, so that back-to-back GEMVs (a decode layer,
 * a CUDA graph of them) lose less time between kernels.
 *   GEMV_OVERLAP_OFF      plain launches.
 *   GEMV_OVERLAP_LAUNCH   each kernel waits for the previous kernel on the stream
 *                         (griddepcontrol.wait) before it reads or writes any memory:
 *                         results and ordering are those of plain launches.  Kernels
 *                         of other libraries after a GEMV are launched as usual.
 *   GEMV_OVERLAP_WEIGHTS  as GEMV_OVERLAP_LAUNCH, but the persistent kernels of 16-bit
 *                         and quantised weights issue their first loads of A (and of its
 *                         scales) before that wait.  Only for weights that the work
 *                         queued before on the stream does not write.
 * Works under CUDA graph capture (the dependency becomes a programmatic edge).
 * GEMV_ERR_INVALID_VALUE for another mode. */
#define GEMV_OVERLAP_OFF 0
#define GEMV_OVERLAP_LAUNCH 1
#define GEMV_OVERLAP_WEIGHTS 2
gemv_status_t gemv_set_launch_overlap(int mode);

/* Human-readable name of a status code (static storage, never NULL). */
const char *gemv_status_string(gemv_status_t status);

/* The cudaError_t of this thread's last GEMV_ERR_CUDA (0 if none). */
int gemv_last_cuda_error(void);

/* Kernels launched by this process so far (all threads, all devices). */
uint64_t gemv_launch_count(void);

/* ------------------------------------------------------------------ dispatcher */

/* Kernel families.  The threads given to one output row are the design axis
 * ("16-sgemv" notes, design-space summary: elements per thread x rows per warp =
 * 32; lesson 3 section 4: warp per row for short rows, block per row for long
 * ones). */
typedef enum gemv_kernel {
  GEMV_KERNEL_AUTO = 0,
  GEMV_KERNEL_ROWS_PER_WARP = 1, /* 1..16 lanes per row, several rows per warp (short K) */
  GEMV_KERNEL_WARP_PER_ROW = 2,  /* one warp per row, 16-byte coalesced loads */
  GEMV_KERNEL_BLOCK_PER_ROW = 3, /* one CTA per row, shared-memory reduction */
  GEMV_KERNEL_SPLIT_K = 4,       /* CTAs over K slices + fixed-order second pass */
  GEMV_KERNEL_BATCHED = 5,       /* B >= 2: x[0..B) in shared memory, R rows per warp */
  GEMV_KERNEL_SCALAR = 6,        /* element loads, for rows that are not 16-byte aligned */
  GEMV_KERNEL_STREAM = 7,        /* B == 1: persistent warps, one row at a time per warp,
                                    loads double-buffered across rows, x in shared memory */
  GEMV_KERNEL_XSPLIT = 8,        /* B <= 4: the 512 threads of a CTA split K, x in fp32
                                    registers, rows streamed by cp.async into per-thread
                                    shared-memory slots */
  GEMV_KERNEL_TC = 9             /* fp16/bf16, B > 16: tcgen05 MMA (M = 128 rows per CTA,
                                    N = B rounded up to 16), fp32 accumulators in tensor
                                    memory; when the row tiles are few, up to 8 K slices per
                                    tile run as one thread-block cluster and are summed in
                                    its distributed shared memory; with more tiles than
                                    two CTAs per SM hold, a persistent form (192 threads,
                                    one CTA per SM over its tiles, two accumulators so that
                                    a tile's epilogue overlaps the next tile's copies);
                                    waits bounded */
} gemv_kernel_t;

/* Where a kernel reads x from (gemv_plan_t.x_staging). */
#define GEMV_X_GLOBAL 0      /* through L1, from the caller's buffer */
#define GEMV_X_SMEM 1        /* copied once per CTA into shared memory as stored */
#define GEMV_X_SMEM_FP32 2   /* widened once per CTA into shared memory as fp32 */
#define GEMV_X_REGS 3        /* each thread's slice widened once into fp32 registers */

typedef struct gemv_plan {
  int kernel;              /* gemv_kernel_t */
  int lanes_per_row;       /* ROWS_PER_WARP / WARP_PER_ROW / SCALAR: threads per row */
  int rows_per_warp;       /* BATCHED: rows one warp carries at once; TC: 64-column
                              swizzle atoms of K per pipeline stage */
  int splits;              /* SPLIT_K: number of K slices (1 otherwise) */
  int unroll;              /* 16-byte chunks of A in flight per lane per step; the
                              BATCHED ring: steps in flight (ring slots per thread /
                              rows_per_warp: 16 slots for one vector, else 8); TC:
                              k-tiles per K slice (per tile in the persistent form) */
  int x_staging;           /* GEMV_X_GLOBAL / GEMV_X_SMEM / GEMV_X_SMEM_FP32 */
  int nb;                  /* vector count the kernel is built for (>= B, power of 2) */
  int threads;             /* threads per CTA (TC: 192 marks the persistent form) */
  int64_t grid;            /* CTAs of the first (or only) kernel */
  int smem_bytes;          /* dynamic shared memory per CTA */
  int64_t workspace_bytes; /* split-K partial sums (stream-ordered pool) */
  int variant;             /* BATCHED: GEMV_BATCHED_* */
} gemv_plan_t;

/* BATCHED kernel variants (gemv_plan_t.variant; also the force parameter + 1). */
#define GEMV_BATCHED_ROWPAIR 0    /* x as stored, 2 rows per warp (4 for 16 vectors of
                                     fp16/bf16), the next loads in registers;
                                     mixed-precision FMAs for fp16/bf16,
                                     packed fp32x2 FMAs for int8/fp32 with up to 8
                                     vectors */
#define GEMV_BATCHED_RING 1       /* A through a per-thread cp.async ring in shared
                                     memory, x widened to fp32 where it fits, packed
                                     fp32x2 FMAs (vector pairs for 8 and 16 vectors) */
#define GEMV_BATCHED_RING_MIXED 2 /* the ring with mixed-precision FMAs on 16-bit A and x */

/* Host-only: the plan the entry points would use on a device with `num_sms` SMs.
 * `aligned16` says whether A and x start on 16-byte boundaries.  Launches nothing,
 * touches no device.  Returns GEMV_ERR_INVALID_VALUE / GEMV_ERR_UNSUPPORTED for
 * arguments the entry points would reject; for M == 0 or B == 0 the plan has
 * kernel = GEMV_KERNEL_AUTO and grid = 0. */
gemv_status_t gemv_plan_for(gemv_dtype_t dtype, int64_t M, int64_t K, int B, int aligned16,
                            int num_sms, gemv_plan_t *plan);

/* TEST ONLY — not thread-safe.  Make every later call use `kernel` with `param`
 * (lanes_per_row, rows_per_warp or splits; 0 = the dispatcher's choice) when the
 * arguments allow it; GEMV_KERNEL_AUTO restores normal dispatch.  STREAM needs
 * B == 1; BATCHED needs x[0..B) to fit in shared memory and takes the variant + 1
 * (GEMV_BATCHED_*; the mixed-precision ring only for fp16/bf16); TC takes
 * param % 1000 as the ring size in KB (32..220; other values keep the dispatcher's
 * choice), param / 1000 % 10 as the number of K slices (1..8; 0 keeps the choice) and
 * param / 10000 % 10 as the cluster scheduling preference (1 spread, 2 load
 * balancing, else the default), param / 100000 % 10 as the 64-column atoms of K
 * per pipeline stage (1 or 2) and param / 1000000 % 10 as the persistent form (1 on
 * wherever K > 0 and no K split is forced, 2 off).  A forced kernel
 * that cannot handle the arguments (e.g. a vectorised kernel on unaligned rows)
 * falls back to the dispatcher's choice. */
gemv_status_t gemv_test_force_kernel(int kernel, int param);

/* TEST ONLY — the plan of this thread's last successful launch. */
gemv_status_t gemv_test_last_plan(gemv_plan_t *plan);

/* Device-side status of the kernels with bounded waits (GEMV_KERNEL_TC).
 * Synchronises `stream`, then returns GEMV_ERR_DEVICE_TIMEOUT if a wait of a kernel
 * launched on the current device since the previous call ran out (the kernel then
 * left its outputs unwritten, freed its tensor memory and returned with nothing in
 * flight), else GEMV_SUCCESS; the status word is cleared.  `bits` (may be NULL)
 * receives which wait ran out: 16 an MMA completion, 32 the final wait for work in
 * flight.  GEMV_ERR_CUDA if the synchronisation or the read fails. */
gemv_status_t gemv_get_device_status(gemv_stream_t stream, int *bits);

/* TEST ONLY — not thread-safe.  With `stall` != 0 every later GEMV_KERNEL_TC launch
 * skips the last MMA of its first CTA (in the persistent form: the MMAs of that CTA's
 * last k-tile), so that CTA's wait for it runs out after
 * `timeout_ns` (<= 0: the default of 2 s) and gemv_get_device_status reports
 * GEMV_ERR_DEVICE_TIMEOUT.  stall = 0 restores normal launches. */
gemv_status_t gemv_test_stall(int stall, int64_t timeout_ns);

#ifdef __cplusplus
}
#endif

#endif /* LIBGEMV_GEMV_H */
