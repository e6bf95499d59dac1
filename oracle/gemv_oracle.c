/*
 * CPU oracle for dense GEMV — TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * this library. It shares no code with the CUDA kernels: its own IEEE decoders,
 * its own loops, fp64 arithmetic throughout.
 *
 * What it computes (the plain definition, no blocking or reordering):
 *
 *   y[b][m] = s_m * ( sum_{k=0}^{K-1} A[m][k] * x[b][k] ) + bias[m]
 *
 *   - "16-sgemv" notes, problem definition: y[m] = sum_k A[m][k] * x[k], A is M x K
 *     row-major, one dot product per row;
 *   - "GEMV and row-level parallelism" lesson, section 1 and the reference answer's
 *     kernel: y = A x + bias, bias optional (NULL means no bias);
 *   - arithmetic-intensity page, "dtype" notes, and the NPU MatMul post, section 1.2
 *     (quantised MatMul): int8 weights with a scale, activations in a 16-bit
 *     float type, accumulation in a wider type.  s_m is the per-row scale of the
 *     int8 weights (s_m = 1 for the float storage types).
 *   - B > 1 ("small-batch decode", arithmetic-intensity page, CUDA experiment):
 *     each of the B activation rows gives one output row.
 *
 * int4 weights (dtype 4; the NPU MatMul post, section 5.2: int4 halves the weight
 * bytes again, with scales and fp32 accumulation) are read as symmetric two's
 * complement nibbles in [-8, 7], two per byte: element k of row m is in byte
 * m*K/2 + k/2, the low nibble for even k and the high nibble for odd k.  Every
 * `group` consecutive elements of a row share one fp32 scale, scale[m][k / group]
 * (an M x K/group array), so the dequantised weight is s[m][k/group] * q[m][k] and
 *
 *   y[b][m] = sum_k s[m][k/group] * q[m][k] * x[b][k] + bias[m].
 *
 * Every stored value is decoded exactly to double, every product and sum is in
 * double, k ascending, and the result is left in double (no output rounding).
 * The companion output absdot[b][m] = sum_k |s_m * A[m][k] * x[b][k]| is the scale
 * against which the GPU's fp32-accumulation error is judged.
 *
 * Fused epilogues (the NPU MatMul post, section 5.1: bias, activation and residual
 * fused into the MatMul) are the same rows followed by the elementwise step, in
 * fp64: oracle_gemv_ex applies act() and adds residual[b][m]; oracle_swiglu takes
 * rows 0..I-1 of A as the gate and rows I..2I-1 as the up projection and returns
 * silu(gate_m) * up_m, with silu(v) = v / (1 + e^-v).
 *
 * Build: gcc -O2 -fPIC -shared -ffp-contract=off -fopenmp (no fast-math, so each
 * double operation rounds once, as written).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_W8 = 3, OR_W4 = 4 };

/* Nibble `hi` (0 low, 1 high) of a byte as a two's complement int4. */
static int oracle_nibble(uint8_t byte, int hi) {
  const int v = hi ? (byte >> 4) & 15 : byte & 15;
  return v >= 8 ? v - 16 : v;
}

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_decode_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
  } else if (e == 31) {
    v = (f == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(1024 + f), e - 25);      /* (1 + f/2^10) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE binary32 — 1 sign bit, 8 exponent bits
 * (bias 127), 7 fraction bits. */
double oracle_decode_bf16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xff;
  int f = h & 0x7f;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -133);                /* subnormal: f * 2^-7 * 2^-126 */
  } else if (e == 255) {
    v = (f == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(128 + f), e - 134);      /* (1 + f/2^7) * 2^(e-127) */
  }
  return sign ? -v : v;
}

/* Element (i) of a stored array of the given kind, decoded exactly. */
static double load_a(int dtype, const void *p, size_t i) {
  switch (dtype) {
    case OR_F32: return (double)((const float *)p)[i];
    case OR_F16: return oracle_decode_f16(((const uint16_t *)p)[i]);
    case OR_BF16: return oracle_decode_bf16(((const uint16_t *)p)[i]);
    default: return (double)((const int8_t *)p)[i];
  }
}

/* x, bias and y share one storage type: fp32, fp16, or bf16 (also bf16 for w8). */
static double load_x(int dtype, const void *p, size_t i) {
  switch (dtype) {
    case OR_F32: return (double)((const float *)p)[i];
    case OR_F16: return oracle_decode_f16(((const uint16_t *)p)[i]);
    default: return oracle_decode_bf16(((const uint16_t *)p)[i]);
  }
}

/*
 * y, absdot: B x M doubles, row-major (y[b*M + m]).
 * A: M x K storage (M x K/2 bytes for OR_W4), x: B x K storage, bias: M storage or
 * NULL.  scale: M floats for OR_W8; M x K/group floats for OR_W4 (group > 0 divides
 * K, K even); ignored otherwise.  nthreads > 1 splits the rows across OpenMP
 * threads; each row is still summed by one thread, k ascending.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_gemv_g(int dtype, const void *A, const float *scale, int64_t group, const void *x,
                  const void *bias, int64_t M, int64_t K, int64_t B, double *y, double *absdot,
                  int nthreads) {
  if (M < 0 || K < 0 || B < 0 || dtype < OR_F32 || dtype > OR_W4) return -1;
  if ((dtype == OR_W8 || dtype == OR_W4) && scale == NULL && M > 0 && K > 0) return -1;
  if (dtype == OR_W4 && (group <= 0 || K % group != 0 || K % 2 != 0)) return -1;
  if (M == 0 || B == 0) return 0;
  if (y == NULL) return -1;
  if (K > 0 && (A == NULL || x == NULL)) return -1;
  const int xt = dtype == OR_W4 ? OR_BF16 : dtype;  /* x, bias: bf16 for int4 */

#ifdef _OPENMP
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
  for (int64_t m = 0; m < M; ++m) {
    double s = (dtype == OR_W8) ? (double)scale[m] : 1.0;
    double bm = (bias != NULL) ? load_x(xt, bias, (size_t)m) : 0.0;
    for (int64_t b = 0; b < B; ++b) {
      double sum = 0.0, asum = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double a;
        if (dtype == OR_W4) {
          const uint8_t byte = ((const uint8_t *)A)[m * (K / 2) + k / 2];
          a = (double)scale[m * (K / group) + k / group] * (double)oracle_nibble(byte, (int)(k & 1));
        } else {
          a = load_a(dtype, A, (size_t)(m * K + k));
        }
        double p = a * load_x(xt, x, (size_t)(b * K + k));
        sum += p;
        asum += fabs(p);
      }
      y[b * M + m] = s * sum + bm;
      if (absdot != NULL) absdot[b * M + m] = fabs(s) * asum;
    }
  }
  return 0;
}

/* The float and int8 storage kinds (no group scales). */
int oracle_gemv(int dtype, const void *A, const float *scale, const void *x,
                const void *bias, int64_t M, int64_t K, int64_t B, double *y,
                double *absdot, int nthreads) {
  if (dtype == OR_W4) return -1;
  return oracle_gemv_g(dtype, A, scale, 0, x, bias, M, K, B, y, absdot, nthreads);
}

/* Decode n stored values of one kind (0: f32, 1: f16, 2: bf16, 3: int8, 4: int4,
 * n elements from n/2 bytes, n even) to double. */
int oracle_decode(int kind, const void *p, int64_t n, double *out) {
  if (n < 0 || kind < OR_F32 || kind > OR_W4) return -1;
  if (kind == OR_W4) {
    if (n % 2 != 0) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = (double)oracle_nibble(((const uint8_t *)p)[i / 2], (int)(i & 1));
    return 0;
  }
  for (int64_t i = 0; i < n; ++i) out[i] = load_a(kind, p, (size_t)i);
  return 0;
}

/* Threads the OpenMP runtime would give a parallel region of nthreads. */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* SiLU in double: v / (1 + e^-v). */
double oracle_silu(double v) { return v / (1.0 + exp(-v)); }

/*
 * y[b][m] = act(row value) + residual[b][m], act 0 = none, 1 = SiLU; residual is
 * B x M in y's storage type (decoded like x) or NULL.  pre[b][m] (may be NULL) gets
 * the value before the activation; absdot as in oracle_gemv_g (group: int4 only).
 */
int oracle_gemv_ex(int dtype, const void *A, const float *scale, int64_t group, const void *x,
                   const void *bias, const void *residual, int64_t M, int64_t K, int64_t B, int act,
                   double *y, double *pre, double *absdot, int nthreads) {
  if (act != 0 && act != 1) return -1;
  int rc = oracle_gemv_g(dtype, A, scale, group, x, bias, M, K, B, y, absdot, nthreads);
  if (rc != 0) return rc;
  for (int64_t i = 0; i < M * B; ++i) {
    double v = y[i];
    if (pre != NULL) pre[i] = v;
    if (act == 1) v = oracle_silu(v);
    if (residual != NULL) v += load_x(dtype, residual, (size_t)i);
    y[i] = v;
  }
  return 0;
}

/*
 * SwiGLU: A is 2I x K (gate rows, then up rows), bias and scale cover the 2I rows
 * (or NULL / unused).  y[b][m] = silu(g) * u with g and u the rows m and m + I of vector b.
 * gate, up, absdot_gate, absdot_up: B x I each (may be NULL).
 */
int oracle_swiglu(int dtype, const void *A, const float *scale, int64_t group, const void *x,
                  const void *bias, int64_t I, int64_t K, int64_t B, double *y, double *gate,
                  double *up, double *absdot_gate, double *absdot_up, int nthreads) {
  if (I < 0 || B < 0) return -1;
  if (I == 0 || B == 0) return 0;
  double *full = (double *)malloc(sizeof(double) * (size_t)(2 * I * B));
  double *fabsd = (double *)malloc(sizeof(double) * (size_t)(2 * I * B));
  if (full == NULL || fabsd == NULL) { free(full); free(fabsd); return -1; }
  int rc = oracle_gemv_g(dtype, A, scale, group, x, bias, 2 * I, K, B, full, fabsd, nthreads);
  if (rc == 0) {
    for (int64_t b = 0; b < B; ++b) {
      for (int64_t m = 0; m < I; ++m) {
        const double g = full[b * 2 * I + m], u = full[b * 2 * I + m + I];
        y[b * I + m] = oracle_silu(g) * u;
        if (gate != NULL) gate[b * I + m] = g;
        if (up != NULL) up[b * I + m] = u;
        if (absdot_gate != NULL) absdot_gate[b * I + m] = fabsd[b * 2 * I + m];
        if (absdot_up != NULL) absdot_up[b * I + m] = fabsd[b * 2 * I + m + I];
      }
    }
  }
  free(full);
  free(fabsd);
  return rc;
}
