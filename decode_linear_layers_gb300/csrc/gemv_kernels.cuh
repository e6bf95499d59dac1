// Device code for libgemv: y[b][m] = s_m * sum_k A[m][k] * x[b][k] + bias[m].
//
// Everything here streams A once from HBM and is bound by HBM bandwidth, or for
// many vectors by the fp32 FMA rate (one multiply-add per A element per vector:
// "16-sgemv" notes, closing summary; lesson 3 "GEMV and row-level parallelism",
// section 1).  The kernels differ in how many threads share one output row and in
// where x lives:
//
//   k_rowteam   TPR = 1..32 lanes per row, x through L1.  TPR < 32: several rows
//               per warp for short rows (the notes' K = 16 kernel, generalised);
//               TPR = 32: one warp per row with 16-byte loads (the notes' float4
//               kernel), non-persistent grid for very tall matrices.  VEC = false
//               loads single elements for rows that are not 16-byte aligned.
//   k_stream    B = 1: persistent warps, one row at a time per warp, loads
//               double-buffered across row boundaries, x in shared memory.
//   k_blockrow  all 256 threads of a CTA on one row (lesson 3's block-per-row
//               kernel), optionally over one K slice of it (split-K pass 1).
//   k_splitk_reduce  split-K pass 2: sums the slices in slice order.
//   k_batched2  2 <= B <= 16 (row pairs): x in shared memory as stored, 2 rows per
//               warp (4 with 16 vectors of 16-bit rows), the next loads in registers;
//               mixed-precision FMAs for 16-bit rows, packed FMAs for int8/fp32 rows
//               with up to 8 vectors.
//   k_batch_ring  2 <= B <= 16, and int8/int4 with B = 1: A through a per-thread
//               cp.async ring, x in shared memory (fp32 where it fits), R rows per
//               warp, packed FMAs (mixed-precision FMAs for some 16-bit forms).
//   k_xsplit    B <= 4: the CTA splits K, x in fp32 registers.
//   k_tc        fp16/bf16, 17..256 vectors: tcgen05 tensor cores (gemv_tc.cuh; with
//               many row tiles the persistent k_tc_persist).
//
// All reductions are fixed trees (xor butterflies, shared memory in warp order,
// slices in index order): no atomics, bitwise-reproducible results.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gemv {

constexpr int kThreads = 256;  // 8 warps: the row-team, block-per-row and second-pass CTAs
constexpr int kWarps = kThreads / 32;

struct Args {
  const void *A = nullptr;
  const void *x = nullptr;
  const void *bias = nullptr;   // nullptr: no bias
  const float *scale = nullptr; // w8 row scale, nullptr otherwise
  void *y = nullptr;
  int64_t M = 0, K = 0;
  int B = 0;
  // fused epilogue (all kernels): activation, then residual[b][m] (y's type, B x M,
  // may be y itself).  SwiGLU (half > 0): A is [gate rows 0..half-1; up rows
  // half..2*half-1], M = 2*half, and y[b][m] = silu(gate_m) * up_m is B x half.
  const void *residual = nullptr;
  int act = 0;          // 0: none, 1: SiLU
  int64_t half = 0;
  // int4 (OpW4): one fp32 scale per 2^gshift consecutive elements of a row,
  // gscale[m][k >> gshift], M x (K >> gshift)
  const float *gscale = nullptr;
  int gshift = 0;
  // kernels with bounded waits (k_tc): device status word they OR a bit into on
  // timeout, the wait limit, and a test switch that withholds one MMA
  int *status = nullptr;
  int64_t timeout_ns = 2000000000;
  int test_stall = 0;
  // programmatic dependent launch: 0 off; 1 the kernel lets the next one launch
  // early and waits for the previous one before touching memory; 2 as 1, but the
  // first loads of A (and its scales) go out before that wait
  int pdl = 0;
};

// Programmatic dependent launch (a no-op in a kernel launched without it).
// Lets the next kernel on the stream be scheduled as SMs free up.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Waits until the previous kernel on the stream has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Start of a kernel: trigger, and wait unless the kernel may prefetch its weights.
__device__ __forceinline__ void pdl_enter(const Args &a, bool may_prefetch) {
  pdl_trigger();
  if (!(may_prefetch && a.pdl == 2)) pdl_wait();
}
// After a kernel's weight prefetch: the wait it put off.
__device__ __forceinline__ void pdl_after_prefetch(const Args &a) {
  if (a.pdl == 2) pdl_wait();
}

// ------------------------------------------------------------------ memory access
// A is read exactly once: skip L1 and mark the L2 lines evict-first so x, y and
// the rest of the working set stay cached.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint4 ld_stream16(const void *ptr, uint64_t pol) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(ptr), "l"(pol));
  return r;
}

// 16-byte global -> shared copy that bypasses registers (completed by
// cp.async.wait_group).
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}

// x is re-read by every row: the read-only path, cached in L1.
__device__ __forceinline__ uint4 ld_x16(const void *ptr) {
  return __ldg(reinterpret_cast<const uint4 *>(ptr));
}

// --------------------------------------------------------------- element decoding
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float2 f16x2_to_f2(uint32_t w) {
  __half2 h = *reinterpret_cast<const __half2 *>(&w);
  return __half22float2(h);
}

// Four 16-bit x values in two words, widened to fp32 (exact for both types).
__device__ __forceinline__ void widen4(uint32_t w0, uint32_t w1, float (&f)[4], __half) {
  const float2 f0 = f16x2_to_f2(w0), f1 = f16x2_to_f2(w1);
  f[0] = f0.x; f[1] = f0.y; f[2] = f1.x; f[3] = f1.y;
}
__device__ __forceinline__ void widen4(uint32_t w0, uint32_t w1, float (&f)[4], __nv_bfloat16) {
  f[0] = bf16_lo(w0); f[1] = bf16_hi(w0); f[2] = bf16_lo(w1); f[3] = bf16_hi(w1);
}
__device__ __forceinline__ float2 widen2(uint32_t w, __half) { return f16x2_to_f2(w); }
__device__ __forceinline__ float2 widen2(uint32_t w, __nv_bfloat16) { return make_float2(bf16_lo(w), bf16_hi(w)); }

// int8 -> fp32 without a conversion instruction: with u = q + 128 (the byte with
// its top bit flipped), the float whose bits are 0x4B0000uu is 2^23 + u exactly,
// so subtracting 2^23 + 128 leaves q exactly.  PRMT builds the bits.
template <int J>
__device__ __forceinline__ float s8_to_f32(uint32_t flipped) {
  return __uint_as_float(__byte_perm(flipped, 0x4B000000u, 0x7540 + J)) - 8388736.0f;
}

// ------------------------------------------------------------------- dtype traits
// Each trait decodes one 16-byte chunk of A (VEC elements) against the matching
// XCH x 16 bytes of one x vector and accumulates into two fp32 partial sums (even
// and odd elements), in element order.
struct OpF32 {
  using TA = float;
  using TX = float;
  static constexpr int VEC = 4;
  static constexpr int XCH = 1;
  static constexpr int EPB = 1;        // elements per byte of A
  static constexpr bool GROUPED = false;  // per-group scales (int4)
  __device__ static __forceinline__ void dot(float &e, float &o, const uint4 &a, const uint4 *xv) {
    e = fmaf(__uint_as_float(a.x), __uint_as_float(xv[0].x), e);
    o = fmaf(__uint_as_float(a.y), __uint_as_float(xv[0].y), o);
    e = fmaf(__uint_as_float(a.z), __uint_as_float(xv[0].z), e);
    o = fmaf(__uint_as_float(a.w), __uint_as_float(xv[0].w), o);
  }
  __device__ static __forceinline__ void dot1(float &acc, const uint4 &a, const uint4 *xv) {
    acc = fmaf(__uint_as_float(a.x), __uint_as_float(xv[0].x), acc);
    acc = fmaf(__uint_as_float(a.y), __uint_as_float(xv[0].y), acc);
    acc = fmaf(__uint_as_float(a.z), __uint_as_float(xv[0].z), acc);
    acc = fmaf(__uint_as_float(a.w), __uint_as_float(xv[0].w), acc);
  }
  __device__ static __forceinline__ void quad2(const uint4 &a, int, float2 &q01, float2 &q23) {
    q01 = make_float2(__uint_as_float(a.x), __uint_as_float(a.y));
    q23 = make_float2(__uint_as_float(a.z), __uint_as_float(a.w));
  }
  // x elements 4w .. 4w+3 of the chunk, from x stored as fp32 at p (16 bytes).
  __device__ static __forceinline__ void xquad(const unsigned char *p, float (&q)[4]) {
    const float4 v = *reinterpret_cast<const float4 *>(p);
    q[0] = v.x; q[1] = v.y; q[2] = v.z; q[3] = v.w;
  }
  __device__ static __forceinline__ float a_elem(const void *A, int64_t i) {
    return __ldg(reinterpret_cast<const float *>(A) + i);
  }
  __device__ static __forceinline__ float x_elem(const void *x, int64_t i) {
    return __ldg(reinterpret_cast<const float *>(x) + i);
  }
  __device__ static __forceinline__ void store(void *y, int64_t i, float v) {
    reinterpret_cast<float *>(y)[i] = v;
  }
};

struct OpBF16 {
  using TA = __nv_bfloat16;
  using TX = __nv_bfloat16;
  static constexpr int VEC = 8;
  static constexpr int XCH = 1;
  static constexpr int EPB = 1;        // elements per byte of A
  static constexpr bool GROUPED = false;  // per-group scales (int4)
  __device__ static __forceinline__ void pair(float &e, float &o, uint32_t a, uint32_t x) {
    e = fmaf(bf16_lo(a), bf16_lo(x), e);
    o = fmaf(bf16_hi(a), bf16_hi(x), o);
  }
  // (e, o) as one fp32 pair, one packed FMA per word (same order as pair()).
  __device__ static __forceinline__ void dot(float &e, float &o, const uint4 &a, const uint4 *xv) {
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, xw[4] = {xv[0].x, xv[0].y, xv[0].z, xv[0].w};
    float2 acc = make_float2(e, o);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      acc = __ffma2_rn(make_float2(bf16_lo(aw[i]), bf16_hi(aw[i])), make_float2(bf16_lo(xw[i]), bf16_hi(xw[i])), acc);
    e = acc.x;
    o = acc.y;
  }
  // acc += a.lo * x.lo + a.hi * x.hi with the mixed-precision FMA (bf16 inputs,
  // fp32 accumulator): the bf16 product is exact in fp32, one rounding per FMA.
  __device__ static __forceinline__ void pair1(float &acc, uint32_t a, uint32_t x) {
    asm("{\n\t.reg .b16 al, ah, xl, xh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {xl, xh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, al, xl, %0;\n\tfma.rn.f32.bf16 %0, ah, xh, %0;\n\t}"
        : "+f"(acc) : "r"(a), "r"(x));
  }
  __device__ static __forceinline__ void dot1(float &acc, const uint4 &a, const uint4 *xv) {
    pair1(acc, a.x, xv[0].x);
    pair1(acc, a.y, xv[0].y);
    pair1(acc, a.z, xv[0].z);
    pair1(acc, a.w, xv[0].w);
  }
  // acc += a * x, bf16 operands, fp32 accumulator (the product is exact in fp32)
  __device__ static __forceinline__ void fma_mixed(float &acc, unsigned short a, unsigned short x) {
    asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a), "h"(x));
  }
  __device__ static __forceinline__ void quad2(const uint4 &a, int w, float2 &q01, float2 &q23) {
    const uint32_t u0 = w ? a.z : a.x, u1 = w ? a.w : a.y;
    q01 = make_float2(bf16_lo(u0), bf16_hi(u0));
    q23 = make_float2(bf16_lo(u1), bf16_hi(u1));
  }
  // 8 x values (16 bytes of bf16) as 4 fp32 pairs.
  __device__ static __forceinline__ void xpairs8(const uint4 &v, float2 (&p)[4]) {
    p[0] = make_float2(bf16_lo(v.x), bf16_hi(v.x));
    p[1] = make_float2(bf16_lo(v.y), bf16_hi(v.y));
    p[2] = make_float2(bf16_lo(v.z), bf16_hi(v.z));
    p[3] = make_float2(bf16_lo(v.w), bf16_hi(v.w));
  }
  // 4 bf16 x values (8 bytes at p) as fp32.
  __device__ static __forceinline__ void xquad(const unsigned char *p, float (&q)[4]) {
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    q[0] = bf16_lo(v.x); q[1] = bf16_hi(v.x); q[2] = bf16_lo(v.y); q[3] = bf16_hi(v.y);
  }
  __device__ static __forceinline__ float a_elem(const void *A, int64_t i) {
    return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16 *>(A) + i));
  }
  __device__ static __forceinline__ float x_elem(const void *x, int64_t i) {
    return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16 *>(x) + i));
  }
  __device__ static __forceinline__ void store(void *y, int64_t i, float v) {
    reinterpret_cast<__nv_bfloat16 *>(y)[i] = __float2bfloat16_rn(v);
  }
};

struct OpF16 {
  using TA = __half;
  using TX = __half;
  static constexpr int VEC = 8;
  static constexpr int XCH = 1;
  static constexpr int EPB = 1;        // elements per byte of A
  static constexpr bool GROUPED = false;  // per-group scales (int4)
  __device__ static __forceinline__ void pair(float &e, float &o, uint32_t a, uint32_t x) {
    float2 fa = f16x2_to_f2(a), fx = f16x2_to_f2(x);
    e = fmaf(fa.x, fx.x, e);
    o = fmaf(fa.y, fx.y, o);
  }
  // (e, o) as one fp32 pair, one packed FMA per word (same order as pair()).
  __device__ static __forceinline__ void dot(float &e, float &o, const uint4 &a, const uint4 *xv) {
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, xw[4] = {xv[0].x, xv[0].y, xv[0].z, xv[0].w};
    float2 acc = make_float2(e, o);
#pragma unroll
    for (int i = 0; i < 4; ++i) acc = __ffma2_rn(f16x2_to_f2(aw[i]), f16x2_to_f2(xw[i]), acc);
    e = acc.x;
    o = acc.y;
  }
  // acc += a.lo * x.lo + a.hi * x.hi with the mixed-precision FMA (fp16 inputs,
  // fp32 accumulator): the fp16 product is exact in fp32, one rounding per FMA.
  __device__ static __forceinline__ void pair1(float &acc, uint32_t a, uint32_t x) {
    asm("{\n\t.reg .b16 al, ah, xl, xh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {xl, xh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, xl, %0;\n\tfma.rn.f32.f16 %0, ah, xh, %0;\n\t}"
        : "+f"(acc) : "r"(a), "r"(x));
  }
  __device__ static __forceinline__ void dot1(float &acc, const uint4 &a, const uint4 *xv) {
    pair1(acc, a.x, xv[0].x);
    pair1(acc, a.y, xv[0].y);
    pair1(acc, a.z, xv[0].z);
    pair1(acc, a.w, xv[0].w);
  }
  // acc += a * x, fp16 operands, fp32 accumulator (the product is exact in fp32)
  __device__ static __forceinline__ void fma_mixed(float &acc, unsigned short a, unsigned short x) {
    asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(a), "h"(x));
  }
  __device__ static __forceinline__ void quad2(const uint4 &a, int w, float2 &q01, float2 &q23) {
    q01 = f16x2_to_f2(w ? a.z : a.x);
    q23 = f16x2_to_f2(w ? a.w : a.y);
  }
  // 8 x values (16 bytes of fp16) as 4 fp32 pairs.
  __device__ static __forceinline__ void xpairs8(const uint4 &v, float2 (&p)[4]) {
    p[0] = f16x2_to_f2(v.x);
    p[1] = f16x2_to_f2(v.y);
    p[2] = f16x2_to_f2(v.z);
    p[3] = f16x2_to_f2(v.w);
  }
  __device__ static __forceinline__ void xquad(const unsigned char *p, float (&q)[4]) {
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    const float2 f0 = f16x2_to_f2(v.x), f1 = f16x2_to_f2(v.y);
    q[0] = f0.x; q[1] = f0.y; q[2] = f1.x; q[3] = f1.y;
  }
  __device__ static __forceinline__ float a_elem(const void *A, int64_t i) {
    return __half2float(__ldg(reinterpret_cast<const __half *>(A) + i));
  }
  __device__ static __forceinline__ float x_elem(const void *x, int64_t i) {
    return __half2float(__ldg(reinterpret_cast<const __half *>(x) + i));
  }
  __device__ static __forceinline__ void store(void *y, int64_t i, float v) {
    reinterpret_cast<__half *>(y)[i] = __float2half_rn(v);
  }
};

// int8 weights, bf16 activations: 16 weights per 16-byte chunk meet 32 bytes of x.
struct OpW8 {
  using TA = int8_t;
  using TX = __nv_bfloat16;
  static constexpr int VEC = 16;
  static constexpr int XCH = 2;
  static constexpr int EPB = 1;        // elements per byte of A
  static constexpr bool GROUPED = false;  // per-group scales (int4)
  __device__ static __forceinline__ void word(float &e, float &o, uint32_t a, uint32_t x01,
                                              uint32_t x23) {
    const uint32_t f = a ^ 0x80808080u;
    e = fmaf(s8_to_f32<0>(f), bf16_lo(x01), e);
    o = fmaf(s8_to_f32<1>(f), bf16_hi(x01), o);
    e = fmaf(s8_to_f32<2>(f), bf16_lo(x23), e);
    o = fmaf(s8_to_f32<3>(f), bf16_hi(x23), o);
  }
  // (e, o) as one fp32 pair: each packed subtraction decodes two weights and each
  // packed FMA adds two products, in the same order per accumulator as word().
  __device__ static __forceinline__ void dot(float &e, float &o, const uint4 &a, const uint4 *xv) {
    float2 acc = make_float2(e, o);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      float2 q01, q23;
      quad2(a, w, q01, q23);
      const uint32_t x01 = (w & 1) ? (w < 2 ? xv[0].z : xv[1].z) : (w < 2 ? xv[0].x : xv[1].x);
      const uint32_t x23 = (w & 1) ? (w < 2 ? xv[0].w : xv[1].w) : (w < 2 ? xv[0].y : xv[1].y);
      acc = __ffma2_rn(q01, make_float2(bf16_lo(x01), bf16_hi(x01)), acc);
      acc = __ffma2_rn(q23, make_float2(bf16_lo(x23), bf16_hi(x23)), acc);
    }
    e = acc.x;
    o = acc.y;
  }
  __device__ static __forceinline__ void word1(float &acc, uint32_t a, uint32_t x01, uint32_t x23) {
    const uint32_t f = a ^ 0x80808080u;
    acc = fmaf(s8_to_f32<0>(f), bf16_lo(x01), acc);
    acc = fmaf(s8_to_f32<1>(f), bf16_hi(x01), acc);
    acc = fmaf(s8_to_f32<2>(f), bf16_lo(x23), acc);
    acc = fmaf(s8_to_f32<3>(f), bf16_hi(x23), acc);
  }
  __device__ static __forceinline__ void dot1(float &acc, const uint4 &a, const uint4 *xv) {
    word1(acc, a.x, xv[0].x, xv[0].y);
    word1(acc, a.y, xv[0].z, xv[0].w);
    word1(acc, a.z, xv[1].x, xv[1].y);
    word1(acc, a.w, xv[1].z, xv[1].w);
  }
  // the same magic-number decode, two weights per packed subtraction
  __device__ static __forceinline__ void quad2(const uint4 &a, int w, float2 &q01, float2 &q23) {
    const uint32_t u = w == 0 ? a.x : w == 1 ? a.y : w == 2 ? a.z : a.w;
    const uint32_t f = u ^ 0x80808080u;
    const float2 mg = make_float2(-8388736.0f, -8388736.0f);
    q01 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(f, 0x4B000000u, 0x7540)),
                                 __uint_as_float(__byte_perm(f, 0x4B000000u, 0x7541))), mg);
    q23 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(f, 0x4B000000u, 0x7542)),
                                 __uint_as_float(__byte_perm(f, 0x4B000000u, 0x7543))), mg);
  }
  // 8 x values (16 bytes of bf16) as 4 fp32 pairs.
  __device__ static __forceinline__ void xpairs8(const uint4 &v, float2 (&p)[4]) {
    p[0] = make_float2(bf16_lo(v.x), bf16_hi(v.x));
    p[1] = make_float2(bf16_lo(v.y), bf16_hi(v.y));
    p[2] = make_float2(bf16_lo(v.z), bf16_hi(v.z));
    p[3] = make_float2(bf16_lo(v.w), bf16_hi(v.w));
  }
  __device__ static __forceinline__ void xquad(const unsigned char *p, float (&q)[4]) {
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    q[0] = bf16_lo(v.x); q[1] = bf16_hi(v.x); q[2] = bf16_lo(v.y); q[3] = bf16_hi(v.y);
  }
  __device__ static __forceinline__ float a_elem(const void *A, int64_t i) {
    return (float)__ldg(reinterpret_cast<const signed char *>(A) + i);
  }
  __device__ static __forceinline__ float x_elem(const void *x, int64_t i) {
    return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16 *>(x) + i));
  }
  __device__ static __forceinline__ void store(void *y, int64_t i, float v) {
    reinterpret_cast<__nv_bfloat16 *>(y)[i] = __float2bfloat16_rn(v);
  }
};

// int4 weights, two per byte (even element in the low nibble), symmetric two's
// complement; one fp32 scale per group of 2^gshift consecutive elements of a row,
// applied once per 16-byte chunk (32 weights, inside one group: groups are at least
// 32 long); bf16 x, bias and y.  Decoding is the int8 magic number at nibble width:
// with u = q + 8 (nibbles XOR 8), the float with bits 0x4B0000uu is 2^23 + u, so
// subtracting 2^23 + 8 leaves q exactly.
struct OpW4 {
  using TA = uint8_t;
  using TX = __nv_bfloat16;
  static constexpr int VEC = 32;
  static constexpr int XCH = 4;
  static constexpr int EPB = 2;
  static constexpr bool GROUPED = true;
  // word a (elements 8w .. 8w+7) against their 8 bf16 x values
  __device__ static __forceinline__ void word(float2 &acc, uint32_t a, const uint4 &xw) {
    const uint32_t f = a ^ 0x88888888u;
    const uint32_t lo = f & 0x0F0F0F0Fu;          // elements 0, 2, 4, 6 in bytes 0..3
    const uint32_t hi = (f >> 4) & 0x0F0F0F0Fu;   // elements 1, 3, 5, 7
    const float2 mg = make_float2(-8388616.0f, -8388616.0f);
    const uint32_t xw4[4] = {xw.x, xw.y, xw.z, xw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 q = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7540 + j)),
                                              __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7540 + j))),
                                  mg);
      acc = __ffma2_rn(q, make_float2(bf16_lo(xw4[j]), bf16_hi(xw4[j])), acc);
    }
  }
  __device__ static __forceinline__ void dot(float &e, float &o, const uint4 &a, const uint4 *xv) {
    float2 acc = make_float2(e, o);
    word(acc, a.x, xv[0]);
    word(acc, a.y, xv[1]);
    word(acc, a.z, xv[2]);
    word(acc, a.w, xv[3]);
    e = acc.x;
    o = acc.y;
  }
  // elements 4w .. 4w+3 of a chunk as two fp32 pairs (unscaled): word w / 2, bytes
  // 2 (w % 2) and 2 (w % 2) + 1, low nibble first
  __device__ static __forceinline__ void quad2(const uint4 &a, int w, float2 &q01, float2 &q23) {
    const int j = w >> 1;
    const uint32_t word = j == 0 ? a.x : j == 1 ? a.y : j == 2 ? a.z : a.w;
    const uint32_t f = word ^ 0x88888888u;
    const uint32_t lo = f & 0x0F0F0F0Fu, hi = (f >> 4) & 0x0F0F0F0Fu;
    const uint32_t b0 = (uint32_t)(w & 1) * 2;
    const float2 mg = make_float2(-8388616.0f, -8388616.0f);
    q01 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7540 + b0)),
                                 __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7540 + b0))), mg);
    q23 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7541 + b0)),
                                 __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7541 + b0))), mg);
  }
  // element k of the row starting at byte `row` (unscaled)
  __device__ static __forceinline__ float nibble(const void *A, int64_t row_byte, int64_t k) {
    const uint32_t b = __ldg(reinterpret_cast<const unsigned char *>(A) + row_byte + (k >> 1));
    const int v = (int)((k & 1) ? (b >> 4) : (b & 15u));
    return (float)(v >= 8 ? v - 16 : v);
  }
  __device__ static __forceinline__ float x_elem(const void *x, int64_t i) {
    return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16 *>(x) + i));
  }
  __device__ static __forceinline__ void store(void *y, int64_t i, float v) {
    reinterpret_cast<__nv_bfloat16 *>(y)[i] = __float2bfloat16_rn(v);
  }
};

// Bytes of one row of A.
template <class Op>
__device__ __forceinline__ int64_t row_bytes(int64_t K) {
  return K * (int64_t)sizeof(typename Op::TA) / Op::EPB;
}

// The group scale of 16-byte chunk c of row `row` (1 for the ungrouped types).
template <class Op>
__device__ __forceinline__ float chunk_scale(const Args &a, int64_t row, int64_t c) {
  if constexpr (Op::GROUPED) {
    return __ldg(a.gscale + row * (a.K >> a.gshift) + ((c * Op::VEC) >> a.gshift));
  } else {
    return 1.f;
  }
}

// One chunk's products added to (e, o); a grouped type sums the chunk first and
// scales it once.
template <class Op>
__device__ __forceinline__ void dot_chunk(float &e, float &o, const uint4 &av, const uint4 *xv, float gs) {
  if constexpr (Op::GROUPED) {
    float le = 0.f, lo = 0.f;
    Op::dot(le, lo, av, xv);
    e = fmaf(gs, le, e);
    o = fmaf(gs, lo, o);
  } else {
    Op::dot(e, o, av, xv);
  }
}

// Element (row, k) of A as a float, with its group scale (element-load paths).
template <class Op>
__device__ __forceinline__ float a_value(const Args &a, int64_t row, int64_t k) {
  if constexpr (Op::GROUPED) {
    return __ldg(a.gscale + row * (a.K >> a.gshift) + (k >> a.gshift)) *
           Op::nibble(a.A, row * (a.K >> 1), k);
  } else {
    return Op::a_elem(a.A, row * a.K + k);
  }
}

// bias is stored in the output type: fp32 for OpF32, otherwise the x type.
template <class Op>
__device__ __forceinline__ float bias_at(const void *bias, int64_t m) {
  return Op::x_elem(bias, m);
}

// SiLU(v) = v / (1 + e^-v), in fp32 with the CUDA math library's expf.
__device__ __forceinline__ float silu(float v) { return v / (1.0f + expf(-v)); }

// Row m of vector b before any activation: s_m * acc + bias[m].
template <class Op>
__device__ __forceinline__ float row_value(const Args &a, int64_t m, float acc) {
  float v = acc;
  if (a.scale != nullptr) v *= __ldg(a.scale + m);
  if (a.bias != nullptr) v += bias_at<Op>(a.bias, m);
  return v;
}

// y = act(s_m * acc + bias[m]) + residual[b][m], rounded once to the output type
// (lesson 3's epilogue adds the bias in fp32 after the reduction, NULL allowed;
// the NPU MatMul post, section 5.1, fuses bias, activation and residual into the
// MatMul instead of separate passes over y).
// The residual may be y itself (in place): a plain, coherent load, not the
// read-only path.
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <class Op>
__device__ __forceinline__ float residual_at(const void *r, int64_t i) {
  return to_f32(reinterpret_cast<const typename Op::TX *>(r)[i]);
}

// act(v) + res, rounded once to the output type, stored at y[i].
template <class Op>
__device__ __forceinline__ void store_act_res(const Args &a, int64_t i, float v, float res) {
  if (a.act == 1) v = silu(v);
  if (a.residual != nullptr) v += res;
  Op::store(a.y, i, v);
}

// (The residual is read after the arithmetic, through the read-only path: each
// output is read and then written by the one thread that owns it and by no other,
// so even in place the value read is the caller's.)
template <class Op>
__device__ __forceinline__ void epilogue_store(const Args &a, int b, int64_t m, float acc) {
  float v = row_value<Op>(a, m, acc);
  if (a.act == 1) v = silu(v);
  const int64_t i = (int64_t)b * a.M + m;
  if (a.residual != nullptr) v += Op::x_elem(a.residual, i);
  Op::store(a.y, i, v);
}

// A row's epilogue operands, loaded when the row's first A loads are issued so
// that they arrive while the row streams instead of after its reduction: the
// scale, the bias and (RES) vector 0's residual, all in registers.
struct RowPre {
  float s, bias, res;
};

template <class Op, bool RES>
__device__ __forceinline__ RowPre row_pre(const Args &a, int64_t m, bool live) {
  RowPre p{1.f, 0.f, 0.f};
  if (live) {
    if (a.scale != nullptr) p.s = __ldg(a.scale + m);
    if (a.bias != nullptr) p.bias = bias_at<Op>(a.bias, m);
    if (RES && a.residual != nullptr) p.res = residual_at<Op>(a.residual, m);
  }
  return p;
}

// s_m * acc + bias[m] from prefetched operands (the same operations as row_value).
template <class Op>
__device__ __forceinline__ float row_value_pre(const Args &a, const RowPre &p, float acc) {
  float v = acc;
  if (a.scale != nullptr) v *= p.s;
  if (a.bias != nullptr) v += p.bias;
  return v;
}

// SwiGLU output m of vector b from the gate row m and the up row m + half.
template <class Op>
__device__ __forceinline__ void epilogue_swiglu(const Args &a, int b, int64_t m, float acc_gate,
                                                float acc_up) {
  const float g = row_value<Op>(a, m, acc_gate);
  const float u = row_value<Op>(a, m + a.half, acc_up);
  Op::store(a.y, (int64_t)b * a.half + m, silu(g) * u);
}

// Butterfly over WIDTH lanes: every lane of each WIDTH-lane group ends with the
// group's sum, groups never mix (xor offsets < WIDTH stay inside the group).
template <int WIDTH>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int off = WIDTH / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// ------------------------------------------------------------------ k_rowteam
// TPR lanes per row, kThreads / TPR rows per CTA per pass, grid-stride over row
// groups.  Lanes of a row take 16-byte chunks TPR apart (so a warp's loads are
// contiguous), U chunks issued before any is consumed.  All 32 lanes of a warp
// reach the butterfly, with rows past M contributing zeros.
template <class Op, int TPR, int NB, int U, bool VEC, int THREADS = kThreads>
__global__ void __launch_bounds__(THREADS) k_rowteam(const Args a) {
  pdl_enter(a, false);
  constexpr int TEAMS = THREADS / TPR;
  const int sub = threadIdx.x & (TPR - 1);
  const int team = threadIdx.x / TPR;
  const int64_t M = a.M, K = a.K;
  const int B = a.B;
  const uint64_t pol = evict_first_policy();
  constexpr int XB = Op::XCH * 16;  // bytes of one x vector per A chunk

  for (int64_t base = (int64_t)blockIdx.x * TEAMS; base < M; base += (int64_t)gridDim.x * TEAMS) {
    const int64_t row = base + team;
    const bool live = row < M;
    // operands loaded ahead of the A loads (not for fp32 rows: measured slower there)
    constexpr bool kPre = sizeof(typename Op::TA) != 4;
    const RowPre pre = kPre ? row_pre<Op, NB == 1>(a, row, live) : RowPre{1.f, 0.f, 0.f};
    float e[NB], o[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) e[b] = o[b] = 0.f;

    if (VEC) {
      const int64_t nch = live ? K / Op::VEC : 0;
      const char *arow = reinterpret_cast<const char *>(a.A) + row * row_bytes<Op>(K);
      const char *xb0 = reinterpret_cast<const char *>(a.x);
      const int64_t xstride = K * (int64_t)sizeof(typename Op::TX);
      for (int64_t c0 = sub; c0 < nch; c0 += (int64_t)TPR * U) {
        uint4 av[U];
        float gs[Op::GROUPED ? U : 1];  // group scales (int4 only)
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t c = c0 + (int64_t)u * TPR;
          av[u] = (c < nch) ? ld_stream16(arow + c * 16, pol) : make_uint4(0, 0, 0, 0);
          if constexpr (Op::GROUPED) gs[u] = (c < nch) ? chunk_scale<Op>(a, row, c) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t c = c0 + (int64_t)u * TPR;
          if (c < nch) {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              if (b < B) {
                uint4 xv[Op::XCH];
#pragma unroll
                for (int h = 0; h < Op::XCH; ++h) xv[h] = ld_x16(xb0 + b * xstride + c * XB + h * 16);
                dot_chunk<Op>(e[b], o[b], av[u], xv, Op::GROUPED ? gs[Op::GROUPED ? u : 0] : 1.f);
              }
            }
          }
        }
      }
    } else {
      const int64_t kend = live ? K : 0;
      for (int64_t k = sub; k < kend; k += TPR) {
        const float av = a_value<Op>(a, row, k);
#pragma unroll
        for (int b = 0; b < NB; ++b)
          if (b < B) e[b] = fmaf(av, Op::x_elem(a.x, (int64_t)b * K + k), e[b]);
      }
    }

#pragma unroll
    for (int b = 0; b < NB; ++b) e[b] = group_sum<TPR>(e[b] + o[b]);
    if (live && sub == 0) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b < B) {
          const int64_t i = (int64_t)b * M + row;
          if (kPre) {
            const float res = NB == 1 ? pre.res : (a.residual != nullptr ? residual_at<Op>(a.residual, i) : 0.f);
            store_act_res<Op>(a, i, row_value_pre<Op>(a, pre, e[b]), res);
          } else {
            epilogue_store<Op>(a, b, row, e[b]);
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------------ k_blockrow
// One CTA per row (grid-stride over rows); blockIdx.y selects a K slice when the
// row is split.  Partial sums: warp butterflies, then warp 0 adds the 8 warp
// totals in warp order.  splits == 1 finishes the row here; otherwise the slice
// total goes to partial[(slice * B + b) * M + row] for k_splitk_reduce.
template <class Op, int NB, int U>
__global__ void __launch_bounds__(kThreads) k_blockrow(const Args a, float *partial,
                                                       int64_t chunks_per_split) {
  pdl_enter(a, false);
  __shared__ float red[NB][kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t M = a.M, K = a.K;
  const int B = a.B;
  const uint64_t pol = evict_first_policy();
  constexpr int XB = Op::XCH * 16;
  const int64_t nch_all = K / Op::VEC;
  const int64_t c_lo = (int64_t)blockIdx.y * chunks_per_split;
  const int64_t c_hi = min(nch_all, c_lo + chunks_per_split);
  const char *xb0 = reinterpret_cast<const char *>(a.x);
  const int64_t xstride = K * (int64_t)sizeof(typename Op::TX);

  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const char *arow = reinterpret_cast<const char *>(a.A) + row * row_bytes<Op>(K);
    float e[NB], o[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) e[b] = o[b] = 0.f;
    for (int64_t c0 = c_lo + tid; c0 < c_hi; c0 += (int64_t)kThreads * U) {
      uint4 av[U];
      float gs[Op::GROUPED ? U : 1];  // group scales (int4 only)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t c = c0 + (int64_t)u * kThreads;
        av[u] = (c < c_hi) ? ld_stream16(arow + c * 16, pol) : make_uint4(0, 0, 0, 0);
        if constexpr (Op::GROUPED) gs[u] = (c < c_hi) ? chunk_scale<Op>(a, row, c) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t c = c0 + (int64_t)u * kThreads;
        if (c < c_hi) {
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            if (b < B) {
              uint4 xv[Op::XCH];
#pragma unroll
              for (int h = 0; h < Op::XCH; ++h) xv[h] = ld_x16(xb0 + b * xstride + c * XB + h * 16);
              dot_chunk<Op>(e[b], o[b], av[u], xv, Op::GROUPED ? gs[Op::GROUPED ? u : 0] : 1.f);
            }
          }
        }
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float w = group_sum<32>(e[b] + o[b]);
      if (lane == 0) red[b][warp] = w;
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b < B && lane == 0) {
          float s = 0.f;
#pragma unroll
          for (int w = 0; w < kWarps; ++w) s += red[b][w];
          if (partial == nullptr) {
            epilogue_store<Op>(a, b, row, s);
          } else {
            partial[((int64_t)blockIdx.y * B + b) * M + row] = s;
          }
        }
      }
    }
    __syncthreads();  // red[] is reused by the next row
  }
}

// Split-K pass 2: one thread per (b, m), vector b = blockIdx.y; slices summed in
// index order.
template <class Op>
__global__ void __launch_bounds__(kThreads) k_splitk_reduce(const Args a, const float *partial,
                                                            int splits) {
  pdl_enter(a, false);  // the partial sums come from the kernel before
  const int64_t M = a.M;
  const int b = (int)blockIdx.y;
  for (int64_t m = (int64_t)blockIdx.x * kThreads + threadIdx.x; m < M; m += (int64_t)gridDim.x * kThreads) {
    float s = 0.f;
    for (int j = 0; j < splits; ++j) s += partial[((int64_t)j * a.B + b) * M + m];
    epilogue_store<Op>(a, b, m, s);
  }
}

// The two 16-bit halves of a word (low half = lower element).
__device__ __forceinline__ void split_halves(uint32_t w, unsigned short &lo, unsigned short &hi) {
  asm("mov.b32 {%0, %1}, %2;" : "=h"(lo), "=h"(hi) : "r"(w));
}

// NB values per lane summed over the 32 lanes of a warp.  The first log2(NB)
// steps halve the values each lane carries (it keeps one half and receives the
// partner's copy of it), the rest are plain xor steps.  Lane l ends with the total
// of value l >> (5 - log2 NB).
template <int NB>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[NB], int lane) {
#pragma unroll
  for (int h = NB / 2, m = 16; h >= 1; h >>= 1, m >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = upper ? v[i] : v[i + h];
      const float keep = upper ? v[i + h] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  float t = v[0];
#pragma unroll
  for (int m = 16 / NB; m >= 1; m >>= 1) t += __shfl_xor_sync(0xffffffffu, t, m);
  return t;
}

// ------------------------------------------------------------------ k_batched2
// 2 <= B <= 16.  x[0..B) copied once per CTA into shared memory as stored, with
// vectors B..NB-1 zero, so the inner loops run over all NB vectors without a
// branch.  Each warp carries R rows and takes U chunks of each per step; the
// next step's loads (possibly of the warp's next row group) are in flight while
// the current step is used.  Every x chunk read from shared memory feeds R rows.
// fp16/bf16: one fp32 accumulator per (row, vector) and mixed-precision FMAs (16-bit
// operands, fp32 accumulator).  int8/fp32 with up to 8 vectors: an (even, odd) fp32
// pair per (row, vector) and packed FMAs; with 16, one accumulator and scalar FMAs.
// The R * NB sums meet in one reduce-scatter butterfly.
template <class Op, int NB, int R, int U, int THREADS, bool SW = false>
__global__ void __launch_bounds__(THREADS, 1) k_batched2(const Args a) {
  pdl_enter(a, true);
  static_assert(!SW || R == 2, "SwiGLU pairs the gate and up row of one output");
  extern __shared__ __align__(16) unsigned char xs[];
  constexpr int WARPS = THREADS / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t M = a.M, K = a.K;
  const int B = a.B;
  constexpr int XB = Op::XCH * 16;  // smem bytes of x per A chunk
  constexpr bool kMixed16 = sizeof(typename Op::TA) == 2 && sizeof(typename Op::TX) == 2;
  // fp32 and int8 rows with up to 8 vectors: (even, odd) accumulator pairs and packed
  // FMAs (int8 with the packed magic-number decode); 16 vectors keep one accumulator
  constexpr bool kF32 = sizeof(typename Op::TA) == 4;
  constexpr bool kPacked = (kF32 || (sizeof(typename Op::TA) == 1 && !Op::GROUPED)) && NB <= 8;
  const int64_t xstride = K * (int64_t)sizeof(typename Op::TX);
  const uint64_t pol = evict_first_policy();
  const int64_t nch = K / Op::VEC;
  const int64_t rowb = K * (int64_t)sizeof(typename Op::TA);
  const char *A = reinterpret_cast<const char *>(a.A);
  // row r of group g: g * R + r, or with SW the gate row g and the up row g + half
  const int64_t groups = SW ? a.half : (M + R - 1) / R;
  auto row_of = [&](int64_t gg, int r) -> int64_t { return SW ? gg + r * a.half : gg * R + r; };
  const int64_t gstride = (int64_t)gridDim.x * WARPS;

  // row groups of R rows dealt to CTAs round-robin: every SM gets an equal share
  int64_t g = blockIdx.x + (int64_t)gridDim.x * warp;
  int64_t base = 0;  // first chunk of the step, the same in every lane of the warp
  // the rows of the group being prefetched: this lane's chunk-0 address in each and
  // which exist, set once per row group
  const char *nrow[R];
  uint32_t nlive = 0;
  auto set_rows = [&](int64_t gg) {
    nlive = 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int64_t row = row_of(gg, r);
      const bool ok = gg < groups && row < M;
      nlive |= (ok ? 1u : 0u) << r;
      nrow[r] = A + (ok ? row * rowb : 0) + lane * 16;
    }
  };
  auto prefetch = [&](uint4 (&dst)[U][R]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool in = base + lane + 32 * u < nch;
#pragma unroll
      for (int r = 0; r < R; ++r)
        dst[u][r] = (in && (nlive & (1u << r))) ? ld_stream16(nrow[r] + (base + 32 * u) * 16, pol)
                                                : make_uint4(0, 0, 0, 0);
    }
  };
  set_rows(g);
  uint4 nxt[U][R];
  prefetch(nxt);
  pdl_after_prefetch(a);
  {
    const int64_t n16 = (xstride * B) / 16, nz16 = (xstride * NB) / 16;
    const char *src = reinterpret_cast<const char *>(a.x);
    for (int64_t i = tid; i < n16; i += THREADS) cp_async16(xs + i * 16, src + i * 16);
    for (int64_t i = n16 + tid; i < nz16; i += THREADS)
      reinterpret_cast<uint4 *>(xs)[i] = make_uint4(0, 0, 0, 0);
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    __syncthreads();
  }

  while (g < groups) {
    float acc[R][NB];
    float2 acc2[kPacked ? R : 1][kPacked ? NB : 1];  // kPacked: (even, odd) element sums
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[r][b] = 0.f;
    if constexpr (kPacked) {
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc2[r][b] = make_float2(0.f, 0.f);
    }
    int64_t ng;
    for (;;) {
      uint4 cur[U][R];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int r = 0; r < R; ++r) cur[u][r] = nxt[u][r];
      const int64_t cb = base + lane;
      ng = g;
      base += 32 * U;
      if (base >= nch) {
        ng = g + gstride;
        base = 0;
        set_rows(ng);
      }
      prefetch(nxt);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t c = cb + 32 * u;
        if (c < nch) {
          if constexpr (kMixed16) {
            // 16-bit A and x: each A half split out once per row, each x half once
            // per vector, then one mixed-precision FMA per product, in element order
            unsigned short ah[R][8];
#pragma unroll
            for (int r = 0; r < R; ++r) {
              split_halves(cur[u][r].x, ah[r][0], ah[r][1]);
              split_halves(cur[u][r].y, ah[r][2], ah[r][3]);
              split_halves(cur[u][r].z, ah[r][4], ah[r][5]);
              split_halves(cur[u][r].w, ah[r][6], ah[r][7]);
            }
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              const uint4 xv = *reinterpret_cast<const uint4 *>(xs + b * xstride + c * XB);
              unsigned short xh[8];
              split_halves(xv.x, xh[0], xh[1]);
              split_halves(xv.y, xh[2], xh[3]);
              split_halves(xv.z, xh[4], xh[5]);
              split_halves(xv.w, xh[6], xh[7]);
#pragma unroll
              for (int r = 0; r < R; ++r)
#pragma unroll
                for (int e = 0; e < 8; ++e) Op::fma_mixed(acc[r][b], ah[r][e], xh[e]);
            }
          } else {
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              const unsigned char *xp = xs + b * xstride + c * XB;
              uint4 xv[Op::XCH];
#pragma unroll
              for (int h = 0; h < Op::XCH; ++h) xv[h] = reinterpret_cast<const uint4 *>(xp)[h];
#pragma unroll
              for (int r = 0; r < R; ++r) {
                if constexpr (kPacked && kF32) {
                  const uint4 &av = cur[u][r];
                  acc2[r][b] = __ffma2_rn(make_float2(__uint_as_float(av.x), __uint_as_float(av.y)),
                                          make_float2(__uint_as_float(xv[0].x), __uint_as_float(xv[0].y)), acc2[r][b]);
                  acc2[r][b] = __ffma2_rn(make_float2(__uint_as_float(av.z), __uint_as_float(av.w)),
                                          make_float2(__uint_as_float(xv[0].z), __uint_as_float(xv[0].w)), acc2[r][b]);
                } else if constexpr (kPacked) {
                  Op::dot(acc2[r][b].x, acc2[r][b].y, cur[u][r], xv);  // int8: packed decode and FMAs
                } else {
                  Op::dot1(acc[r][b], cur[u][r], xv);
                }
              }
            }
          }
        }
      }
      if (ng != g) break;
    }
    // the R * NB sums by reduce-scatter butterflies of V <= 32 sums (RH rows each):
    // in butterfly h, lane l ends with sum l >> (5 - log2 V) (row h * RH + index /
    // NB, vector index % NB), replicated over 32 / V lanes
    constexpr int V = R * NB > 32 ? 32 : R * NB, RH = V / NB;
    constexpr int LOGV = V == 32 ? 5 : V == 16 ? 4 : V == 8 ? 3 : V == 4 ? 2 : 1;
    static_assert((1 << LOGV) == V && R % RH == 0, "R * NB must be a power of two");
    const int idx = lane >> (5 - LOGV);
    const bool owner = (lane & ((32 >> LOGV) - 1)) == 0;
#pragma unroll
    for (int h = 0; h < R / RH; ++h) {
      float v[V];
#pragma unroll
      for (int r = 0; r < RH; ++r)
#pragma unroll
        for (int b = 0; b < NB; ++b)
          v[r * NB + b] = kPacked ? acc2[h * RH + r][b].x + acc2[h * RH + r][b].y : acc[h * RH + r][b];
      const float part = warp_reduce_scatter<V>(v, lane);
      if constexpr (SW) {
        // gate sum b (row 0) sits at lane b * 32 / V, its up sum (row 1) 16 lanes above
        const float up = __shfl_down_sync(0xffffffffu, part, 16);
        if (owner && idx < NB && idx < B) epilogue_swiglu<Op>(a, idx, g, part, up);
      } else {
        const int r = h * RH + idx / NB, b = idx % NB;
        if (owner && b < B && g * R + r < M) epilogue_store<Op>(a, b, g * R + r, part);
      }
    }
    g = ng;
  }
}

// ------------------------------------------------------------------ k_stream
// B = 1, rows of at least one chunk per lane: persistent warps, one row at a time
// per warp, U chunks per lane in flight, double-buffered across row boundaries
// (the next row's first loads are issued before the current row is reduced), so
// a warp never waits on an empty pipeline between rows.  Rows are dealt to CTAs
// round-robin so that every SM gets an equal share.  x is read through L1
// (XSM = 0), or from shared memory where the CTA copies it once: as stored (1), or
// widened to fp32 (2) in quad planes [w][c][4] (lanes read consecutive 16-byte
// words), so that no lane widens an x element per row.
// CTAs per SM the stream plan launches (4 for fp32 rows, 2 otherwise): the
// register budget must let them all be resident.
template <class Op>
constexpr int stream_ctas_per_sm() { return sizeof(typename Op::TA) == 4 ? 4 : 2; }

template <class Op, int U, int THREADS, int XSM, bool SW = false, int CPS = stream_ctas_per_sm<Op>()>
__global__ void __launch_bounds__(THREADS, CPS) k_stream(const Args a) {
  // (fp32 rows run at the 32-register cap: they take no weight prefetch, which
  // would cost registers across the prologue)
  constexpr bool kPrefetch = sizeof(typename Op::TA) != 4;
  pdl_enter(a, kPrefetch);
  extern __shared__ __align__(16) unsigned char xs[];
  constexpr bool XS = XSM != 0;
  static_assert(XSM != 2 || sizeof(typename Op::TX) == 2, "fp32 staging widens 16-bit x");
  constexpr int WARPS = THREADS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t M = a.M, K = a.K;
  constexpr int XB = Op::XCH * 16;
  const unsigned char *xb = XS ? xs : reinterpret_cast<const unsigned char *>(a.x);
  const uint64_t pol = evict_first_policy();
  const int64_t nch = K / Op::VEC;
  const int64_t rstride = (int64_t)gridDim.x * WARPS;
  const int64_t rowb = row_bytes<Op>(K);
  const char *A = reinterpret_cast<const char *>(a.A);

  // `row` and `base` (first chunk of the current load group) are the same in all
  // lanes of a warp, so every lane leaves a row at the same step.  With SW
  // (M = 2 * half) the warp walks pairs: gate row p, then up row p + half, then
  // gate row p + rstride; once the next pair index reaches half, the row becomes
  // M, which ends the loop.
  const int64_t half = a.half;
  auto next_row = [&](int64_t r) -> int64_t {
    if (!SW) return r + rstride;
    if (r < half) return r + half;                 // gate -> its up row
    const int64_t np = r - half + rstride;         // up -> next pair's gate row
    return np < half ? np : M;
  };
  auto row_live = [&](int64_t r) -> bool { return r < M; };
  int64_t row = blockIdx.x + (int64_t)gridDim.x * warp;
  if (SW && row >= half) row = M;  // a pair index past the last pair: no work
  int64_t unit = warp;  // the row's (pair's) unit index in the CTA: warp + WARPS * j
  int64_t base = 0;
  float gate_val = 0.f;
  uint4 buf[U];
  float gbuf[Op::GROUPED ? U : 1];  // group scales of the chunks in buf (int4 only)
  // prologue: first group of the first row
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t c = base + lane + 32 * u;
    buf[u] = (row_live(row) && c < nch) ? ld_stream16(A + row * rowb + c * 16, pol) : make_uint4(0, 0, 0, 0);
    if constexpr (Op::GROUPED) gbuf[u] = (row_live(row) && c < nch) ? chunk_scale<Op>(a, row, c) : 0.f;
  }
  if constexpr (kPrefetch) pdl_after_prefetch(a);
  // x is copied into shared memory (as stored) while those loads are in flight;
  // one barrier below covers it and the epilogue operands.
  if constexpr (XSM == 1) {
    const int64_t n16 = nch * Op::XCH;
    const char *src = reinterpret_cast<const char *>(a.x);
    for (int64_t i = threadIdx.x; i < n16; i += THREADS) cp_async16(xs + i * 16, src + i * 16);
    asm volatile("cp.async.commit_group;" ::: "memory");
  } else if constexpr (XSM == 2) {
    // quad q (elements 4q..4q+3) of chunk c = 4q / VEC, quad w = (4q % VEC) / 4 goes to
    // plane w, word c; eight quads per thread in flight at a time
    const int64_t nq = K / 4;
    const uint2 *src = reinterpret_cast<const uint2 *>(a.x);
    for (int64_t q0 = threadIdx.x; q0 < nq; q0 += 8 * THREADS) {
      uint2 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t q = q0 + (int64_t)u * THREADS;
        v[u] = q < nq ? src[q] : make_uint2(0, 0);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t q = q0 + (int64_t)u * THREADS;
        if (q < nq) {
          float f[4];
          widen4(v[u].x, v[u].y, f, typename Op::TX());
          const int64_t c = (4 * q) / Op::VEC, w = ((4 * q) % Op::VEC) / 4;
          *reinterpret_cast<float4 *>(xs + (w * nch + c) * 16) = make_float4(f[0], f[1], f[2], f[3]);
        }
      }
    }
  }
  // The epilogue operands of the CTA's first THREADS rows (pairs with SW) are
  // staged in shared memory too, so that no row waits on a bias, scale or residual
  // load after its reduction.  The j-th row of warp w is unit t = w + WARPS * j of
  // the CTA: row (or pair) blockIdx.x + gridDim.x * t.
  // (fp32 rows run four CTAs per SM at 32 registers: they load the operands after
  // the reduction instead, which measured faster than the staging's extra registers)
  constexpr bool kStage = sizeof(typename Op::TA) != 4;
  __shared__ float ops[4][kStage ? THREADS : 1];
  const bool staged = kStage && (a.bias != nullptr || a.scale != nullptr || a.residual != nullptr);
  if (kStage && staged) {
    const int t = threadIdx.x;
    const int64_t r = blockIdx.x + (int64_t)gridDim.x * t;
    if (SW ? r < half : r < M) {
      if (SW) {
        ops[0][t] = a.bias != nullptr ? bias_at<Op>(a.bias, r) : 0.f;
        ops[1][t] = a.scale != nullptr ? __ldg(a.scale + r) : 1.f;
        ops[2][t] = a.bias != nullptr ? bias_at<Op>(a.bias, r + half) : 0.f;
        ops[3][t] = a.scale != nullptr ? __ldg(a.scale + r + half) : 1.f;
      } else {
        ops[0][t] = a.bias != nullptr ? bias_at<Op>(a.bias, r) : 0.f;
        ops[1][t] = a.scale != nullptr ? __ldg(a.scale + r) : 1.f;
        ops[2][t] = a.residual != nullptr ? residual_at<Op>(a.residual, r) : 0.f;
      }
    }
  }
  if (XSM == 1) asm volatile("cp.async.wait_group 0;" ::: "memory");
  if (XS || staged) __syncthreads();
  while (row_live(row)) {
    float e = 0.f, o = 0.f;
    for (;;) {
      uint4 cur[U];
      float gcur[Op::GROUPED ? U : 1];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        cur[u] = buf[u];
        if constexpr (Op::GROUPED) gcur[u] = gbuf[u];
      }
      const int64_t cc = base + lane;
      // next group: same row, or the first group of this warp's next row (whose
      // epilogue operand is fetched with it)
      int64_t nrow = row;
      base += 32 * U;
      if (base >= nch) { nrow = next_row(row); base = 0; }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t c = base + lane + 32 * u;
        buf[u] = (row_live(nrow) && c < nch) ? ld_stream16(A + nrow * rowb + c * 16, pol) : make_uint4(0, 0, 0, 0);
        if constexpr (Op::GROUPED) gbuf[u] = (row_live(nrow) && c < nch) ? chunk_scale<Op>(a, nrow, c) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t c = cc + 32 * u;
        if (c < nch) {
          if constexpr (XSM == 2) {
            // quads in element order, (even, odd) pairs: the same sums as dot_chunk
            float2 acc = make_float2(0.f, 0.f);
            if constexpr (!Op::GROUPED) acc = make_float2(e, o);
#pragma unroll
            for (int w = 0; w < Op::VEC / 4; ++w) {
              float2 q01, q23;
              Op::quad2(cur[u], w, q01, q23);
              const float4 xq = *reinterpret_cast<const float4 *>(xs + (w * nch + c) * 16);
              acc = __ffma2_rn(q01, make_float2(xq.x, xq.y), acc);
              acc = __ffma2_rn(q23, make_float2(xq.z, xq.w), acc);
            }
            if constexpr (Op::GROUPED) {
              const float gs = gcur[Op::GROUPED ? u : 0];
              e = fmaf(gs, acc.x, e);
              o = fmaf(gs, acc.y, o);
            } else {
              e = acc.x;
              o = acc.y;
            }
          } else {
            uint4 xv[Op::XCH];
#pragma unroll
            for (int h = 0; h < Op::XCH; ++h)
              xv[h] = XS ? *reinterpret_cast<const uint4 *>(xb + c * XB + h * 16) : ld_x16(xb + c * XB + h * 16);
            dot_chunk<Op>(e, o, cur[u], xv, Op::GROUPED ? gcur[Op::GROUPED ? u : 0] : 1.f);
          }
        }
      }
      if (nrow != row) break;
    }
    const float s = group_sum<32>(e + o);
    if (lane == 0) {
      const bool up = SW && row >= half;
      const int64_t t = kStage ? unit : 0;
      RowPre p{1.f, 0.f, 0.f};
      if (kStage && staged && t < THREADS) {
        p.bias = ops[up ? 2 : 0][t];
        p.s = ops[up ? 3 : 1][t];
        if (!SW) p.res = ops[2][t];
      } else {
        p = row_pre<Op, !SW>(a, row, true);
      }
      const float v = row_value_pre<Op>(a, p, s);
      if (!SW) store_act_res<Op>(a, row, v, p.res);
      else if (!up) gate_val = v;
      else Op::store(a.y, row - half, silu(gate_val) * v);
    }
    if (!SW || row >= half) unit += WARPS;  // (with SW: after the pair's up row)
    row = next_row(row);
  }
}

// ------------------------------------------------------------------ k_xsplit
// B <= 4 (NB in {1, 2, 4}): the 512 threads of a CTA split K.  Thread L (= warp *
// 32 + lane) owns chunks c = L + 512 j (j < J) of every row and keeps x for those
// chunks, all NB vectors, in fp32 registers for the whole kernel: x is never read
// from shared memory and never widened twice.  A CTA takes a contiguous block of
// rows (balanced to within one); each thread copies its own chunks of the coming
// rows into its own shared-memory slots with cp.async, P rows per commit group and
// G groups in flight (P * G rows, P * G * J * 8 KB per SM, at no register cost),
// and reads back only what it copied (no barrier for A).  Per row, each warp
// reduces its NB partial sums with a reduce-scatter butterfly and leaves them in
// red[]; every kXsT rows one barrier, then kXsT * NB threads add the 16 warp
// partials in warp order and run the epilogue.  Fixed orders throughout: results
// are reproducible.
constexpr int kXsThreads = 512;
constexpr int kXsWarps = kXsThreads / 32;
constexpr int kXsT = 16;  // rows per barrier (a multiple of P)

// ------------------------------------------------------------------ k_batch_ring
// 2 <= B <= 16 (NB in {2, 4, 8, 16}).  One 512-thread CTA per SM, persistent; each
// warp carries R rows at a time (row groups dealt round-robin over CTAs and warps,
// so every SM gets an equal share).
// - A streams through a per-thread cp.async ring in shared memory: at step j of a
//   row group, lane l uses chunk 32j + l of each of the R rows.  Every step is one
//   commit group, issued G steps ahead (across row-group boundaries), and a lane
//   reads back only the slots it filled itself, so A needs no barrier and no
//   registers while in flight.
// - x[0..NB) is staged once per CTA, fp32 when it fits (XE = 4) else as stored, in
//   planes of 16-byte words indexed by chunk, so that the lanes of a warp
//   (consecutive chunks) read consecutive words: no bank conflicts.  Vectors
//   B..NB-1 are zero.
// - NB <= 4: (even, odd) accumulator pairs per (row, vector); a plane holds one
//   vector's quad w of every chunk.  NB >= 8 (PAIRS): one accumulator pair per
//   (row, vector pair), i.e. vectors 2p and 2p + 1, which halves the accumulator
//   registers; a plane holds vector pair p interleaved element by element
//   (x[2p][k], x[2p+1][k]) and each A element is broadcast to both halves.  Either
//   way each A element is widened once and meets all NB vectors through packed
//   FMAs, and every sum is taken in element order.
// - A row group's R * NB sums are reduced by one reduce-scatter butterfly, after
//   which lane l holds sum l (row l / NB, vector l % NB, replicated over 32 / (R*NB)
//   lanes) and runs its epilogue, with the operands it loaded when the group began.
// SW (R = 2): the two rows are SwiGLU's gate row g and up row g + half.

__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds8(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// inner-loop forms of k_batch_ring
constexpr int kRingEvenOdd = 0;  // (even, odd) accumulator pairs per (row, vector)
constexpr int kRingPairs = 1;    // one accumulator pair per (row, vector pair)
constexpr int kRingMixed = 2;    // one fp32 accumulator per (row, vector), 16-bit operands

template <class Op, int NB, int R, int G, int XE, bool SW, int MODE = (NB >= 8 ? kRingPairs : kRingEvenOdd),
          int THREADS = 512>
__global__ void __launch_bounds__(THREADS, 1) k_batch_ring(const Args a, float *partial,
                                                           int64_t chunks_per_split) {
  pdl_enter(a, true);
  constexpr int WARPS = THREADS / 32;
  constexpr bool PAIRS = MODE == kRingPairs;
  static_assert(MODE != kRingMixed || (XE == 2 && Op::VEC == 8), "mixed FMAs take 16-bit A and x");
  constexpr int NP = NB / 2;                      // vector pairs
  constexpr int QW = Op::VEC / 4;                 // 4-element quads per chunk
  constexpr int SX = (int)sizeof(typename Op::TX);
  constexpr int V = R * NB;                       // sums per row group
  constexpr int LOGV = V == 32 ? 5 : V == 16 ? 4 : V == 8 ? 3 : V == 4 ? 2 : 1;
  static_assert((1 << LOGV) == V, "R * NB must be a power of two up to 32");
  static_assert(XE == 4 || (XE == 2 && SX == 2), "x staged as fp32 or as stored 16-bit");
  static_assert(!SW || R == 2, "SwiGLU pairs the gate and up row of one output");
  // bytes of one staged word per chunk and plane: 16 for PAIRS and fp32 quads, 8 for
  // 16-bit quads
  constexpr int WB = PAIRS ? 16 : 4 * XE;
  // planes: PAIRS fp32: [p][k pair h < VEC/2]; PAIRS 16-bit: [p][quad w];
  // otherwise [b][quad w]
  constexpr int PPV = PAIRS ? (XE == 4 ? Op::VEC / 2 : QW) : QW;  // planes per vector (pair)
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t M = a.M, K = a.K;
  const int B = a.B;
  // K slice blockIdx.y: chunks c0 .. c0 + nch - 1 of every row (all of K when the
  // grid has one slice); its sums go to partial[slice][b][m] for k_splitk_reduce
  const int64_t c0 = (int64_t)blockIdx.y * chunks_per_split;
  const int64_t nch_all = K / Op::VEC;
  const int64_t nch = nch_all - c0 < chunks_per_split ? nch_all - c0 : chunks_per_split;
  if (nch <= 0) return;  // K = 0 never reaches this kernel; the plan has no empty slice
  // the slice's x is staged in shared memory, so its chunk and step counts fit 32 bits
  const int nch32 = (int)nch, nsteps = (nch32 + 31) / 32;
  const int64_t rowb = row_bytes<Op>(K);
  const char *A = reinterpret_cast<const char *>(a.A) + c0 * 16;
  const int64_t k0 = c0 * Op::VEC;  // first element of the slice
  const int64_t groups = SW ? a.half : (M + R - 1) / R;
  auto row_of = [&](int64_t gg, int r) -> int64_t { return SW ? gg + r * a.half : gg * R + r; };
  const int64_t gstride = (int64_t)gridDim.x * WARPS;

  // shared memory: x planes, then the ring [warp][stage][row][lane] of 16-byte slots
  const int64_t pstride = nch * WB;  // bytes per plane
  const uint32_t ps32 = (uint32_t)pstride;  // shared-memory offsets fit 32 bits
  const int64_t xbytes = (int64_t)(PAIRS ? NP : NB) * PPV * pstride;
  const uint32_t xs_s = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t ring_s = xs_s + (uint32_t)xbytes + (uint32_t)((warp * G * R * 32 + lane) * 16);
  // Shared-memory reads of the ring slots and of x.  int4 (except 8 vectors) uses
  // plain loads, which the compiler schedules freely (the copies' waits and issues,
  // inline assembly with a memory clobber, still order them); the inline-assembly
  // loads made it spill: int4 8192x8192 B = 16 93.4 -> 76.8 us, B = 4 32.7 -> 30.9
  // (event means).  8 int4 vectors (45.6 -> 47.0) and the other types (int8
  // 8192x8192 B = 8 39.9 -> 41.0) keep the assembly loads.
  constexpr bool PLAIN_LDS = Op::GROUPED && NB != 8;
  auto ld16 = [&](uint32_t s) -> uint4 {
    if constexpr (PLAIN_LDS) return *reinterpret_cast<const uint4 *>(smem + (s - xs_s));
    else return lds16(s);
  };
  auto ld8 = [&](uint32_t s) -> uint2 {
    if constexpr (PLAIN_LDS) return *reinterpret_cast<const uint2 *>(smem + (s - xs_s));
    else return lds8(s);
  };
  // int4: each slot's group scale, in a second ring [warp][stage][row][lane] of floats
  constexpr bool GRP = Op::GROUPED;
  const uint32_t sc_s = xs_s + (uint32_t)xbytes + (uint32_t)(WARPS * G * R * 32 * 16) +
                        (uint32_t)((warp * G * R * 32 + lane) * 4);
  const int64_t gpr = K >> a.gshift;  // groups per row (int4)

  // producer position: row group pg, step pj (chunks 32 pj + lane).  Which rows of
  // group pg exist is set once per row group; with few vectors (registers to spare)
  // so are the rows' addresses of this lane's step-0 chunk (and int4 group-scale
  // rows), and a step costs one add per row.
  constexpr bool CACHE = NB <= 4;
  int64_t pg = blockIdx.x + (int64_t)gridDim.x * warp;
  int pj = 0;
  const char *pa[CACHE ? R : 1];
  const float *pscale[CACHE && GRP ? R : 1];
  uint32_t plive = 0;  // bit r: row r of group pg exists (none once pg >= groups)
  auto set_rows = [&]() {
    plive = 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int64_t row = row_of(pg, r);
      const bool ok = pg < groups && row < M;
      plive |= (ok ? 1u : 0u) << r;
      if constexpr (CACHE) {
        pa[r] = A + (ok ? row * rowb : 0) + lane * 16;
        if constexpr (GRP) pscale[r] = a.gscale + (ok ? row * gpr : 0);
      }
    }
  };
  set_rows();
  auto issue = [&](int stage) {
    const int c = 32 * pj + lane;
    if (plive != 0 && c < nch32) {
      const uint32_t dst = ring_s + (uint32_t)(stage * R * 32 * 16);
      const int64_t aoff = (int64_t)(pj * (32 * 16));
      [[maybe_unused]] int64_t goff = 0;
      if constexpr (GRP) goff = ((c0 + c) * Op::VEC) >> a.gshift;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (plive & (1u << r)) {
          const char *src;
          [[maybe_unused]] const float *gsrc = nullptr;
          if constexpr (CACHE) {
            src = pa[r] + aoff;
            if constexpr (GRP) gsrc = pscale[r] + goff;
          } else {
            const int64_t row = row_of(pg, r);
            src = A + row * rowb + c * 16;
            if constexpr (GRP) gsrc = a.gscale + row * gpr + goff;
          }
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + (uint32_t)(r * 32 * 16)), "l"(src)
                       : "memory");
          if constexpr (GRP)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sc_s + (uint32_t)((stage * R + r) * 32 * 4)),
                         "l"(gsrc) : "memory");
        }
      }
    }
    if (pg < groups && ++pj == nsteps) {
      pj = 0;
      pg += gstride;
      set_rows();
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // x staging.  Copied as stored (planes of one vector's quads): cp.async straight
  // into place, one commit group issued before A's first steps.  Interleaved or
  // widened: eight items (quads of one vector or of a vector pair) per thread in
  // flight through registers at a time.
  const unsigned char *xsrc = reinterpret_cast<const unsigned char *>(a.x) + k0 * SX;
  const int64_t nq = nch * Op::VEC / 4;  // quads per vector in the slice
  constexpr bool XCOPY = !PAIRS && XE == SX;
  // (with weight prefetch before the launch dependency is resolved, A's first steps go
  // out first and x's copy after the wait, as the newest group)
  const bool x_first = a.pdl != 2;
  // Both staging loops visit items tid, tid + THREADS, ... of the order [vector (or
  // vector pair)][quad].  A thread carries its item's (vector, quad) position in 32
  // bits (the slice's x fits in shared memory) and steps it without dividing: a
  // 64-bit division per item cost about 3 instructions per weight of A at 4 vectors.
  const uint32_t nq32 = (uint32_t)nq, nch32u = (uint32_t)nch;
  const uint32_t step_v = (uint32_t)THREADS / nq32, step_q = (uint32_t)THREADS % nq32;
  auto advance = [&](uint32_t &v, uint32_t &q) {
    v += step_v;
    q += step_q;
    if (q >= nq32) {
      q -= nq32;
      ++v;
    }
  };
  auto copy_x = [&]() {
    uint32_t b = (uint32_t)tid / nq32, q = (uint32_t)tid % nq32;
    for (; b < (uint32_t)B; advance(b, q)) {
      const uint32_t c = q / QW, w = q % QW;  // chunk 4q / VEC, quad (4q mod VEC) / 4
      const uint32_t dst = xs_s + ((b * PPV + w) * nch32u + c) * WB;
      const unsigned char *sp = xsrc + ((int64_t)b * K + 4 * (int64_t)q) * SX;
      if constexpr (WB == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(sp) : "memory");
      else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(sp) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    for (int64_t i = (int64_t)B * PPV * pstride / 16 + tid; i < xbytes / 16; i += THREADS)
      reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);  // vectors B..NB-1
  };
  if (XCOPY && x_first) copy_x();
#pragma unroll
  for (int s = 0; s < G; ++s) issue(s);
  pdl_after_prefetch(a);

  if constexpr (XCOPY) {
    if (x_first) {
      asm volatile("cp.async.wait_group %0;" ::"n"(G) : "memory");  // x's group (the oldest)
    } else {
      copy_x();
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
  } else {
    // quad q of vector b (zero past B), as 4 fp32 values or 2 words of 16-bit values
    auto load_quad = [&](int64_t b, int64_t q) -> uint4 {
      uint4 v = make_uint4(0, 0, 0, 0);
      if (b < B) {
        const unsigned char *sp = xsrc + (b * K + 4 * q) * SX;
        if (SX == 4) {
          v = *reinterpret_cast<const uint4 *>(sp);
        } else {
          const uint2 h = *reinterpret_cast<const uint2 *>(sp);
          v.x = h.x;
          v.y = h.y;
        }
      }
      return v;
    };
    auto to_f32 = [&](const uint4 &v, float (&f)[4]) {
      if constexpr (SX == 4) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
      } else {
        widen4(v.x, v.y, f, typename Op::TX());
      }
    };
    constexpr uint32_t NV = PAIRS ? NP : NB;  // items per quad index: vector pairs or vectors
    uint32_t iv = (uint32_t)tid / nq32, q = (uint32_t)tid % nq32;
    while (iv < NV) {
      // the loads of 8 items, then (walking the same 8 positions again) their stores
      const uint32_t iv0 = iv, q0 = q;
      uint4 v0[8], v1[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        v0[u] = make_uint4(0, 0, 0, 0);
        v1[u] = make_uint4(0, 0, 0, 0);
        if (iv < NV) {
          v0[u] = load_quad(PAIRS ? 2 * iv : iv, q);
          if (PAIRS) v1[u] = load_quad(2 * iv + 1, q);
        }
        advance(iv, q);
      }
      iv = iv0;
      q = q0;
#pragma unroll
      for (int u = 0; u < 8; ++u, advance(iv, q)) {
        if (iv >= NV) continue;
        const uint32_t c = q / QW, w = q % QW;
        if constexpr (PAIRS && XE == 4) {
          float f0[4], f1[4];
          to_f32(v0[u], f0);
          to_f32(v1[u], f1);
          unsigned char *d0 = smem + ((iv * PPV + 2 * w) * nch32u + c) * WB;
          *reinterpret_cast<float4 *>(d0) = make_float4(f0[0], f1[0], f0[1], f1[1]);
          *reinterpret_cast<float4 *>(d0 + pstride) = make_float4(f0[2], f1[2], f0[3], f1[3]);
        } else if constexpr (PAIRS) {
          unsigned char *d = smem + ((iv * PPV + w) * nch32u + c) * WB;
          *reinterpret_cast<uint4 *>(d) =
              make_uint4(__byte_perm(v0[u].x, v1[u].x, 0x5410), __byte_perm(v0[u].x, v1[u].x, 0x7632),
                         __byte_perm(v0[u].y, v1[u].y, 0x5410), __byte_perm(v0[u].y, v1[u].y, 0x7632));
        } else {  // widened to fp32, one vector's quads
          float f0[4];
          to_f32(v0[u], f0);
          unsigned char *d = smem + ((iv * PPV + w) * nch32u + c) * WB;
          *reinterpret_cast<float4 *>(d) = make_float4(f0[0], f0[1], f0[2], f0[3]);
        }
      }
    }
  }
  __syncthreads();

  const int idx = lane >> (5 - LOGV);  // the sum this lane ends with
  const bool owner = (lane & ((32 >> LOGV) - 1)) == 0;
  int stage = 0;
  for (int64_t g = blockIdx.x + (int64_t)gridDim.x * warp; g < groups; g += gstride) {
    // this lane's epilogue operands (row idx / NB, vector idx % NB), in flight
    // while the group streams
    const int er = idx / NB, eb = idx % NB;
    const int64_t erow = row_of(g, er);
    const bool live = owner && eb < B && erow < M && !SW;
    RowPre pre = row_pre<Op, false>(a, erow, live && partial == nullptr);
    if (live && partial == nullptr && a.residual != nullptr)
      pre.res = residual_at<Op>(a.residual, (int64_t)eb * M + erow);

    constexpr int NA = PAIRS ? NP : NB;  // accumulator pairs per row
    float2 acc[R][NA];
    float accm[R][NB];  // kRingMixed
#pragma unroll
    for (int r = 0; r < R; ++r) {
#pragma unroll
      for (int i = 0; i < NA; ++i) acc[r][i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int b = 0; b < NB; ++b) accm[r][b] = 0.f;
    }
    for (int j = 0; j < nsteps; ++j) {
      asm volatile("cp.async.wait_group %0;" ::"n"(G - 1) : "memory");  // this step has landed
      uint4 av[R];
#pragma unroll
      for (int r = 0; r < R; ++r) av[r] = ld16(ring_s + (uint32_t)((stage * R + r) * 32 * 16));
      float gsc[GRP ? R : 1];
      if constexpr (GRP) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint32_t sa = sc_s + (uint32_t)((stage * R + r) * 32 * 4);
          if constexpr (PLAIN_LDS) gsc[r] = *reinterpret_cast<const float *>(smem + (sa - xs_s));
          else asm volatile("ld.shared.f32 %0, [%1];" : "=f"(gsc[r]) : "r"(sa));
        }
      }
      issue(stage);  // this lane's slots of the stage are free again
      stage = stage + 1 == G ? 0 : stage + 1;
      const int c = 32 * j + lane;
      if (c >= nch32) continue;
      const uint32_t xc = xs_s + (uint32_t)c * (uint32_t)WB;
      // int4 with few sums per row group: the chunk's unscaled sums, scaled once
      // after the chunk (one packed FMA per sum pair instead of scaling every weight)
      constexpr bool CSC = GRP && !PAIRS;
      float2 cacc[CSC ? R : 1][CSC ? NA : 1];
      if constexpr (CSC) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int i = 0; i < NA; ++i) cacc[r][i] = make_float2(0.f, 0.f);
      }
      auto sum = [&](int r, int i) -> float2 & {
        if constexpr (CSC) return cacc[r][i]; else return acc[r][i];
      };
#pragma unroll
      for (int w = 0; w < QW; ++w) {
        if constexpr (MODE == kRingMixed) {
          // the 16-bit halves of A (once per row) and of x (once per vector), then
          // one mixed-precision FMA per product
          unsigned short ah[R][4];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            split_halves(w ? av[r].z : av[r].x, ah[r][0], ah[r][1]);
            split_halves(w ? av[r].w : av[r].y, ah[r][2], ah[r][3]);
          }
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const uint2 h = ld8(xc + (uint32_t)(b * PPV + w) * ps32);
            unsigned short xh[4];
            split_halves(h.x, xh[0], xh[1]);
            split_halves(h.y, xh[2], xh[3]);
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
              for (int e = 0; e < 4; ++e) Op::fma_mixed(accm[r][b], ah[r][e], xh[e]);
          }
          continue;
        }
        float2 q01[R], q23[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          Op::quad2(av[r], w, q01[r], q23[r]);
          if constexpr (GRP && !CSC) {  // int4: the chunk's group scale, applied to the weights
            q01[r] = __fmul2_rn(q01[r], make_float2(gsc[r], gsc[r]));
            q23[r] = __fmul2_rn(q23[r], make_float2(gsc[r], gsc[r]));
          }
        }
        if constexpr (PAIRS) {
#pragma unroll
          for (int p = 0; p < NP; ++p) {
            float2 X[4];
            if constexpr (XE == 4) {
              const uint4 u0 = ld16(xc + (uint32_t)(p * PPV + 2 * w) * ps32);
              const uint4 u1 = ld16(xc + (uint32_t)(p * PPV + 2 * w + 1) * ps32);
              X[0] = make_float2(__uint_as_float(u0.x), __uint_as_float(u0.y));
              X[1] = make_float2(__uint_as_float(u0.z), __uint_as_float(u0.w));
              X[2] = make_float2(__uint_as_float(u1.x), __uint_as_float(u1.y));
              X[3] = make_float2(__uint_as_float(u1.z), __uint_as_float(u1.w));
            } else {
              const uint4 u = ld16(xc + (uint32_t)(p * PPV + w) * ps32);
              X[0] = widen2(u.x, typename Op::TX());
              X[1] = widen2(u.y, typename Op::TX());
              X[2] = widen2(u.z, typename Op::TX());
              X[3] = widen2(u.w, typename Op::TX());
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
              float2 &t = sum(r, p);
              t = __ffma2_rn(make_float2(q01[r].x, q01[r].x), X[0], t);
              t = __ffma2_rn(make_float2(q01[r].y, q01[r].y), X[1], t);
              t = __ffma2_rn(make_float2(q23[r].x, q23[r].x), X[2], t);
              t = __ffma2_rn(make_float2(q23[r].y, q23[r].y), X[3], t);
            }
          }
        } else {
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const uint32_t xa = xc + (uint32_t)(b * PPV + w) * ps32;
            float2 x01, x23;
            if constexpr (XE == 4) {
              const uint4 u = ld16(xa);
              x01 = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
              x23 = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
            } else {
              const uint2 h = ld8(xa);
              float f[4];
              widen4(h.x, h.y, f, typename Op::TX());
              x01 = make_float2(f[0], f[1]);
              x23 = make_float2(f[2], f[3]);
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
              float2 &t = sum(r, b);
              t = __ffma2_rn(q01[r], x01, t);
              t = __ffma2_rn(q23[r], x23, t);
            }
          }
        }
      }
      if constexpr (CSC) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int i = 0; i < NA; ++i) acc[r][i] = __ffma2_rn(cacc[r][i], make_float2(gsc[r], gsc[r]), acc[r][i]);
      }
    }
    float v[V];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b)
        v[r * NB + b] = MODE == kRingMixed ? accm[r][b]
                        : PAIRS ? ((b & 1) ? acc[r][b / 2].y : acc[r][b / 2].x)
                                : acc[r][b].x + acc[r][b].y;
    const float part = warp_reduce_scatter<V>(v, lane);
    if constexpr (SW) {
      // gate sum b sits at lane b * 32 / V, its up sum 16 lanes above
      const float up = __shfl_down_sync(0xffffffffu, part, 16);
      if (owner && idx < NB && idx < B) epilogue_swiglu<Op>(a, idx, g, part, up);
    } else if (partial != nullptr) {
      if (live) partial[((int64_t)blockIdx.y * B + eb) * M + erow] = part;
    } else {
      if (live) store_act_res<Op>(a, (int64_t)eb * M + erow, row_value_pre<Op>(a, pre, part), pre.res);
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// 16-byte global -> shared copy to a shared-memory address given as a 32-bit offset.
__device__ __forceinline__ void cp_async16_s(uint32_t s, const void *gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}

// The ring holds G groups of P rows: group gi sits in slots (gi % G) * P + q, so a
// group's slots are free again once the group G before it has been read.  All
// indexes inside the CTA's block of rows are 32-bit and the slot addresses are
// 32-bit shared-memory offsets: the only 64-bit arithmetic per group is one pointer
// to its first row.
template <class Op, int NB, int J, int P, int G>
__global__ void __launch_bounds__(kXsThreads, 1) k_xsplit(const Args a) {
  pdl_enter(a, true);
  static_assert(NB == 1 || NB == 2 || NB == 4, "NB");
  static_assert(kXsT % P == 0 && (kXsT & (kXsT - 1)) == 0, "a barrier batch is whole groups");
  static_assert((G & (G - 1)) == 0, "G is a power of two");
  extern __shared__ __align__(16) unsigned char ring[];  // [G][P][J][512] 16-byte slots
  __shared__ float red[2][kXsT][kXsWarps][NB];
  constexpr int PV = Op::VEC / 2;               // fp32 pairs per chunk
  constexpr uint32_t kSlot = kXsThreads * 16;  // bytes between one thread's consecutive slots
  constexpr int LOGT = kXsT == 16 ? 4 : kXsT == 8 ? 3 : kXsT == 4 ? 2 : kXsT == 2 ? 1 : 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t M = a.M, K = a.K, nch = K / Op::VEC;
  const int B = a.B;
  const int64_t rowb = row_bytes<Op>(K);
  const int64_t r0 = M * blockIdx.x / gridDim.x, r1 = M * (blockIdx.x + 1) / gridDim.x;
  const int n = (int)(r1 - r0);  // rows of this CTA
  const int ngroups = (n + P - 1) / P;
  bool cj[J];  // does this thread own chunk tid + 512 j of a row?
#pragma unroll
  for (int j = 0; j < J; ++j) cj[j] = tid + (int64_t)kXsThreads * j < nch;
  // this thread's chunk 0 of the CTA's first row; chunk tid + 512 j is j * kSlot further
  const char *At = reinterpret_cast<const char *>(a.A) + r0 * rowb + (int64_t)tid * 16;
  const uint32_t ring_t = (uint32_t)__cvta_generic_to_shared(ring) + (uint32_t)tid * 16;

  // this thread's chunks of group gi's rows into their slots; one commit group per
  // call (empty past the last row, so every iteration waits on the same count)
  auto issue = [&](int gi) {
    const char *pg = At + (int64_t)gi * P * rowb;
    const uint32_t sg = ring_t + (uint32_t)((gi & (G - 1)) * P * J) * kSlot;
#pragma unroll
    for (int q = 0; q < P; ++q) {
      if (gi * P + q < n) {
#pragma unroll
        for (int j = 0; j < J; ++j)
          if (cj[j]) cp_async16_s(sg + (uint32_t)(q * J + j) * kSlot, pg + q * rowb + (int64_t)j * kSlot);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
#pragma unroll
  for (int gi = 0; gi < G; ++gi) issue(gi);
  pdl_after_prefetch(a);

  float2 xr[J][NB][PV];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int64_t c = tid + (int64_t)kXsThreads * j;
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int p = 0; p < PV; ++p) {
        const int64_t k = c * Op::VEC + 2 * p;
        xr[j][b][p] = (c < nch && b < B) ? make_float2(Op::x_elem(a.x, (int64_t)b * K + k),
                                                       Op::x_elem(a.x, (int64_t)b * K + k + 1))
                                         : make_float2(0.f, 0.f);
      }
  }

  // epilogue operands of this thread's output in the current batch (threads
  // tid < kXsT * NB: row tid / NB of the batch, vector tid % NB), loaded when the
  // batch starts so that they have arrived when its sums are ready
  RowPre pre{1.f, 0.f, 0.f};
  constexpr int V = P * NB;  // values one group reduces (row q, vector b at q * NB + b)
  constexpr int LOGV = V == 16 ? 4 : V == 8 ? 3 : V == 4 ? 2 : V == 2 ? 1 : 0;
  static_assert((1 << LOGV) == V && V <= 32, "P * NB must be a power of two up to 32");
  for (int gi = 0; gi < ngroups; ++gi) {
    const int i0 = gi * P;
    const int t0 = i0 & (kXsT - 1);  // the group's first row within its barrier batch
    if (t0 == 0 && tid < kXsT * NB) {
      const int64_t row = r0 + i0 + tid / NB;
      const int b = tid % NB;
      const bool live = row < r1 && b < B;
      pre = row_pre<Op, false>(a, row, live);
      if (live && a.residual != nullptr) pre.res = residual_at<Op>(a.residual, (int64_t)b * M + row);
    }
    asm volatile("cp.async.wait_group %0;" ::"n"(G - 1) : "memory");  // group gi has landed
    // the group's P rows (rows past n contribute zeros), then one reduction for all
    const uint32_t sg = ring_t + (uint32_t)((gi & (G - 1)) * P * J) * kSlot;
    float v[V];
#pragma unroll
    for (int q = 0; q < P; ++q) {
      float2 acc[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[b] = make_float2(0.f, 0.f);
      if (i0 + q < n) {
#pragma unroll
        for (int j = 0; j < J; ++j) {
          if (cj[j]) {
            const uint4 av = lds16(sg + (uint32_t)(q * J + j) * kSlot);
#pragma unroll
            for (int w = 0; w < Op::VEC / 4; ++w) {
              float2 q01, q23;
              Op::quad2(av, w, q01, q23);
#pragma unroll
              for (int b = 0; b < NB; ++b) {
                acc[b] = __ffma2_rn(q01, xr[j][b][2 * w], acc[b]);
                acc[b] = __ffma2_rn(q23, xr[j][b][2 * w + 1], acc[b]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) v[q * NB + b] = acc[b].x + acc[b].y;
    }
    issue(gi + G);  // the group's slots are free again (this thread read them above)
    const float part = warp_reduce_scatter<V>(v, lane);
    const int hb = (i0 >> LOGT) & 1;
    if ((lane & ((32 >> LOGV) - 1)) == 0) {
      const int idx = lane >> (5 - LOGV);
      red[hb][t0 + idx / NB][warp][idx % NB] = part;
    }
    const int ilast = min(i0 + P, n) - 1;  // the group's last real row
    const int t = ilast & (kXsT - 1);
    if (t == kXsT - 1 || ilast == n - 1) {
      __syncthreads();
      if (tid < (t + 1) * NB) {
        const int rr = tid / NB, b = tid % NB;
        if (b < B) {
          float sum = 0.f;
#pragma unroll
          for (int w = 0; w < kXsWarps; ++w) sum += red[hb][rr][w][b];
          store_act_res<Op>(a, (int64_t)b * M + r0 + (ilast - t) + rr, row_value_pre<Op>(a, pre, sum), pre.res);
        }
      }
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

}  // namespace gemv
