// Host-side shape dispatcher for libgemv (no CUDA calls; unit-tested on the CPU).
//
// The one design axis of a GEMV is how many threads share an output row ("16-sgemv"
// notes, design-space summary: elements per thread x rows per warp = 32; a short
// row wastes lanes, few rows leave SMs idle).  Lesson 3 "GEMV and row-level
// parallelism", section 4, gives the same rule by row length: a warp per row for
// short rows, a CTA per row for long ones; the NPU MatMul post, sections 1.3 and
// 3.4, asks for the kernel to be picked from (M, N, K, dtype, hardware) at run time.
//
// Rules used here, in the order they are tried (per call, from dtype, M, K, B,
// alignment and the SM count; the thresholds come from timing every kernel on
// GB300).  "Chunk" is 16 bytes of a row; rows/SM is M over the SM count.
//   fp16/bf16 with 17..256 vectors        -> TC (tcgen05 small-N GEMM)
//   rows not 16-byte aligned              -> SCALAR (element loads)
//   rows of <= 16 chunks                  -> ROWS_PER_WARP, lanes = next pow2 of chunks
//   XSPLIT (K split over a CTA, x in registers; x slice within the register budget):
//     fp32, B == 1, 8 rows/SM <= M <= 12288
//     fp32, B == 2, >= 8 rows/SM, M < 65536
//     K >= 8192, M >= one row/SM: fp16/bf16 with B == 2 and M <= 4096, or fp32
//     with B == 4 and M <= 8192
//     fp16/bf16, B == 1, K >= 8192, 1..11 rows/SM (1..15 for K >= 12288)
//   fp32, B == 2, rows of >= 2048 chunks, 2..31 rows/SM -> BLOCK_PER_ROW
//   BATCHED, when x[0..B) can be staged and rows have >= 32 chunks, for B >= 2,
//     and for B == 1 of int8 (>= 48 rows/SM) or int4 (>= 16 rows/SM) below 65536
//     rows with x staged whole: the row-pair kernel for at most one row pair per
//     warp with 4..16 vectors (int8 2..16, fp32 5..16), for at most one ring row
//     group per warp with 4 int8 or 5..8 fp16/bf16 vectors, for 16 vectors of
//     16-bit/fp32 rows, 8 vectors of 16-bit rows whose ring would stage x as stored,
//     and x too large for the ring; otherwise the cp.async ring (mixed-precision FMAs
//     for fp16/bf16 with 2 or 16 vectors, 5..8 over K slices, and 4 vectors on up to
//     2048 rows), over K slices with a second pass when x does not fit whole
//   M >= 65536                            -> WARP_PER_ROW (non-persistent grid)
//   B == 1, >= 16 rows/SM (fp32) or >= 12 (other types) -> STREAM (persistent
//     warps), except fp32 rows of >= 1024 chunks whose row walk would leave the
//     streaming warps below 75% busy -> WARP_PER_ROW
//   >= 16 rows/SM, or rows of <= 512 chunks -> WARP_PER_ROW
//   >= 2 rows/SM, or rows of < 1024 chunks  -> BLOCK_PER_ROW
//   fewer rows                            -> SPLIT_K over enough K slices to give
//                                            every SM about four CTAs
#include <stdint.h>

#include "../../include/gemv.h"
#include "gemv_plan.h"

namespace gemv {

namespace {

int next_pow2(int64_t v) {
  int p = 1;
  while (p < v && p < (1 << 30)) p <<= 1;
  return p;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

int elem_bytes_a(int dtype) {
  switch (dtype) {
    case GEMV_DTYPE_F32: return 4;
    case GEMV_DTYPE_F16:
    case GEMV_DTYPE_BF16: return 2;
    default: return 1;  // int8; int4 packs two elements per byte
  }
}

int elem_bytes_x(int dtype) { return dtype == GEMV_DTYPE_F32 ? 4 : 2; }

int chunk_elems(int dtype) {
  switch (dtype) {
    case GEMV_DTYPE_F32: return 4;
    case GEMV_DTYPE_F16:
    case GEMV_DTYPE_BF16: return 8;
    case GEMV_DTYPE_W8: return 16;
    default: return 32;  // int4: two per byte
  }
}

static bool rowteam_lanes_ok(int l) { return l == 1 || l == 2 || l == 4 || l == 8 || l == 16; }

// The row-pair kernel stages x[0..NB) as stored.
static bool rowpair_fits(int nb, int64_t K, int sx) { return (int64_t)nb * K * sx <= kBatchedSmemMax; }

// x staging of the BATCHED ring kernel: fp32 where x and the ring fit, else as
// stored; -1 if x does not fit.
static int ring_staging(int nb, int64_t K, int sx, int64_t extra) {
  const int64_t room = kRingSmemMax - ring_bytes(nb) - extra;
  if (sx != 4 && (int64_t)nb * K * 4 <= room) return GEMV_X_SMEM_FP32;
  if ((int64_t)nb * K * sx <= room) return GEMV_X_SMEM;
  return -1;
}

// K slices of the ring kernel: 1 when x[0..NB) fits with the ring, else the fewest
// slices (at most 64) whose share of x fits as stored; 0 if none does.
static int ring_slices(int nb, int64_t nch, int vec, int sx, int64_t extra) {
  for (int s = 1; s <= 64; ++s) {
    const int64_t cps = (nch + s - 1) / s;
    if (ring_staging(nb, cps * vec, sx, extra) >= 0) return s;
  }
  return 0;
}

gemv_status_t plan(int dtype, int64_t M, int64_t K, int B, bool aligned16, int num_sms,
                   int force_kernel, int force_param, gemv_plan_t *out) {
  if (out == nullptr || num_sms < 1) return GEMV_ERR_INVALID_VALUE;
  if (dtype < GEMV_DTYPE_F32 || dtype > GEMV_DTYPE_W4) return GEMV_ERR_INVALID_VALUE;
  if (M < 0 || K < 0 || B < 0) return GEMV_ERR_INVALID_VALUE;
  const bool half16 = dtype == GEMV_DTYPE_F16 || dtype == GEMV_DTYPE_BF16;
  if (B > GEMV_MAX_BATCH && !(half16 && B <= GEMV_MAX_BATCH_TC)) return GEMV_ERR_UNSUPPORTED;
  gemv_plan_t p = {};
  p.kernel = GEMV_KERNEL_AUTO;
  p.splits = 1;
  p.threads = kPlanThreads;
  if (M == 0 || B == 0) {
    *out = p;
    return GEMV_SUCCESS;
  }
  const int sx = elem_bytes_x(dtype);
  const int vec = chunk_elems(dtype);
  const bool vec_ok = aligned16 && (K % vec == 0);
  const int64_t nch = vec_ok ? K / vec : 0;
  p.nb = B > GEMV_MAX_BATCH ? (B + 15) / 16 * 16 : next_pow2(B);
  // more than 16 vectors: only the tensor-core kernel, which needs 16-byte rows
  if (B > GEMV_MAX_BATCH && !vec_ok) return GEMV_ERR_UNSUPPORTED;
  const bool tc_ok = half16 && vec_ok;
  // the ring kernel over rslices K slices (x staged per slice), the row-pair kernel
  // over all of K (int4: the ring also carries each slot's group scale; the row-pair
  // kernel is not built for grouped scales)
  const int64_t rextra = dtype == GEMV_DTYPE_W4 ? ring_scale_bytes(p.nb) : 0;
  const int rslices = nch == 0 ? 0 : ring_slices(p.nb, nch, vec, sx, rextra);
  const int64_t rcps = rslices > 0 ? ceil_div(nch, rslices) : 0;  // chunks per slice
  const int rstage = rslices > 0 ? ring_staging(p.nb, rcps * vec, sx, rextra) : -1;
  const bool rowpair_ok = dtype != GEMV_DTYPE_W4 && rowpair_fits(p.nb, K, sx);
  const bool mixed_ok = half16 && rstage >= 0;  // x as stored fits wherever fp32 x does
  const bool batched_ok = rstage >= 0 || rowpair_ok;
  // XSPLIT: chunks per thread J (a power of two up to 4) and x registers
  const int xs_j = vec_ok && nch > 0 ? next_pow2(ceil_div(nch, kXsplitThreads)) : 0;
  const bool xs_ok = vec_ok && dtype != GEMV_DTYPE_W4 && p.nb <= 4 && xs_j >= 1 && xs_j <= 4 &&
                     xs_j * p.nb * vec <= kXsplitMaxXRegs;

  int kernel = GEMV_KERNEL_AUTO;
  int param = 0;
  if (force_kernel != GEMV_KERNEL_AUTO) {
    bool ok = false;
    switch (force_kernel) {
      case GEMV_KERNEL_ROWS_PER_WARP:
        ok = vec_ok && (force_param == 0 || rowteam_lanes_ok(force_param));
        break;
      case GEMV_KERNEL_WARP_PER_ROW:
      case GEMV_KERNEL_BLOCK_PER_ROW:
        ok = vec_ok;
        break;
      case GEMV_KERNEL_SPLIT_K:
        ok = vec_ok && nch >= 2 && force_param >= 0;
        break;
      case GEMV_KERNEL_BATCHED:
        ok = vec_ok && (B >= 2 || force_param == 1 + GEMV_BATCHED_RING) &&
             ((force_param == 0 && batched_ok) || (force_param == 1 + GEMV_BATCHED_RING && rstage >= 0) ||
              (force_param == 1 + GEMV_BATCHED_ROWPAIR && rowpair_ok) ||
              (force_param == 1 + GEMV_BATCHED_RING_MIXED && mixed_ok));
        break;
      case GEMV_KERNEL_STREAM:
        ok = vec_ok && B == 1;
        break;
      case GEMV_KERNEL_XSPLIT:
        ok = xs_ok && B <= GEMV_MAX_BATCH;
        break;
      case GEMV_KERNEL_TC:
        ok = tc_ok;
        break;
      case GEMV_KERNEL_SCALAR:
        ok = force_param == 0 || force_param == 4 || force_param == 32;
        break;
      default:
        ok = false;
    }
    if (ok) {
      kernel = force_kernel;
      param = force_param;
    }
  }

  if (B > GEMV_MAX_BATCH) kernel = GEMV_KERNEL_TC;  // the only kernel for 17..256 vectors
  if (kernel == GEMV_KERNEL_AUTO) {
    if (!vec_ok) {
      kernel = GEMV_KERNEL_SCALAR;
    } else if (nch <= 16) {
      kernel = GEMV_KERNEL_ROWS_PER_WARP;
    } else if (xs_ok && dtype == GEMV_DTYPE_F32 && B == 1 && M >= (int64_t)num_sms * 8 && M <= 12288) {
      // fp32, one vector, up to 12288 rows of at most 8192 elements: the K-split kernel
      // (4096x4096 16.4 us against 20.6 streaming, 4096x8192 24.9 against 29.4 warp
      // per row, 8192x8192 43.4 against 47.6, 12288x8192 62.5 against 69.2,
      // 2048x8192 16.4 against 22.6)
      kernel = GEMV_KERNEL_XSPLIT;
    } else if (xs_ok && dtype == GEMV_DTYPE_F32 && B == 2 && M >= (int64_t)num_sms * 8 && M < 65536) {
      // fp32 with 2 vectors: K split over a CTA, x in registers (measured: fp32
      // 8192x4096 26.6 us against 28.7 in the ring kernel, 2048x8192 16.7 against
      // 28.8; for 16-bit types and more vectors the ring kernel is faster, with one
      // vector the streaming one)
      kernel = GEMV_KERNEL_XSPLIT;
    } else if (xs_ok && K >= 8192 && M >= num_sms &&
               ((half16 && B == 2 && M <= 4096) || (dtype == GEMV_DTYPE_F32 && B == 4 && M <= 8192))) {
      // long rows, few of them: the K-split kernel for 2 fp16/bf16 vectors (bf16
      // 1024x16384 14.4 us against 20.5 in the mixed ring, 4096x14336 25.2 against
      // 26.6) and 4 fp32 vectors (8192x8192 46.4 against 52.1 in the ring, 2048x8192
      // 18.5 against 28.5 in the row pairs)
      kernel = GEMV_KERNEL_XSPLIT;
    } else if (xs_ok && half16 && B == 1 && K >= 8192 && M >= num_sms &&
               M < (int64_t)num_sms * (K >= 12288 ? 16 : 12)) {
      // one vector of few long 16-bit rows: the K-split kernel spreads each row over a
      // CTA (bf16 1024x16384 12.3 us against 15.1 block per row, 1536x16384 14.4 against
      // 18.4, 1024x8192 10.2 against 11.6, 256x16384 9.2 against 13.7 split-K, 2048x14336
      // 16.4 against 17.7 streaming; f16 1024x16384 12.3 against 16.2; the streaming
      // kernel from 12 rows per SM of 8192 elements, bf16 2048x8192 12.4 against 14.2 block
      // per row, and from 16 of longer ones: 4096x14336 24.6 each)
      kernel = GEMV_KERNEL_XSPLIT;
    } else if (dtype == GEMV_DTYPE_F32 && p.nb == 2 && nch >= 2048 && M >= (int64_t)num_sms * 2 &&
               M < (int64_t)num_sms * 32) {
      // two vectors of few long fp32 rows: block per row, where the batched kernels'
      // row groups of 4 would leave most warps idle (1024x16384 24.9 us against 50.0,
      // 2048x12288 27.6 against 41.0, 4096x14336 47.3 against 52.8, 1024x8192 16.4
      // against 28.8; at 8192x14336 the ring leads, 79.6 against 81.3)
      kernel = GEMV_KERNEL_BLOCK_PER_ROW;
    } else if ((B > 1 || ((dtype == GEMV_DTYPE_W8 || dtype == GEMV_DTYPE_W4) && rslices == 1 &&
                          M >= (int64_t)num_sms * (dtype == GEMV_DTYPE_W8 ? 48 : 16) && M < 65536)) &&
               batched_ok && nch >= 32) {
      // (one vector of int8 or int4 weights too: the decode-bound rows gain from the
      // ring's deeper prefetch and fp32 x; int8 8192x8192 18.4 us against 20.4 in the
      // streaming kernel, int4 20.5 against 22.6.  int8 with fewer than 48 rows per SM
      // leaves most ring warps without a row group: 4096x16384 20.5 us streaming
      // against 22.5, 4096x28672 30.2 against 33.3, 4096x8192 a tie)
      kernel = GEMV_KERNEL_BATCHED;
    } else if (M >= 65536) {
      kernel = GEMV_KERNEL_WARP_PER_ROW;
    } else if (B == 1 && M >= (int64_t)num_sms * (dtype == GEMV_DTYPE_F32 ? 16 : 12)) {
      // (16-bit and int8 rows stream from 12 rows per SM: bf16 2048x8192 12.4 us
      // against 14.2 block per row, int8 10.3 against 12.3)
      // fp32 rows of 4096 or more elements whose row walk would leave the streaming
      // warps unbalanced (rows per warp well short of a whole number): one warp per row
      // instead (14336x4096 38.9 us against 41.4, 4096x32768 90.5 against 122.6;
      // 16384x4096 streams)
      const int64_t walkers = (int64_t)num_sms * 4 * (kStreamThreads / 32);  // 4 fp32 CTAs per SM
      const int64_t turns = ceil_div(M, walkers);
      const bool unbalanced = dtype == GEMV_DTYPE_F32 && nch >= 1024 && 4 * M < 3 * turns * walkers;
      kernel = unbalanced ? GEMV_KERNEL_WARP_PER_ROW : GEMV_KERNEL_STREAM;
    } else if (M >= (int64_t)num_sms * 16 || nch <= kPlanThreads) {
      kernel = GEMV_KERNEL_WARP_PER_ROW;  // many rows, or rows of at most 4 KB
    } else if (M >= (int64_t)num_sms * 2 || nch < 2 * kPlanThreads) {
      kernel = GEMV_KERNEL_BLOCK_PER_ROW;
    } else {
      kernel = GEMV_KERNEL_SPLIT_K;
    }
  }

  p.kernel = kernel;
  p.unroll = 1;
  p.x_staging = GEMV_X_GLOBAL;
  switch (kernel) {
    case GEMV_KERNEL_ROWS_PER_WARP: {
      int lanes = param != 0 ? param : next_pow2(nch < 1 ? 1 : nch);
      if (lanes > 16) lanes = 16;
      p.lanes_per_row = lanes;
      const int64_t groups = ceil_div(M, kPlanThreads / lanes);
      p.grid = groups < (int64_t)num_sms * 32 ? groups : (int64_t)num_sms * 32;
      break;
    }
    case GEMV_KERNEL_WARP_PER_ROW: {
      p.lanes_per_row = 32;
      p.unroll = kUnrollWarpRow;
      const int64_t groups = ceil_div(M, kPlanThreads / 32);
      p.grid = groups < (int64_t)num_sms * 32 ? groups : (int64_t)num_sms * 32;
      break;
    }
    case GEMV_KERNEL_SCALAR: {
      int lanes = param != 0 ? param : (K <= 4 ? 4 : 32);
      p.lanes_per_row = lanes;
      const int64_t groups = ceil_div(M, kPlanThreads / lanes);
      p.grid = groups < (int64_t)num_sms * 32 ? groups : (int64_t)num_sms * 32;
      break;
    }
    case GEMV_KERNEL_BLOCK_PER_ROW: {
      p.unroll = kUnrollBlockRow;
      p.grid = M < (int64_t)num_sms * 16 ? M : (int64_t)num_sms * 16;
      break;
    }
    case GEMV_KERNEL_SPLIT_K: {
      int64_t s = param;
      if (s <= 0) {
        s = ceil_div((int64_t)num_sms * 4, M);
        const int64_t cap = nch / kPlanThreads;  // at least one chunk per thread
        if (s > cap) s = cap;
        if (s < 2) s = 2;
      }
      if (s > nch) s = nch;
      if (s > 65535) s = 65535;
      const int64_t per = ceil_div(nch, s);
      s = ceil_div(nch, per);  // no empty slices
      p.splits = (int)s;
      p.unroll = kUnrollBlockRow;
      p.grid = M < (int64_t)num_sms * 16 ? M : (int64_t)num_sms * 16;
      p.workspace_bytes = s * (int64_t)B * M * 4;
      break;
    }
    case GEMV_KERNEL_BATCHED: {
      // x is staged once per CTA, so the grid is persistent: one 512-thread CTA
      // per SM; each warp carries R rows.
      // x[0..NB) is staged (vectors B..NB-1 zero): the inner loops have no branch
      p.threads = kBatchedThreads;
      p.grid = num_sms;
      // variant: forced (param = variant + 1), else the row-pair kernel where it
      // measured faster (GB300, event means in us, clean-L2 flush), else the ring,
      // with mixed-precision FMAs for fp16/bf16 with 2 vectors (bf16 14336x4096
      // B = 2 23.9 against 26.6 packed) and packed FMAs otherwise.  Row pair:
      // - at most one row pair per warp (M <= 2 x 16 x SMs) with 4..16 vectors (int8:
      //   2..16), fp32 with 3..4 vectors excepted (bf16 4096x4096 B = 4 13.1 against
      //   14.1 ring, 4096x8192 20.3 against 21.3; int8 4096x4096 B = 2 10.3 against
      //   12.3, 2048x8192 B = 4 12.3 against 16.2; fp32 4096x4096 B = 8 20.2 against
      //   20.8, but B = 4 19.5 against 16.6 ring, 2048x4096 16.6 against 12.9);
      // - above that, at most one ring row group per warp (M <= 4 x 16 x SMs) for 4
      //   vectors of int8 and 5..8 of fp16/bf16 (int8 8192x8192 B = 4 26.4 against
      //   27.3 ring; bf16 8192x8192 B = 8 36.9 against 40.9).  The ring takes the
      //   other shapes of that range since its x staging lost its divisions: bf16
      //   6144x4096 B = 4 16.1 against 18.5, 8192x8192 B = 4 30.5 against 32.6; int8
      //   6144x4096 B = 2 12.3 against 14.4, 9216x4096 B = 8 24.6 against 26.6;
      // - 16 vectors of fp16/bf16/fp32 whenever x fits (bf16 14336x4096 53.2 against
      //   61.4 mixed ring, 128256x4096 409.6 against 450.6, fp32 32768x2048 75.8
      //   against 82.0; int8 14336x4096 is a tie and keeps the ring);
      // - 8 vectors of fp16/bf16 whose ring would read x as stored (f16 16384x6144
      //   53.2 against 59.4; with fp32 x the ring wins at scale: bf16 28672x4096
      //   55.3 against 59.4);
      // - x too large for the ring, or for its whole K (the ring's slices).
      const int64_t ring_group_rows = ring_rows(p.nb, dtype == GEMV_DTYPE_W4, dtype == GEMV_DTYPE_F32);
      const bool one_group_per_warp = M <= (int64_t)num_sms * 16 * ring_group_rows;
      const bool one_pair_per_warp = M <= (int64_t)num_sms * 16 * 2;
      int v;
      if (param != 0) {
        v = param - 1;
      } else if (half16 && p.nb == 4 && M <= 2048 && mixed_ok && rslices == 1) {
        // 4 vectors of few 16-bit rows: the mixed-precision ring (bf16 1024x16384
        // 24.6 us against 26.8 in the row pairs, 2048x16384 26.8 against 28.7, 2048x8192
        // 16.6 against 18.4; from 4096 rows the row pairs lead: 4096x14336 29.2 against
        // 32.2)
        v = GEMV_BATCHED_RING_MIXED;
      } else if (rstage < 0 ||
                 (rowpair_ok &&
                  (rslices > 1 ||
                   (one_pair_per_warp && (p.nb >= 8 || (p.nb == 4 && dtype != GEMV_DTYPE_F32) ||
                                          (dtype == GEMV_DTYPE_W8 && p.nb >= 2))) ||
                   (one_group_per_warp && ((dtype == GEMV_DTYPE_W8 && p.nb == 4) || (half16 && p.nb == 8))) ||
                   (p.nb == 16 && dtype != GEMV_DTYPE_W8) ||
                   (p.nb == 8 && half16 && rstage == GEMV_X_SMEM)))) {
        v = GEMV_BATCHED_ROWPAIR;
      } else {
        // (8 vectors over K slices read x as stored as well: bf16 1024x16384 B = 8
        // 23.4 us mixed against 25.6 packed, 4096x14336 41.8 against 42.1)
        v = (half16 && (p.nb == 16 || p.nb == 2 || (p.nb == 8 && rslices > 1)) && mixed_ok)
                ? GEMV_BATCHED_RING_MIXED
                : GEMV_BATCHED_RING;
      }
      p.variant = v;
      if (v == GEMV_BATCHED_ROWPAIR) {
        p.rows_per_warp = rowpair_rows(p.nb, half16);  // (SwiGLU: 2, the gate and up row)
        p.x_staging = GEMV_X_SMEM;
        p.unroll = p.rows_per_warp == 4 ? 1 : 2;
        p.smem_bytes = (int)((int64_t)p.nb * K * sx);
      } else {
        // ring: R rows per warp, a G = slots / R step ring; the mixed form reads x as
        // stored.  Over rslices K slices (x too large to stage whole): grid.x CTAs per
        // slice, one CTA per SM in all, partial sums [slice][b][m], then a second pass.
        const int xs = v == GEMV_BATCHED_RING_MIXED ? GEMV_X_SMEM : rstage;
        p.rows_per_warp = v == GEMV_BATCHED_RING_MIXED ? 2 : ring_rows(p.nb, dtype == GEMV_DTYPE_W4, dtype == GEMV_DTYPE_F32);
        p.x_staging = xs;
        p.unroll = ring_slots(p.nb) / p.rows_per_warp;
        p.smem_bytes = (int)((int64_t)p.nb * rcps * vec * (xs == GEMV_X_SMEM_FP32 ? 4 : sx) + ring_bytes(p.nb) + rextra);
        p.splits = rslices;
        p.grid = num_sms / rslices > 0 ? num_sms / rslices : 1;
        p.workspace_bytes = rslices > 1 ? (int64_t)rslices * B * M * 4 : 0;
      }
      break;
    }
    case GEMV_KERNEL_TC: {
      // N = B rounded up to 16 (p.nb); one 128-thread CTA per 128-row tile and K
      // slice (p.splits slices of p.unroll k-tiles)
      if (B <= GEMV_MAX_BATCH) p.nb = (B + 15) / 16 * 16;
      const int64_t tiles = ceil_div(M, kTcPlanTileM);
      // More tiles than two CTAs per SM hold at once, unsplit: the persistent form
      // (one CTA per SM walks its tiles, deep ring, each tile's epilogue behind the next
      // tile's copies; forced: param / 1000000 % 10 = 1 on, 2 off).  Measured on bf16
      // 128256x4096 (us, against two CTAs per SM): B = 32 169.3 / 176.7, 64 176.4 /
      // 188.7, 80 184.4 / 204.8, 128 191.6 / 222.8, 256 253.8 / 304.5.
      const int pk = param % 1000, ps = param / 1000 % 10, pp = param / 1000000 % 10;
      const bool persist = K > 0 && ps <= 1 && pp != 2 && (pp == 1 || tiles > 2 * (int64_t)num_sms);
      // 64-column swizzle atoms per stage (forced: param / 100000 % 10 in 1..2); the
      // persistent form takes 2 for every N (B = 128: 191.6 us against 266.2 with 1)
      const int pa = param / 100000 % 10;
      const int atoms = pa == 1 || pa == 2 ? pa : persist ? 2 : tc_plan_atoms(p.nb);
      const int64_t ktiles = K > 0 ? ceil_div(K, (int64_t)kTcPlanTileK * atoms) : 1;
      // K slices so that all CTAs run in one wave (as many per SM as shared memory
      // allows).  A deep ring (one CTA per SM) for up to 64 vectors while the tiles
      // cover half the SMs or more but not all of them; otherwise two CTAs per SM,
      // which for few tiles doubles the K slices (measured, us: 14336 rows B = 32
      // 30.7 deep against 33.6, B = 64 33.5 against 37.7, B = 128 49.1 against 46.3;
      // 4096 rows B = 64 23.3 against 21.4; 28672 rows B = 32 57.3 against 45.1)
      // (and 64 or more vectors on at most a quarter as many tiles as SMs: K slices on
      // deep rings, one CTA per SM; f16 4096x4096 B = 256 34.6 us against 40.1 on two
      // 100 KB rings per SM, B = 64 18.8 against 20.1)
      const bool deep = (p.nb <= 64 && tiles < num_sms && 2 * tiles >= num_sms) ||
                        (p.nb >= 64 && 4 * tiles <= num_sms);
      // (forced: param % 1000 in 32..220 is the ring size in KB, param / 1000 % 10 in
      // 1..8 the number of K slices, param / 10000 % 10 the cluster scheduling
      // preference: 1 spread, 2 load balancing; param / 100000 % 10 the atoms above)
      // (the persistent form adds 8 KB of epilogue staging after its ring: at most 200 KB)
      int ring_kb = pk >= 32 && pk <= 220 ? pk : (deep || persist) ? 200 : 100;
      if (persist && ring_kb > 200) ring_kb = 200;
      const int64_t smem = (int64_t)tc_plan_stages(p.nb, ring_kb, atoms) * tc_plan_stage_bytes(p.nb, atoms) + 1024;
      int64_t per_sm = kSmemPerSm / (smem + 1024);
      if (per_sm < 1) per_sm = 1;
      // (the slices of a tile run as one cluster and are summed inside the kernel, so
      // they are at most the cluster size)
      int64_t s = (int64_t)num_sms * per_sm / tiles;
      if (ps >= 1 && ps <= kTcMaxCluster) s = ps;
      if (s > ktiles) s = ktiles;
      if (s > kTcMaxCluster) s = kTcMaxCluster;
      if (s < 1) s = 1;
      const int64_t per = ceil_div(ktiles, s);
      s = ceil_div(ktiles, per);  // no empty slice
      p.threads = kTcPlanThreads;
      p.grid = tiles;
      p.splits = (int)s;
      p.unroll = (int)per;
      p.lanes_per_row = kTcPlanThreads;
      if (persist) {  // (threads = 192 marks the form; k-tiles per tile in unroll)
        p.threads = kTcPlanPersistThreads;
        p.lanes_per_row = kTcPlanPersistThreads;
        p.grid = tiles < num_sms * per_sm ? tiles : num_sms * per_sm;  // (per_sm: 1 with the deep ring)
        p.splits = 1;
        p.unroll = (int)ktiles;
      }
      p.rows_per_warp = atoms;  // (for this kernel: 64-column atoms per stage)
      p.smem_bytes = (int)smem;
      p.workspace_bytes = 0;
      p.variant = param / 10000 % 10;  // (forced only) cluster scheduling preference
      break;
    }
    case GEMV_KERNEL_XSPLIT: {
      // one 512-thread CTA per SM (at most one per row) over a contiguous block of
      // rows; each thread J chunks of every row, x in registers
      p.lanes_per_row = kXsplitThreads;
      p.threads = kXsplitThreads;
      p.unroll = xs_j;
      p.x_staging = GEMV_X_REGS;
      p.smem_bytes = xsplit_depth(xs_j) * xs_j * kXsplitThreads * 16;
      p.grid = M < num_sms ? M : num_sms;
      break;
    }
    case GEMV_KERNEL_STREAM: {
      // fp32 rows: x through L1, four CTAs per SM; 16-bit, int8 and int4 rows: x in
      // shared memory (when it fits in 96 KB; int4: widened to fp32), two CTAs per
      // SM, deeper unroll.
      p.lanes_per_row = 32;
      p.rows_per_warp = 1;
      p.threads = kStreamThreads;
      const bool f32 = dtype == GEMV_DTYPE_F32;
      p.unroll = f32 ? 2 : 4;
      p.x_staging = (!f32 && K * sx <= kStreamSmemMax) ? GEMV_X_SMEM : GEMV_X_GLOBAL;
      // int4 decodes 32 weights per chunk: x widened once per CTA takes the widening
      // off every row (8192x8192 22.5 us against 24.4; for the other types no gain)
      if (dtype == GEMV_DTYPE_W4 && K * 4 <= kStreamSmemMax) p.x_staging = GEMV_X_SMEM_FP32;
      // forced: param = x staging + 1 (GEMV_X_GLOBAL, GEMV_X_SMEM, GEMV_X_SMEM_FP32)
      if (param == 1 + GEMV_X_GLOBAL) p.x_staging = GEMV_X_GLOBAL;
      if (param == 1 + GEMV_X_SMEM && K * sx <= kStreamSmemMax) p.x_staging = GEMV_X_SMEM;
      if (param == 1 + GEMV_X_SMEM_FP32 && !f32 && K * 4 <= kStreamSmemMax) p.x_staging = GEMV_X_SMEM_FP32;
      p.smem_bytes = p.x_staging == GEMV_X_SMEM ? (int)(K * sx) : p.x_staging == GEMV_X_SMEM_FP32 ? (int)(K * 4) : 0;
      // Every CTA of the persistent grid is launched even when M needs fewer warps:
      // rows are dealt to CTAs round-robin, so each SM gets an equal share.
      const int64_t per_sm = f32 ? 4 : 2;
      p.grid = per_sm * num_sms;
      break;
    }
    default:
      return GEMV_ERR_INVALID_VALUE;
  }
  *out = p;
  return GEMV_SUCCESS;
}

}  // namespace gemv

extern "C" gemv_status_t gemv_plan_for(gemv_dtype_t dtype, int64_t M, int64_t K, int B,
                                       int aligned16, int num_sms, gemv_plan_t *plan) {
  return gemv::plan((int)dtype, M, K, B, aligned16 != 0, num_sms, GEMV_KERNEL_AUTO, 0, plan);
}
