// Internal interface between the C-ABI entry points, the dispatcher and the
// per-dtype launch units.
#pragma once

#include <stdint.h>

#include "../../include/gemv.h"

namespace gemv {

constexpr int kPlanThreads = 256;
// Largest x[0..B) the batched kernel stages in shared memory.
constexpr int64_t kBatchedSmemMax = 200 * 1024;
// Shared memory one SM can give to resident CTAs (sm_100-class: 228 KB).
constexpr int64_t kSmemPerSm = 228 * 1024;
// Largest x the streaming kernel copies into shared memory.
constexpr int64_t kStreamSmemMax = 96 * 1024;
constexpr int kBatchedThreads = 512;
// Row-pair kernel (GEMV_BATCHED_ROWPAIR): rows per warp.  16 vectors of 16-bit rows
// take 4 (one chunk per lane in flight per row): each x chunk read from shared
// memory, and each x half split out of its word, then feeds 4 rows instead of 2
// (event means on GB300, us: bf16 128256x4096 B = 16 397.1 -> 344.1, 28672x4096
// 96.0 -> 82.7, 14336x4096 51.2 -> 46.7, f16 4096x4096 21.5 -> 20.5).  Otherwise 2
// (two chunks per lane in flight per row).
constexpr int rowpair_rows(int nb, bool mixed16) { return (nb == 16 && mixed16) ? 4 : 2; }
// BATCHED ring kernel: R rows per warp and a per-thread cp.async ring of G = slots / R
// steps: 16 warps x slots x 512 bytes after x (ring_slots below).  R = 2 for 16 vectors (the
// accumulators' registers), for int4 with 3 or more vectors (32 weights per chunk to
// decode) and for fp32 with 4 vectors, else 4 (measured on GB300, event means in us:
// int4 8192x8192 B = 1 18.8 with R = 4 against 19.6 with R = 2, int4 14336x4096
// B = 1 16.7 against 18.3, B = 4 33.2 either way; fp32 8192x4096 B = 4 27.0 against
// 28.6; bf16 14336x4096 B = 4 29.3 against 27.1 and int8 8192x8192 B = 4 32.8
// against 32.5 keep R = 4).  SwiGLU: R = 2.
constexpr int64_t kRingSmemMax = 227 * 1024;  // dynamic shared memory one CTA may use
// Ring slots per thread (G x R): 8 (64 KB per CTA), and 16 (128 KB) for one vector,
// whose steps are short and whose warps wait on HBM (ncu: long_scoreboard the top
// stall).  Event means (us, A/B in one run, 8 -> 16 slots): int8 16384x8192 B = 1
// 28.3 -> 26.9, 32768x8192 47.8 -> 46.9, 14336x4096 16.6 -> 16.5, 8192x8192 18.4
// either way; int4 within 1.3 %.
constexpr int ring_slots(int nb) { return nb == 1 ? 16 : 8; }
constexpr int64_t ring_bytes(int nb) { return (int64_t)16 * ring_slots(nb) * 512; }
constexpr int64_t ring_scale_bytes(int nb) { return (int64_t)16 * ring_slots(nb) * 32 * 4; }  // int4: a group scale per slot
constexpr int ring_rows(int nb, bool grouped, bool a32) {
  return nb == 16 ? 2 : grouped ? (nb <= 2 ? 4 : 2) : (a32 && nb == 4) ? 2 : 4;
}
constexpr int kStreamThreads = 512;
// 16-byte chunks in flight per lane: warp-per-row and block-per-row kernels.
constexpr int kUnrollWarpRow = 4;
constexpr int kUnrollBlockRow = 4;

// XSPLIT: 512 threads split K; J chunks per thread; rows stream through a
// cp.async ring of 16 / J rows (P rows per commit group, 4 groups in flight), so
// the ring is 16 * 8 KB = 128 KB for every J; x slice <= 64 fp32 registers.
constexpr int kXsplitThreads = 512;
constexpr int kXsplitMaxXRegs = 64;
constexpr int kXsplitGroups = 4;
constexpr int xsplit_rows_per_group(int J) { return J == 1 ? 4 : J == 2 ? 2 : 1; }
constexpr int xsplit_depth(int J) { return xsplit_rows_per_group(J) * kXsplitGroups; }

// TC (tcgen05, fp16/bf16, B > 16): 128-row tiles, stages of one or two 64-column
// swizzle atoms along K; as many stages (at most 8) as fit in the ring, plus 1024
// bytes to align them.
constexpr int kTcPlanThreads = 128;
constexpr int kTcPlanPersistThreads = 192;  // the persistent form: copy, MMA and 4 epilogue warps
constexpr int kTcPlanMaxStages = 16;  // pipeline stages in one CTA's ring
// K slices of one row tile run as one thread-block cluster (the portable maximum size)
constexpr int kTcMaxCluster = 8;
constexpr int kTcPlanTileM = 128;
constexpr int kTcPlanTileK = 64;
// 64-column atoms per stage: two for N <= 64, one above.
constexpr int tc_plan_atoms(int n) { return n <= 64 ? 2 : 1; }
constexpr int tc_plan_stage_bytes(int n, int atoms) { return (kTcPlanTileM + n) * kTcPlanTileK * 2 * atoms; }
constexpr int tc_plan_stage_bytes(int n) { return tc_plan_stage_bytes(n, tc_plan_atoms(n)); }
// ring_kb: 200 (one CTA per SM, the deeper ring) when the row tiles leave SMs
// free, 100 (two CTAs per SM) when there are at least as many tiles as SMs.
constexpr int tc_plan_stages(int n, int ring_kb, int atoms) {
  return ring_kb * 1024 / tc_plan_stage_bytes(n, atoms) < kTcPlanMaxStages ? ring_kb * 1024 / tc_plan_stage_bytes(n, atoms)
                                                                          : kTcPlanMaxStages;
}
constexpr int tc_plan_stages(int n, int ring_kb) {
  return tc_plan_stages(n, ring_kb, tc_plan_atoms(n));
}

// Tensor maps of A (K x M) and x (K x B), 16-bit values, boxes 64 x 128 and 64 x N,
// 128-byte swizzle, written to map_a and map_x (CUtensorMap, 128 bytes each).
// Defined in gemv_api.cu; false if the driver's encoder is missing or refuses.
bool tc_tensor_maps(int dtype, const void *A, const void *x, int64_t M, int64_t K, int B, int N, void *map_a,
                    void *map_x);

int elem_bytes_a(int dtype);
int elem_bytes_x(int dtype);
// Elements of A in one 16-byte chunk.
int chunk_elems(int dtype);

// Defined in gemv_api.cu.
void record_cuda_error(int e);
void count_launches(int n);
int launch_overlap();  // the calling thread's gemv_set_launch_overlap mode

gemv_status_t plan(int dtype, int64_t M, int64_t K, int B, bool aligned16, int num_sms,
                   int force_kernel, int force_param, gemv_plan_t *out);

}  // namespace gemv
