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

int elem_bytes_a(int dtype);
int elem_bytes_x(int dtype);
// Elements of A in one 16-byte chunk.
int chunk_elems(int dtype);

// Defined in gemv_api.cu.
void record_cuda_error(int e);
void count_launches(int n);

gemv_status_t plan(int dtype, int64_t M, int64_t K, int B, bool aligned16, int num_sms,
                   int force_kernel, int force_param, gemv_plan_t *out);

}  // namespace gemv
