// Plan -> kernel instantiation.  Included once per storage type (gemv_<dtype>.cu),
// so the four types compile in parallel.
#pragma once

#include <cuda_runtime.h>

#include <cstring>
#include <utility>

#include "gemv_kernels.cuh"
#include "gemv_plan.h"
#include "gemv_tc.cuh"

namespace gemv {

// Every launch goes through cudaLaunchKernelEx: with a.pdl it is a programmatic
// dependent launch, which the GPU may start while the previous kernel on the stream
// is finishing (the kernel then waits for it with griddepcontrol.wait, see
// pdl_enter, before touching memory that kernel could have written).
template <class... P, class... A2>
cudaError_t launch_k(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int pdl,
                     A2 &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl != 0) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, std::forward<A2>(args)...);
}

// The same, as clusters of (1, cy, 1) CTAs.
template <typename... P, typename... A2>
cudaError_t launch_k_cluster(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int pdl,
                             int cy, int policy, A2 &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)cy;
  attr[0].val.clusterDim.z = 1;
  int na = 1;
  if (pdl != 0) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (policy == 1 || policy == 2) {
    attr[na].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
    attr[na].val.clusterSchedulingPolicyPreference =
        policy == 1 ? cudaClusterSchedulingPolicySpread : cudaClusterSchedulingPolicyLoadBalancing;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<A2>(args)...);
}

// Dynamic shared memory above 48 KB has to be allowed per kernel.
template <typename Kern>
cudaError_t allow_smem(Kern kern, int bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <class Op, int NB>
cudaError_t launch_rowteam(const gemv_plan_t &p, const Args &a, cudaStream_t s) {
  const dim3 grid((unsigned)p.grid), block(kThreads);
  if (p.kernel == GEMV_KERNEL_SCALAR) {
    switch (p.lanes_per_row) {
      case 4: return launch_k(k_rowteam<Op, 4, NB, 1, false>, grid, block, 0, s, a.pdl, a);
      default: return launch_k(k_rowteam<Op, 32, NB, 1, false>, grid, block, 0, s, a.pdl, a);
    }
    return cudaSuccess;
  }
  switch (p.lanes_per_row) {
    case 1: return launch_k(k_rowteam<Op, 1, NB, 1, true>, grid, block, 0, s, a.pdl, a);
    case 2: return launch_k(k_rowteam<Op, 2, NB, 1, true>, grid, block, 0, s, a.pdl, a);
    case 4: return launch_k(k_rowteam<Op, 4, NB, 1, true>, grid, block, 0, s, a.pdl, a);
    case 8: return launch_k(k_rowteam<Op, 8, NB, 1, true>, grid, block, 0, s, a.pdl, a);
    case 16: return launch_k(k_rowteam<Op, 16, NB, 1, true>, grid, block, 0, s, a.pdl, a);
    case 32: return launch_k(k_rowteam<Op, 32, NB, kUnrollWarpRow, true>, grid, block, 0, s, a.pdl, a);
    default: return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

template <class Op, int NB>
cudaError_t launch_batched(const gemv_plan_t &p, const Args &a, float *ws, cudaStream_t s) {
  {
    constexpr int T = kBatchedThreads;
    static_assert(T == 512, "the ring kernel is built for 512 threads");
    const dim3 block(T);
    const bool sw = a.half > 0;  // SwiGLU: gate and up row of one output per row pair
    if (p.splits < 1 || (p.splits > 1 && (ws == nullptr || sw || p.variant == GEMV_BATCHED_ROWPAIR)))
      return cudaErrorInvalidValue;
    // the ring over K slice blockIdx.y (p.splits slices of chunks_per_split chunks),
    // then with several slices the fixed-order sum of the slices and the epilogue
    const int64_t nch = a.K / Op::VEC;
    const int64_t cps = (nch + p.splits - 1) / p.splits;
    auto ring = [&](auto kern) -> cudaError_t {
      cudaError_t e = allow_smem(kern, p.smem_bytes);
      if (e != cudaSuccess) return e;
      e = launch_k(kern, dim3((unsigned)p.grid, (unsigned)p.splits), block, (size_t)p.smem_bytes, s, a.pdl, a,
                   p.splits > 1 ? ws : nullptr, cps);
      if (e != cudaSuccess || p.splits == 1) return e;
      int64_t g = (a.M + kThreads - 1) / kThreads;  // (b, m): grid row b, m grid-strided
      if (g > 65535) g = 65535;
      return launch_k(k_splitk_reduce<Op>, dim3((unsigned)g, (unsigned)a.B), dim3(kThreads), 0, s, a.pdl, a,
                      (const float *)ws, p.splits);
    };
    constexpr int SX = (int)sizeof(typename Op::TX);
    constexpr bool A16 = sizeof(typename Op::TA) == 2;  // mixed-precision FMAs need 16-bit A
    switch (p.variant) {
      case GEMV_BATCHED_ROWPAIR:
        if constexpr (!Op::GROUPED && NB >= 2) {  // not built for int4's group scales
          // R rows per warp (SwiGLU: the gate and up row of one output), U chunks each
          constexpr int R = rowpair_rows(NB, A16 && SX == 2), U = R == 4 ? 1 : 2;
          auto kern = sw ? k_batched2<Op, NB, 2, 2, T, true> : k_batched2<Op, NB, R, U, T>;
          cudaError_t e = allow_smem(kern, p.smem_bytes);
          if (e != cudaSuccess) return e;
          return launch_k(kern, dim3((unsigned)p.grid), block, (size_t)p.smem_bytes, s, a.pdl, a);
        }
        return cudaErrorInvalidValue;
      case GEMV_BATCHED_RING: {
        constexpr int R = ring_rows(NB, Op::GROUPED, sizeof(typename Op::TA) == 4), G = ring_slots(NB) / R;
        constexpr int MODE = NB >= 8 ? kRingPairs : kRingEvenOdd;
        const bool x32 = p.x_staging == GEMV_X_SMEM_FP32 || SX == 4;
        if (!sw && (p.rows_per_warp != R || p.unroll != G)) return cudaErrorInvalidValue;
        if (sw)
          return x32 ? ring(k_batch_ring<Op, NB, 2, 4, 4, true, MODE>) : ring(k_batch_ring<Op, NB, 2, 4, SX, true, MODE>);
        return x32 ? ring(k_batch_ring<Op, NB, R, G, 4, false, MODE>) : ring(k_batch_ring<Op, NB, R, G, SX, false, MODE>);
      }
      case GEMV_BATCHED_RING_MIXED:
        if constexpr (A16 && SX == 2 && Op::VEC == 8 && NB >= 2) {
          if (p.rows_per_warp != 2 || p.x_staging != GEMV_X_SMEM) return cudaErrorInvalidValue;
          return sw ? ring(k_batch_ring<Op, NB, 2, 4, 2, true, kRingMixed>)
                    : ring(k_batch_ring<Op, NB, 2, 4, 2, false, kRingMixed>);
        }
        return cudaErrorInvalidValue;
      default:
        return cudaErrorInvalidValue;
    }
  }
}

template <class Op>
cudaError_t launch_stream(const gemv_plan_t &p, const Args &a, cudaStream_t s) {
  constexpr int T = kStreamThreads;
  const dim3 grid((unsigned)p.grid), block(T);
  const bool sw = a.half > 0;  // SwiGLU row pairs
  auto run = [&](auto kern) -> cudaError_t {
    cudaError_t e = allow_smem(kern, p.smem_bytes);
    if (e != cudaSuccess) return e;
    return launch_k(kern, grid, block, (size_t)p.smem_bytes, s, a.pdl, a);
  };
  if (p.x_staging == GEMV_X_SMEM_FP32) {
    if constexpr (sizeof(typename Op::TX) == 2) {
      return sw ? run(k_stream<Op, 4, T, 2, true>) : run(k_stream<Op, 4, T, 2>);
    }
    return cudaErrorInvalidValue;
  }
  if (p.x_staging == GEMV_X_SMEM)
    return sw ? run(k_stream<Op, 4, T, 1, true>) : (p.unroll == 2 ? run(k_stream<Op, 2, T, 1>) : run(k_stream<Op, 4, T, 1>));
  return sw ? (p.unroll == 2 ? run(k_stream<Op, 2, T, 0, true>) : run(k_stream<Op, 4, T, 0, true>))
            : (p.unroll == 2 ? run(k_stream<Op, 2, T, 0>) : run(k_stream<Op, 4, T, 0>));
}

template <class Op, int NB, int J>
cudaError_t launch_xsplit_j(const gemv_plan_t &p, const Args &a, cudaStream_t s) {
  if constexpr (Op::GROUPED || (NB != 1 && NB != 2 && NB != 4) || J * NB * Op::VEC > kXsplitMaxXRegs) {
    return cudaErrorInvalidValue;  // not built; the planner never picks it
  } else {
    auto kern = k_xsplit<Op, NB, J, xsplit_rows_per_group(J), kXsplitGroups>;
    cudaError_t e = allow_smem(kern, p.smem_bytes);
    if (e != cudaSuccess) return e;
    return launch_k(kern, dim3((unsigned)p.grid), dim3(kXsThreads), (size_t)p.smem_bytes, s, a.pdl, a);
  }
}

template <class Op, int NB>
cudaError_t launch_xsplit(const gemv_plan_t &p, const Args &a, cudaStream_t s) {
  switch (p.unroll) {
    case 1: return launch_xsplit_j<Op, NB, 1>(p, a, s);
    case 2: return launch_xsplit_j<Op, NB, 2>(p, a, s);
    case 4: return launch_xsplit_j<Op, NB, 4>(p, a, s);
    default: return cudaErrorInvalidValue;
  }
}

template <class Op, int NB>
cudaError_t launch_nb(const gemv_plan_t &p, const Args &a, float *ws, cudaStream_t s) {
  switch (p.kernel) {
    case GEMV_KERNEL_ROWS_PER_WARP:
    case GEMV_KERNEL_WARP_PER_ROW:
    case GEMV_KERNEL_SCALAR:
      return launch_rowteam<Op, NB>(p, a, s);
    case GEMV_KERNEL_BLOCK_PER_ROW:
      return launch_k(k_blockrow<Op, NB, kUnrollBlockRow>, dim3((unsigned)p.grid, 1), dim3(kThreads), 0, s, a.pdl,
                      a, (float *)nullptr, (int64_t)(a.K / Op::VEC));
    case GEMV_KERNEL_SPLIT_K: {
      const int64_t nch = a.K / Op::VEC;
      const int64_t per = (nch + p.splits - 1) / p.splits;
      cudaError_t e = launch_k(k_blockrow<Op, NB, kUnrollBlockRow>, dim3((unsigned)p.grid, (unsigned)p.splits),
                               dim3(kThreads), 0, s, a.pdl, a, ws, per);
      if (e != cudaSuccess) return e;
      int64_t g = (a.M + kThreads - 1) / kThreads;  // (b, m): grid row b, m grid-strided
      if (g > 65535) g = 65535;
      return launch_k(k_splitk_reduce<Op>, dim3((unsigned)g, (unsigned)a.B), dim3(kThreads), 0, s, a.pdl, a,
                      (const float *)ws, p.splits);
    }
    case GEMV_KERNEL_BATCHED:
      return launch_batched<Op, NB>(p, a, ws, s);
    case GEMV_KERNEL_STREAM:
      if constexpr (NB == 1) return launch_stream<Op>(p, a, s);
      return cudaErrorInvalidValue;
    case GEMV_KERNEL_XSPLIT:
      return launch_xsplit<Op, NB>(p, a, s);
    default:
      return cudaErrorInvalidValue;
  }
}

// fp16/bf16 with more than 16 vectors (or forced): the tensor-core kernel; a split K
// range runs as clusters of the tile's slices, reduced inside the kernel.
template <class Op>
cudaError_t launch_tc(const gemv_plan_t &p, const Args &a, float *, cudaStream_t s) {
  if constexpr (!TcFormat<Op>::ok) {
    return cudaErrorInvalidValue;  // the planner never picks it for these types
  } else {
    if (p.nb < 16 || p.nb > kTcMaxN || p.nb % 16 != 0 || p.splits < 1 || p.splits > kTcMaxCluster)
      return cudaErrorInvalidValue;
    const int ka = p.rows_per_warp == 1 || p.rows_per_warp == 2 ? p.rows_per_warp : tc_atoms(p.nb);
    const int sb = tc_stage_bytes(p.nb, ka), stages = (p.smem_bytes - 1024) / sb;
    if (stages < 2 || stages > kTcMaxStages || p.smem_bytes != stages * sb + 1024) return cudaErrorInvalidValue;
    CUtensorMap map_a, map_x;
    std::memset(&map_a, 0, sizeof map_a);
    std::memset(&map_x, 0, sizeof map_x);
    const int dt = TcFormat<Op>::bf16 ? GEMV_DTYPE_BF16 : GEMV_DTYPE_F16;
    if (a.K > 0 && !tc_tensor_maps(dt, a.A, a.x, a.M, a.K, a.B, p.nb, &map_a, &map_x)) return cudaErrorInvalidValue;
    if (p.threads == kTcPThreads) {  // the persistent form: one CTA per SM over its tiles
      if (p.splits != 1 || a.K <= 0 || p.grid < 1) return cudaErrorInvalidValue;
      // the ring, then the epilogue warps' staging buffers
      auto pk = ka == 2 ? k_tc_persist<Op, 2> : k_tc_persist<Op, 1>;
      const int smem = p.smem_bytes + kTcPEpBytes;
      cudaError_t e = allow_smem(pk, smem);
      if (e != cudaSuccess) return e;
      return launch_k(pk, dim3((unsigned)p.grid), dim3(kTcPThreads), (size_t)smem, s, a.pdl, map_a, map_x, a, p.nb,
                      stages);
    }
    auto kern = ka == 2 ? k_tc<Op, 2> : k_tc<Op, 1>;
    cudaError_t e = allow_smem(kern, p.smem_bytes);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)p.grid, (unsigned)p.splits);
    if (p.splits == 1)
      return launch_k(kern, grid, dim3(kTcThreads), (size_t)p.smem_bytes, s, a.pdl, map_a, map_x, a,
                      (int64_t)p.unroll, p.nb, stages);
    return launch_k_cluster(kern, grid, dim3(kTcThreads), (size_t)p.smem_bytes, s, a.pdl, p.splits, p.variant, map_a,
                            map_x, a, (int64_t)p.unroll, p.nb, stages);
  }
}

template <class Op>
cudaError_t launch(const gemv_plan_t &p, const Args &a, float *ws, cudaStream_t s) {
  if (p.kernel == GEMV_KERNEL_TC) return launch_tc<Op>(p, a, ws, s);
  switch (p.nb) {
    case 1: return launch_nb<Op, 1>(p, a, ws, s);
    case 2: return launch_nb<Op, 2>(p, a, ws, s);
    case 4: return launch_nb<Op, 4>(p, a, ws, s);
    case 8: return launch_nb<Op, 8>(p, a, ws, s);
    case 16: return launch_nb<Op, 16>(p, a, ws, s);
    default: return cudaErrorInvalidValue;
  }
}

// Defined in gemv_f32.cu, gemv_f16.cu, gemv_bf16.cu, gemv_w8.cu, gemv_w4.cu.
cudaError_t launch_f32(const gemv_plan_t &p, const Args &a, float *ws, cudaStream_t s);
cudaError_t launch_f16(const gemv_plan_t &p, const Args &a, float *ws, cudaStream_t s);
cudaError_t launch_bf16(const gemv_plan_t &p, const Args &a, float *ws, cudaStream_t s);
cudaError_t launch_w8(const gemv_plan_t &p, const Args &a, float *ws, cudaStream_t s);
cudaError_t launch_w4(const gemv_plan_t &p, const Args &a, float *ws, cudaStream_t s);

}  // namespace gemv
