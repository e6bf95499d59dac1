// k_tc: 16 < B <= 256 vectors, fp16/bf16 storage.  With more than 16 vectors the
// GEMV becomes a small-N GEMM (B multiply-adds per weight byte pair), so it runs on
// the 5th-generation tensor cores: Y^T (M x N) = A (M x K) . X^T (K x N), N = B
// rounded up to a multiple of 16, fp32 accumulation in tensor memory.
//
// One CTA of 128 threads per 128-row tile of A, and per K slice when the tiles are
// too few to occupy the SMs (split-K).  The S slices of a tile run as one thread-block
// cluster: CTA r owns rows [ceil(128 r / S), ceil(128 (r + 1) / S)) of the tile, and
// every CTA stores its partial sums of those rows into the owner's shared memory
// (distributed shared memory stores, one slot per slice); after a cluster barrier
// each owner adds its rows' S partial sums in slice order from its own shared memory
// (deterministic, no atomics, no second kernel, no global workspace).  Two threads
// run the pipeline.  A producer (lane 0 of warp 0)
// has the tensor-memory accelerator (TMA) copy each k-tile (128 x 64 or 128 x 128
// of A and N x 64/128 of x, 128-byte swizzle, zeros outside the matrix) into a free
// stage, completing on the stage's "full" mbarrier; an MMA issuer (lane 0 of warp 1)
// waits for it, issues the stage's MMAs (K = 16 each) and commits them to the
// stage's "empty" mbarrier, which frees the stage for the producer.  The 128-byte
// swizzle TMA writes is the tensor cores' canonical K-major layout: 8-row x 128-byte
// atoms, 1024 bytes apart.  No CTA barrier runs inside the loop.
//
// Every wait on an mbarrier is bounded (globaltimer); on timeout the CTA ORs a bit
// into the device status word, waits (bounded) for its MMAs and copies in flight,
// frees its tensor memory and returns.
//
// k_tc_persist (below) is the form for more tiles than two CTAs per SM hold: one CTA
// per SM over its tiles, with copy, MMA and epilogue warps and two accumulators.
#pragma once

#include <cuda.h>  // CUtensorMap (the encoder is fetched from the driver at run time)

#include "gemv_kernels.cuh"

namespace gemv {

constexpr int kTcThreads = 128;  // one warpgroup: warp w reads TMEM lanes 32w..32w+31
constexpr int kTcM = 128;        // rows per tile (the MMA's M)
constexpr int kTcK = 64;         // K per stage: one 128-byte swizzle atom of 16-bit values
constexpr int kTcMaxStages = 16;
constexpr int kTcMaxN = 256;
constexpr int kTcMaxSlices = 8;  // K slices of a tile: one cluster (the portable maximum size)

// device status bits (ORed into *Args::status)
constexpr int kTcStatusMma = 16;   // a copy or an MMA commit did not arrive in time
constexpr int kTcStatusDrain = 32; // the final wait for work in flight ran out

__device__ __forceinline__ uint32_t tc_smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void tc_mbar_init(uint64_t *b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(tc_smem_u32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ bool tc_mbar_try_wait(uint64_t *b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(tc_smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t tc_global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of the given parity; false after timeout_ns.
__device__ __forceinline__ bool tc_mbar_wait(uint64_t *b, uint32_t parity, int64_t timeout_ns) {
  if (tc_mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = tc_global_ns();
  for (uint32_t i = 1;; ++i) {
    if (tc_mbar_try_wait(b, parity)) return true;
    if ((i & 63) == 0 && (int64_t)(tc_global_ns() - t0) > timeout_ns) return false;
  }
}

// The same wait for one of two cooperating threads: it gives up early once the
// other has set *abort, and sets *abort itself on timeout.
__device__ __forceinline__ bool tc_mbar_wait_or_abort(uint64_t *b, uint32_t parity, int64_t timeout_ns,
                                                      volatile int *abort) {
  if (tc_mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = tc_global_ns();
  for (uint32_t i = 1;; ++i) {
    if (tc_mbar_try_wait(b, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort) return false;
      if ((int64_t)(tc_global_ns() - t0) > timeout_ns) {
        *abort = 1;
        return false;
      }
    }
  }
}

// Shared-memory matrix descriptor of a K-major operand in 128-byte swizzle atoms
// (8 rows x 128 bytes, atoms 1024 bytes apart along M/N: the stride byte offset;
// the leading byte offset is not used by swizzled K-major layouts), descriptor
// version 1, layout type 2 (128-byte swizzle).  Units of 16 bytes.  Steps of
// K = 16 within an atom advance the start address by 32 bytes.
__device__ __forceinline__ uint64_t tc_smem_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void tc_mbar_arrive_expect_tx(uint64_t *b, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   tc_smem_u32(b)),
               "r"(bytes)
               : "memory");
}

// 2-D tile copy global -> shared by the tensor-memory accelerator, completing as
// transaction bytes on `bar`.  c0 is the inner (K) coordinate: a multiple of 64
// elements, so 128-byte aligned.
__device__ __forceinline__ void tc_tma_2d(void *dst, const CUtensorMap *map, int32_t c0, int32_t c1, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          tc_smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(tc_smem_u32(bar))
      : "memory");
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B both fp16 (0) or
// both bf16 (1), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__device__ __forceinline__ uint32_t tc_idesc(bool bf16, int n) {
  const uint32_t ab = bf16 ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier gets one arrival when every MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t *b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   tc_smem_u32(b))
               : "memory");
}

// The tensor-core path's storage types: fp16 (A/B format 0) and bf16 (format 1).
template <class Op> struct TcFormat { static constexpr bool ok = false, bf16 = false; };
template <> struct TcFormat<OpF16> {
  static constexpr bool ok = true, bf16 = false;
  // the output's rounding and the residual's widening, as Op::store and Op::x_elem do them
  __device__ static __forceinline__ unsigned short round(float v) { return __half_as_ushort(__float2half_rn(v)); }
  __device__ static __forceinline__ float widen(unsigned short h) { return __half2float(__ushort_as_half(h)); }
};
template <> struct TcFormat<OpBF16> {
  static constexpr bool ok = true, bf16 = true;
  __device__ static __forceinline__ unsigned short round(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
  __device__ static __forceinline__ float widen(unsigned short h) { return __uint_as_float((uint32_t)h << 16); }
};

// 16 accumulator columns of a warp's 32 tensor-memory lanes (this thread's lane):
// `addr` = tensor memory base + (first lane << 16) + first column.  Warp-aligned.
__device__ __forceinline__ void tc_tmem_ld16(uint32_t addr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(addr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// y[i0 .. i0 + 7] of a 16-bit output: v (scale, bias and activation applied) plus the
// residual's 8 values, each rounded once (as epilogue_store does it value by value),
// one 16-byte store.  y and the residual 16-byte aligned at i0.
template <class Op>
__device__ __forceinline__ void tc_store8(const Args &a, int64_t i0, float (&v)[8]) {
  if (a.residual != nullptr) {
    const uint4 rv = *reinterpret_cast<const uint4 *>(reinterpret_cast<const unsigned short *>(a.residual) + i0);
    const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] += TcFormat<Op>::widen((unsigned short)(rw[e / 2] >> (16 * (e & 1))));
  }
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    o[e] = (uint32_t)TcFormat<Op>::round(v[2 * e]) | ((uint32_t)TcFormat<Op>::round(v[2 * e + 1]) << 16);
  *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned short *>(a.y) + i0) = make_uint4(o[0], o[1], o[2], o[3]);
}

// A stage holds KA = 1 or 2 swizzle atoms along K (64 or 128 columns): 128 x 64 A
// boxes, then N x 64 x boxes.  The number of stages comes with the plan (its
// shared-memory size).
__host__ __device__ constexpr int tc_stage_bytes(int n, int ka) { return (kTcM + n) * kTcK * 2 * ka; }
// Wider stages for narrow N: each stage costs a fixed time to turn around, so it
// should carry at least ~24 KB.
__host__ __device__ constexpr int tc_atoms(int n) { return n <= 64 ? 2 : 1; }

// Distributed shared memory: four floats into the shared memory of the cluster's CTA
// `rank`, at the same offset as `p` has in this CTA.  A store: it does not wait for a
// reply.
__device__ __forceinline__ void tc_st_dsmem4(const float *p, uint32_t rank, float a, float b, float c, float d) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(tc_smem_u32(p)), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(ra), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void tc_st_dsmem_int(const int *p, uint32_t rank, int v) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(tc_smem_u32(p)), "r"(rank));
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(ra), "r"(v) : "memory");
}
// Every thread of every CTA of the cluster: writes before it are visible to the
// cluster's reads after it.  The barrier is warp-aligned: each warp first reconverges.
__device__ __forceinline__ void tc_cluster_sync() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// grid (ceil(M / 128), S); k-tiles [y * kt_per_split, ...) of K.  S > 1: launched as
// clusters of (1, S, 1), the slices of a tile reduced through distributed shared
// memory (above).  map_a: A as (K, M) 16-bit values, box 64 x 128; map_x: x as (K,
// B), box 64 x N; both 128-byte swizzle.
template <class Op, int KA>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_tc(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_x, const Args a,
         int64_t kt_per_split, int N, int stages) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full[kTcMaxStages], empty[kTcMaxStages];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;                                  // set by either role on timeout
  __shared__ int abort_of[kTcMaxSlices];                      // the cluster's abort flags, by rank
  __shared__ long long sh_loaded, sh_consumed, sh_committed;  // for the drain after an abort
  pdl_enter(a, false);  // every read (TMA included) after the kernel before has finished
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t M = a.M, K = a.K;
  const int B = a.B;
  const int64_t m0 = (int64_t)blockIdx.x * kTcM;
  constexpr int KT = kTcK * KA;  // K per stage
  const int64_t ktiles = (K + KT - 1) / KT;
  const int64_t kt_lo = (int64_t)blockIdx.y * kt_per_split;
  const int64_t kt_hi = kt_lo + kt_per_split < ktiles ? kt_lo + kt_per_split : ktiles;
  const int64_t nt = kt_hi - kt_lo;  // at least 1 when K > 0 (the planner makes no empty slice)
  const int S = stages;
  // the swizzle atoms need 1024-byte alignment of every stage
  unsigned char *smem = smem_raw + ((1024u - (tc_smem_u32(smem_raw) & 1023u)) & 1023u);
  constexpr uint32_t a_atom = kTcM * kTcK * 2;  // one 128 x 64 box of A
  const uint32_t x_atom = (uint32_t)N * kTcK * 2, a_bytes = a_atom * KA, st_bytes = (a_atom + x_atom) * KA;
  const uint32_t ncols = N <= 32 ? 32u : N <= 64 ? 64u : N <= 128 ? 128u : 256u;

  if (nt <= 0) {  // K == 0: the empty sum (one slice; every CTA of a cluster has K == 0)
    const int64_t m = m0 + tid;
    for (int b = 0; b < B && m < M && blockIdx.y == 0; ++b) epilogue_store<Op>(a, b, m, 0.f);
    return;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tc_smem_u32(&tmem_slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      tc_mbar_init(&full[s], 1);
      tc_mbar_init(&empty[s], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    abort_flag = 0;
    sh_loaded = sh_consumed = sh_committed = -1;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncwarp();  // lane 0 of warp 0 rejoins its warp: the CTA barrier counts whole warps
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_slot;

  // Two roles, one thread each: lane 0 of warp 0 copies k-tiles into free stages,
  // lane 0 of warp 1 issues the MMAs of landed stages; the other threads wait at the
  // barrier below for the accumulators.
  auto stage_a = [&](int s) { return smem + (size_t)s * st_bytes; };
  volatile int *abort = &abort_flag;
  if (warp == 0 && lane == 0) {
    int64_t loaded = -1;
    for (int64_t t = 0; t < nt; ++t) {
      const int s = (int)(t % S);
      // the stage is free once the MMAs of tile t - S have completed
      if (t >= S && !tc_mbar_wait_or_abort(&empty[s], (uint32_t)(((t - S) / S) & 1), a.timeout_ns, abort)) break;
      tc_mbar_arrive_expect_tx(&full[s], st_bytes);
      const int32_t k0 = (int32_t)((kt_lo + t) * KT);
#pragma unroll
      for (int j = 0; j < KA; ++j) {
        tc_tma_2d(stage_a(s) + j * a_atom, &map_a, k0 + j * kTcK, (int32_t)m0, &full[s]);
        tc_tma_2d(stage_a(s) + a_bytes + j * x_atom, &map_x, k0 + j * kTcK, 0, &full[s]);
      }
      loaded = t;
    }
    sh_loaded = loaded;
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = tc_idesc(TcFormat<Op>::bf16, N);
    int64_t consumed = -1, committed = -1;
    bool ok = true;
    for (int64_t i = 0; i < nt; ++i) {
      const int s = (int)(i % S);
      if (!tc_mbar_wait_or_abort(&full[s], (uint32_t)((i / S) & 1), a.timeout_ns, abort)) {
        ok = false;
        break;
      }
      consumed = i;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (!(a.test_stall && blockIdx.x == 0 && blockIdx.y == 0 && i == nt - 1)) {  // test: the last tile never completes
        const uint32_t sa = tc_smem_u32(stage_a(s)), sx = sa + a_bytes;
#pragma unroll
        for (int j = 0; j < KA; ++j)
#pragma unroll
          for (int kk = 0; kk < kTcK / 16; ++kk)
            tc_mma(tmem, tc_smem_desc(sa + j * a_atom + kk * 32), tc_smem_desc(sx + j * x_atom + kk * 32), idesc,
                   (i > 0 || j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&empty[s]);
        committed = i;
      }
    }
    // the last commit covers every MMA of the CTA
    if (ok) tc_mbar_wait_or_abort(&empty[(nt - 1) % S], (uint32_t)(((nt - 1) / S) & 1), a.timeout_ns, abort);
    sh_consumed = consumed;
    sh_committed = committed;
  }
  // the two role threads rejoin their warps first: the CTA barrier counts whole warps,
  // so without this the other lanes of warp 1 would let it complete (and the epilogue
  // read tensor memory) before the MMA thread has seen its last commit
  __syncwarp();
  __syncthreads();
  const bool aborted = abort_flag != 0;
  if (aborted) {
    // nothing may be in flight when the CTA frees its tensor memory and exits: the
    // last committed MMAs (their commit covers all earlier ones) and every copy
    // issued but not waited for
    if (tid == 0) {
      if (a.status != nullptr) atomicOr(a.status, kTcStatusMma);
      const int64_t committed = sh_committed, consumed = sh_consumed, loaded = sh_loaded;
      bool drained = committed < 0 ||
                     tc_mbar_wait(&empty[committed % S], (uint32_t)((committed / S) & 1), a.timeout_ns);
      for (int64_t t = consumed + 1; t <= loaded && drained; ++t)
        drained = tc_mbar_wait(&full[t % S], (uint32_t)((t / S) & 1), a.timeout_ns);
      if (!drained && a.status != nullptr) atomicOr(a.status, kTcStatusDrain);
    }
    __syncwarp();
    __syncthreads();
  }

  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const int row = warp * 32 + lane;  // this thread's tile row: TMEM lane 32 * warp + lane
  const int64_t m = m0 + row;
  // 16 accumulator columns c0 .. c0 + 15 of this thread's row
  auto tmem_ld16 = [&](int c0, uint32_t (&r)[16]) { tc_tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, r); };
  const int nslices = (int)gridDim.y;
  if (nslices == 1) {
    if (!aborted) {
      // The tile's outputs leave through shared memory (the stages are idle now): each
      // thread stages its row's values, scale, bias and activation applied, as fp32
      // [column][row]; then each thread takes 8 consecutive rows of one vector, adds the
      // residual and rounds once (as epilogue_store does) and writes them with one
      // 16-byte store instead of eight 2-byte ones.  CW columns per pass.
      float *stg = reinterpret_cast<float *>(smem);
      int cw = (stages * (int)st_bytes) / (kTcM * 4);
      cw = cw / 16 * 16;
      if (cw > N) cw = N;
      const bool vec = M % 8 == 0 && (reinterpret_cast<uintptr_t>(a.y) & 15) == 0 &&
                       (a.residual == nullptr || (reinterpret_cast<uintptr_t>(a.residual) & 15) == 0);
      for (int c0 = 0; c0 < N; c0 += cw) {
        const int w = N - c0 < cw ? N - c0 : cw;
        for (int cc = 0; cc < w; cc += 16) {
          uint32_t r[16];
          tmem_ld16(c0 + cc, r);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float v = 0.f;
            if (m < M) {
              v = row_value<Op>(a, m, __uint_as_float(r[j]));
              if (a.act == 1) v = silu(v);
            }
            stg[(cc + j) * kTcM + row] = v;
          }
        }
        __syncthreads();
        for (int k = tid; k < w * (kTcM / 8); k += kTcThreads) {
          const int col = k / (kTcM / 8), r0 = (k % (kTcM / 8)) * 8;
          const int b = c0 + col;
          const int64_t mm = m0 + r0;
          if (b >= B || mm >= M) continue;
          const float4 lo = *reinterpret_cast<const float4 *>(stg + col * kTcM + r0);
          const float4 hi = *reinterpret_cast<const float4 *>(stg + col * kTcM + r0 + 4);
          float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
          const int64_t i0 = (int64_t)b * M + mm;
          if (vec) {  // M % 8 == 0: all 8 rows exist
            tc_store8<Op>(a, i0, v);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              if (mm + e >= M) break;
              float ve = v[e];
              if (a.residual != nullptr) ve += Op::x_elem(a.residual, i0 + e);
              Op::store(a.y, i0 + e, ve);
            }
          }
        }
        __syncthreads();  // the staging buffer is read before the next columns overwrite it
      }
    }
  } else {
    // The cluster's slices of this tile.  The stages are idle now (every copy has
    // landed and every MMA has completed, or the CTA drained them above), so they hold
    // the owner buffers, CW columns at a time: part[slice][owned row][c], rows padded
    // to CW + 4 floats (16-byte rows whose bank offsets differ across a warp's rows).
    uint32_t rank;  // this CTA's rank in the cluster of the tile's slices
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const int S = nslices;
    const int maxrows = (kTcM + S - 1) / S;
    const int ring = stages * (int)st_bytes;
    int cw = ring / (4 * S * maxrows) - 4;
    cw = (cw / 16) * 16;
    if (cw > N) cw = N;
    const int rs = cw + 4;
    float *part = reinterpret_cast<float *>(smem);
    auto first_row = [&](int r) { return (kTcM * r + S - 1) / S; };
    const int owner = row * S / kTcM;  // the CTA that sums this thread's row
    const int orow = row - first_row(owner);
    const int rlo = first_row((int)rank), nrows = first_row((int)rank + 1) - rlo;
    // every CTA of the cluster has finished with its stages (and has started): only
    // now may peers store into them
    tc_cluster_sync();
    if (tid < S) tc_st_dsmem_int(&abort_of[rank], (uint32_t)tid, aborted ? 1 : 0);
    for (int c0 = 0; c0 < N; c0 += cw) {
      const int w = N - c0 < cw ? N - c0 : cw;
      if (!aborted) {
        const float *dst = part + ((int)rank * maxrows + orow) * rs;
        for (int cc = 0; cc < w; cc += 16) {
          uint32_t r[16];
          tmem_ld16(c0 + cc, r);
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            tc_st_dsmem4(dst + cc + j, (uint32_t)owner, __uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                         __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
        }
      }
      tc_cluster_sync();  // every slice's partial sums of the owned rows (and every abort flag) are here
      bool any_abort = false;
      for (int q = 0; q < S; ++q) any_abort |= abort_of[q] != 0;
      if (!any_abort) {
        // consecutive threads on consecutive rows (coalesced stores of y[b][m]), four
        // columns each; slices added in index order
        for (int idx = tid; idx < nrows * (w / 4); idx += kTcThreads) {
          const int rl = idx % nrows, c = (idx / nrows) * 4;
          float4 v = *reinterpret_cast<const float4 *>(part + rl * rs + c);
          for (int q = 1; q < S; ++q) {
            const float4 u = *reinterpret_cast<const float4 *>(part + (q * maxrows + rl) * rs + c);
            v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w;
          }
          const int64_t mm = m0 + rlo + rl;
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (c0 + c + j < B && mm < M) epilogue_store<Op>(a, c0 + c + j, mm, vv[j]);
        }
      }
      // the owners are done reading before the next columns arrive (after the last
      // columns no CTA touches a peer's shared memory again: no barrier)
      if (c0 + cw < N) tc_cluster_sync();
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncwarp();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
}


// ------------------------------------------------------------------ k_tc_persist
// The same product for more tiles than one wave holds, without a K split: one CTA per
// SM walks tiles blockIdx.x, blockIdx.x + gridDim.x, ... with its stage ring running
// on across tiles.  Warp 0 (lane 0) copies k-tiles, warp 1 (lane 0) issues the MMAs,
// warps 2..5 run the epilogue.  Two accumulators of ncols columns alternate in tensor
// memory: while the epilogue warps read tile j's (and store y), the MMAs of tile j + 1
// fill the other, so a tile's epilogue hides behind the next tile's copies.  "accf"
// (one arrival: the tile's last MMA commit) hands an accumulator to the epilogue;
// "acce" (one arrival per epilogue warp) hands it back.  Epilogue warp w reads tensor
// memory lanes 32 (w mod 4) .. + 31, the lanes a warp of that rank may access.
constexpr int kTcPThreads = 192;
// after the stage ring: each epilogue warp's staging buffer, 16 columns x 32 rows fp32
constexpr int kTcPEpBytes = 4 * 16 * 32 * 4;

__device__ __forceinline__ void tc_mbar_arrive(uint64_t *b) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(tc_smem_u32(b)) : "memory");
}

template <class Op, int KA>
__global__ void __launch_bounds__(kTcPThreads, 1)
    k_tc_persist(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_x, const Args a,
                 int N, int stages) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t full[kTcMaxStages], empty[kTcMaxStages], accf[2], acce[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;  // set by any role on timeout
  __shared__ long long sh_loaded, sh_consumed, sh_committed, sh_acc_committed;  // for the drain after an abort
  pdl_enter(a, false);  // every read (TMA included) after the kernel before has finished
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t M = a.M, K = a.K;
  const int B = a.B;
  constexpr int KT = kTcK * KA;  // K per stage
  const int64_t nkt = (K + KT - 1) / KT;            // k-tiles per row tile (K > 0: the planner's rule)
  const int64_t ntiles = (M + kTcM - 1) / kTcM;
  const int64_t my_tiles = (int64_t)blockIdx.x < ntiles ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int64_t total = my_tiles * nkt;             // k-tiles this CTA streams
  const int S = stages;
  unsigned char *smem = smem_raw + ((1024u - (tc_smem_u32(smem_raw) & 1023u)) & 1023u);
  constexpr uint32_t a_atom = kTcM * kTcK * 2;
  const uint32_t x_atom = (uint32_t)N * kTcK * 2, a_bytes = a_atom * KA, st_bytes = (a_atom + x_atom) * KA;
  const uint32_t ncols = N <= 32 ? 32u : N <= 64 ? 64u : N <= 128 ? 128u : 256u;  // per accumulator

  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tc_smem_u32(&tmem_slot)),
                 "r"(2 * ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      tc_mbar_init(&full[s], 1);
      tc_mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc_mbar_init(&accf[b], 1);
      tc_mbar_init(&acce[b], 4);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    abort_flag = 0;
    sh_loaded = sh_consumed = sh_committed = sh_acc_committed = -1;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncwarp();
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_slot;
  auto stage_a = [&](int s) { return smem + (size_t)s * st_bytes; };
  volatile int *abort = &abort_flag;

  if (warp == 0) {
    if (lane == 0) {  // producer
      int64_t loaded = -1;
      for (int64_t g = 0; g < total; ++g) {
        const int s = (int)(g % S);
        if (g >= S && !tc_mbar_wait_or_abort(&empty[s], (uint32_t)(((g - S) / S) & 1), a.timeout_ns, abort)) break;
        const int64_t j = g / nkt, kt = g - j * nkt;
        const int32_t m0 = (int32_t)(((int64_t)blockIdx.x + j * gridDim.x) * kTcM);
        tc_mbar_arrive_expect_tx(&full[s], st_bytes);
        const int32_t k0 = (int32_t)(kt * KT);
#pragma unroll
        for (int jj = 0; jj < KA; ++jj) {
          tc_tma_2d(stage_a(s) + jj * a_atom, &map_a, k0 + jj * kTcK, m0, &full[s]);
          tc_tma_2d(stage_a(s) + a_bytes + jj * x_atom, &map_x, k0 + jj * kTcK, 0, &full[s]);
        }
        loaded = g;
      }
      sh_loaded = loaded;
    }
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      const uint32_t idesc = tc_idesc(TcFormat<Op>::bf16, N);
      int64_t consumed = -1, committed = -1, acc_committed = -1;
      bool ok = true;
      for (int64_t j = 0; j < my_tiles && ok; ++j) {
        const int buf = (int)(j & 1);
        // the epilogue has read this accumulator's previous tile (j - 2)
        if (j >= 2 && !tc_mbar_wait_or_abort(&acce[buf], (uint32_t)(((j - 2) / 2) & 1), a.timeout_ns, abort)) {
          ok = false;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        bool stalled = false;
        for (int64_t kt = 0; kt < nkt; ++kt) {
          const int64_t g = j * nkt + kt;
          const int s = (int)(g % S);
          if (!tc_mbar_wait_or_abort(&full[s], (uint32_t)((g / S) & 1), a.timeout_ns, abort)) {
            ok = false;
            break;
          }
          consumed = g;
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          if (a.test_stall && blockIdx.x == 0 && g == total - 1) {  // test: the last tile never completes
            stalled = true;
            continue;
          }
          const uint32_t sa = tc_smem_u32(stage_a(s)), sx = sa + a_bytes;
#pragma unroll
          for (int jj = 0; jj < KA; ++jj)
#pragma unroll
            for (int kk = 0; kk < kTcK / 16; ++kk)
              tc_mma(tmem + (uint32_t)buf * ncols, tc_smem_desc(sa + jj * a_atom + kk * 32),
                     tc_smem_desc(sx + jj * x_atom + kk * 32), idesc, (kt > 0 || jj > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty[s]);
          committed = g;
        }
        if (!ok || stalled) break;
        tc_commit(&accf[buf]);  // arrives once every MMA of the tile has completed
        acc_committed = j;
      }
      sh_consumed = consumed;
      sh_committed = committed;
      sh_acc_committed = acc_committed;
    }
  } else {
    // epilogue warps 2..5: tensor memory lanes 32 (warp mod 4) .. + 31
    const int ew = warp & 3;
    float *ep = reinterpret_cast<float *>(smem + (size_t)S * st_bytes) + ew * 16 * 32;
    // 16-byte stores of 8 rows: M a multiple of 8, y and the residual 16-byte aligned
    const bool vec = M % 8 == 0 && (reinterpret_cast<uintptr_t>(a.y) & 15) == 0 &&
                     (a.residual == nullptr || (reinterpret_cast<uintptr_t>(a.residual) & 15) == 0);
    for (int64_t j = 0; j < my_tiles; ++j) {
      const int buf = (int)(j & 1);
      // lane 0 waits for the tile's accumulator and the warp follows it (a warp-uniform
      // decision before the warp-aligned tensor-memory loads)
      int ok = 0;
      if (lane == 0) ok = tc_mbar_wait_or_abort(&accf[buf], (uint32_t)((j / 2) & 1), a.timeout_ns, abort) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int64_t m0w = ((int64_t)blockIdx.x + j * gridDim.x) * kTcM + ew * 32;  // the warp's first row
      const int64_t m = m0w + lane;
      for (int c0 = 0; c0 < N; c0 += 16) {
        uint32_t r[16];
        tc_tmem_ld16(tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)buf * ncols + (uint32_t)c0, r);
        if (vec) {
          // the 16 columns of the warp's 32 rows staged as fp32 [column][row] (scale, bias
          // and activation applied), then per lane 8 rows of one column: residual added,
          // rounded once, one 16-byte store (as epilogue_store does it, value by value)
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            float v = 0.f;
            if (m < M) {
              v = row_value<Op>(a, m, __uint_as_float(r[jj]));
              if (a.act == 1) v = silu(v);
            }
            ep[jj * 32 + lane] = v;
          }
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int cc = (lane >> 2) + 8 * h, r0 = (lane & 3) * 8;
            const int b = c0 + cc;
            const int64_t mm = m0w + r0;
            if (b < B && mm < M) {  // M % 8 == 0: all 8 rows exist
              const float4 lo = *reinterpret_cast<const float4 *>(ep + cc * 32 + r0);
              const float4 hi = *reinterpret_cast<const float4 *>(ep + cc * 32 + r0 + 4);
              float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
              tc_store8<Op>(a, (int64_t)b * M + mm, v);
            }
          }
          __syncwarp();  // read before the next columns overwrite the buffer
        } else if (m < M) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            if (c0 + jj < B) epilogue_store<Op>(a, c0 + jj, m, __uint_as_float(r[jj]));
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) tc_mbar_arrive(&acce[buf]);  // this warp is done with the accumulator
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncwarp();  // the role threads rejoin their warps: the CTA barrier counts whole warps
  __syncthreads();
  if (abort_flag != 0) {
    // nothing may be in flight when the CTA frees its tensor memory and exits: the last
    // committed MMAs (their commit covers all earlier ones), every copy issued but not
    // waited for, and the last accumulator hand-over
    if (tid == 0) {
      if (a.status != nullptr) atomicOr(a.status, kTcStatusMma);
      const int64_t committed = sh_committed, consumed = sh_consumed, loaded = sh_loaded, accc = sh_acc_committed;
      bool drained = committed < 0 ||
                     tc_mbar_wait(&empty[committed % S], (uint32_t)((committed / S) & 1), a.timeout_ns);
      for (int64_t t = consumed + 1; t <= loaded && drained; ++t)
        drained = tc_mbar_wait(&full[t % S], (uint32_t)((t / S) & 1), a.timeout_ns);
      if (drained && accc >= 0) drained = tc_mbar_wait(&accf[accc & 1], (uint32_t)((accc / 2) & 1), a.timeout_ns);
      if (!drained && a.status != nullptr) atomicOr(a.status, kTcStatusDrain);
    }
    __syncwarp();
    __syncthreads();
  }
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * ncols) : "memory");
  }
}

}  // namespace gemv
