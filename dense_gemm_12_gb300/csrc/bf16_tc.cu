// bf16_tc.cu -- bf16-input, fp32-accumulate, fp32-output GEMM on the
// 5th-generation tensor cores:  C = alpha * A * B + beta * C.
//
// The pages stop at the tensor-core rung: "Tiled matrix multiplication"
// ("How it works") names mma.sync and Hopper's wgmma reading operands from
// shared memory, fed by TMA into multi-buffered shared memory; "A GEMM
// Kernel, Step by Step" ("Those four are the end of this ladder") describes
// the kernel in which one instruction hands a whole tile to the tensor core, a
// copy engine fetches the next tile on one thread's say-so, and the remaining
// warps run the pipeline.  This file is that kernel for sm_103a:
//   * warp 0      -- TMA producer: 128 x 64 slices of A (K-major, 128-B
//                    swizzle) and 64 x 256 slices of B (row-major B is
//                    N-contiguous, i.e. MN-major, 4 swizzled 64-column boxes)
//                    into a 4-stage shared-memory ring (full/empty mbarriers);
//   * warp 1      -- allocates 512 TMEM columns (two 128 x 256 fp32
//                    accumulators) and one lane issues tcgen05.mma
//                    (M=128, N=256, K=16, four per stage), committing each
//                    stage back to the producer and each finished tile to the
//                    epilogue;
//   * warps 2..5  -- epilogue: tcgen05.ld of the accumulator, alpha/beta,
//                    masked stores; the second accumulator lets the MMAs of
//                    the next tile run while this one drains.
// Persistent CTAs (one per SM) walk the 128 x 256 tiles in a grouped raster
// order for L2 reuse.  TMA zero-fills beyond M, N, K.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace g12 {
namespace {

constexpr int BM = kTcBM, BN = kTcBN, BK = kTcBK;
constexpr int STAGES = 4;
constexpr int kStageBytesA = BM * BK * 2;            // 16 KB
constexpr int kStageBytesB = BK * BN * 2;            // 32 KB
constexpr int kBoxBytesB = BK * 64 * 2;              // one 64-column box, 8 KB
constexpr int kStageBytes = kStageBytesA + kStageBytesB;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr int kGroupM = 16;
constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN, /*A MN-major*/ 0, /*B MN-major*/ 1);

struct __align__(8) TcSmemTail {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

constexpr size_t kSmemBytes = 1024 + STAGES * kStageBytes + sizeof(TcSmemTail);

__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int& tm, int& tn) {
  const int per_group = kGroupM * tiles_n;
  const int g = t / per_group;
  const int first_m = g * kGroupM;
  const int rows = min(tiles_m - first_m, kGroupM);
  const int local = t - g * per_group;
  tm = first_m + local % rows;
  tn = local / rows;
}

__device__ __forceinline__ void store_row_chunk(const TcArgs& p, int row, int col0,
                                                const uint32_t (&r)[32]) {
  float* c_row = p.C + static_cast<int64_t>(row) * p.ldc;
  const bool read_c = (p.beta != 0.0f);
  if (p.c_vec4 && col0 + 31 < p.N) {
    // Old values first, then the stores (see the note in the else branch).
    float4 old[8];
    if (read_c) {
#pragma unroll
      for (int q = 0; q < 8; ++q) old[q] = *reinterpret_cast<const float4*>(c_row + col0 + 4 * q);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float4* dst = reinterpret_cast<float4*>(c_row + col0 + 4 * q);
      float4 v = make_float4(__uint_as_float(r[4 * q + 0]), __uint_as_float(r[4 * q + 1]),
                             __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
      if (read_c) {
        const float4 o = old[q];
        v.x = fmaf(p.alpha, v.x, p.beta * o.x);
        v.y = fmaf(p.alpha, v.y, p.beta * o.y);
        v.z = fmaf(p.alpha, v.z, p.beta * o.z);
        v.w = fmaf(p.alpha, v.w, p.beta * o.w);
      } else {
        v.x *= p.alpha;
        v.y *= p.alpha;
        v.z *= p.alpha;
        v.w *= p.alpha;
      }
      *dst = v;
    }
  } else {
    // Ragged or unaligned edge.  Loading every old value before the first
    // store keeps the loads independent; interleaved load/store pairs to
    // possibly aliasing addresses would cost one memory round trip each.
    float old[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) old[c] = (read_c && col0 + c < p.N) ? c_row[col0 + c] : 0.0f;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const int col = col0 + c;
      if (col < p.N) {
        const float v = __uint_as_float(r[c]);
        c_row[col] = read_c ? fmaf(p.alpha, v, p.beta * old[c]) : p.alpha * v;
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    tc_bf16_kernel(const TcArgs p, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem<1024>(smem_raw);
  TcSmemTail* tail = reinterpret_cast<TcSmemTail*>(smem + STAGES * kStageBytes);
  volatile int* abort_flag = &tail->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int num_tiles = tiles_m * tiles_n;
  const int num_kb = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&tail->full[s], 1);
      mbar_init(&tail->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tail->tmem_full[b], 1);
      mbar_init(&tail->tmem_empty[b], kEpiThreads);
    }
    mbar_init(&tail->drain, 1);
    tail->abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&tail->tmem_base, kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tail->tmem_base;

  if (warp == 0) {
    // -------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int tm, tn;
        tile_coords(t, tiles_m, tiles_n, tm, tn);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t round = it / STAGES;
          if (!mbar_wait(&tail->empty[s], (round & 1u) ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * kStageBytes;
          uint8_t* sb = sa + kStageBytesA;
          mbar_arrive_expect_tx(&tail->full[s], kStageBytes);
          tma_load_2d(sa, &tmA, kb * BK, tm * BM, &tail->full[s]);
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_2d(sb + j * kBoxBytesB, &tmB, tn * BN + j * 64, kb * BK, &tail->full[s]);
        }
      }
      if (!ok) {
        const uint32_t first = it > STAGES ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j)
          mbar_drain_wait(&tail->full[j % STAGES], (j / STAGES) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0;
      uint32_t j = 0;
      bool ok = true;
      bool issued = false;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++j) {
        const uint32_t ab = j & 1u, ar = j >> 1;
        if (!mbar_wait(&tail->tmem_empty[ab], (ar & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + ab * BN;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t round = it / STAGES;
          if (!mbar_wait(&tail->full[s], round & 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = smem_u32(smem + s * kStageBytes);
          const uint32_t sb = sa + kStageBytesA;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // A: K-major, 8-row groups 1024 B apart; a K step of 16 is 32 B.
            const uint64_t adesc = smem_desc_sw128(sa + kk * 32, 16, 1024);
            // B: MN-major, 64-column boxes 8 KB apart (LBO), 8-row k groups
            // 1024 B apart (SBO); a K step of 16 rows is 2048 B.
            const uint64_t bdesc = smem_desc_sw128(sb + kk * 2048, kBoxBytesB, 1024);
            tc_mma_f16(d_tmem, adesc, bdesc, kIdesc, (kb | kk) != 0 ? 1u : 0u);
          }
          issued = true;
          tc_commit(&tail->empty[s]);
        }
        if (!ok) break;
        tc_commit(&tail->tmem_full[ab]);
      }
      if (!ok && issued) {
        // Let every MMA this thread issued finish before TMEM is released.
        tc_commit(&tail->drain);
        mbar_drain_wait(&tail->drain, 0);
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    uint32_t j = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++j) {
      int tm, tn;
      tile_coords(t, tiles_m, tiles_n, tm, tn);
      const uint32_t ab = j & 1u, ar = j >> 1;
      if (!mbar_wait(&tail->tmem_full[ab], ar & 1u, abort_flag, p.err)) break;
      tc_fence_after_sync();
      const int row = tm * BM + quarter * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + ab * BN;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c * 32, r);
        tc_wait_ld();
        if (row < p.M) store_row_chunk(p, row, tn * BN + c * 32, r);
      }
      tc_fence_before_sync();
      mbar_arrive(&tail->tmem_empty[ab]);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace

cudaError_t launch_tc_bf16(const TcArgs& a, const CUtensorMap* tmA, const CUtensorMap* tmB,
                           int num_sms, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(tc_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  tc_bf16_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a, *tmA, *tmB);
  return cudaGetLastError();
}

}  // namespace g12
