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
// order for L2 reuse.  TMA zero-fills beyond M, N, K.  CTAs run in clusters of
// two along M that share each 64 x 256 slice of B: each CTA loads one half and
// multicasts it to both (see tc_bf16_kernel).
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace g12 {
namespace {

constexpr int BM = kTcBM, BN = kTcBN, BK = kTcBK;
#ifndef G12_TC_STAGES
#define G12_TC_STAGES 4
#endif
#ifndef G12_TC_GROUP_M
#define G12_TC_GROUP_M 8
#endif
constexpr int STAGES = G12_TC_STAGES;
constexpr int kStageBytesA = BM * BK * 2;            // 16 KB
constexpr int kStageBytesB = BK * BN * 2;            // 32 KB
constexpr int kBoxBytesB = BK * 64 * 2;              // one 64-column box, 8 KB
constexpr int kStageBytes = kStageBytesA + kStageBytesB;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr int kGroupM = G12_TC_GROUP_M;  // raster group height (tile rows or row pairs)
constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN, /*A MN-major*/ 0, /*B MN-major*/ 1);
#ifndef G12_TC_CLUSTER_M
#define G12_TC_CLUSTER_M 2
#endif
constexpr int kClusterM = G12_TC_CLUSTER_M;  // CTAs per cluster along M (1 or 2)
static_assert(kClusterM == 1 || kClusterM == 2, "cluster of 1 or 2 CTAs");

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

// One 32-column chunk of an accumulator row: D = act(alpha*acc + beta*C + bias).
// Old C values are all loaded before the first store, so the loads overlap
// (interleaved load/store pairs to possibly aliasing addresses would cost a
// memory round trip each).
__device__ __forceinline__ void store_row_chunk(const TcArgs& p, int row, int col0,
                                                const uint32_t (&r)[32]) {
  const Epilogue& e = p.epi;
  const bool read_c = (e.beta != 0.0f);
  const float* c_row = e.C + static_cast<int64_t>(row) * e.ldc;
  if (col0 + 31 < p.N) {
    float old[32];
    if (read_c) {
      if (e.c_vec4) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 o = *reinterpret_cast<const float4*>(c_row + col0 + 4 * q);
          old[4 * q + 0] = o.x;
          old[4 * q + 1] = o.y;
          old[4 * q + 2] = o.z;
          old[4 * q + 3] = o.w;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) old[c] = c_row[col0 + c];
      }
    }
    float bias[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) bias[c] = epi_bias(e, col0 + c);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      float v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        v[c] = epi_value(e, __uint_as_float(r[8 * h + c]), read_c ? old[8 * h + c] : 0.0f,
                         bias[8 * h + c]);
      if (e.d_vec) {
        epi_store8(e, row, col0 + 8 * h, v);
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) epi_store1(e, row, col0 + 8 * h + c, v[c]);
      }
    }
  } else {
    // ragged right edge
    float old[32], bias[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      old[c] = (read_c && col0 + c < p.N) ? c_row[col0 + c] : 0.0f;
      bias[c] = (col0 + c < p.N) ? epi_bias(e, col0 + c) : 0.0f;
    }
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const int col = col0 + c;
      if (col < p.N) epi_store1(e, row, col, epi_value(e, __uint_as_float(r[c]), old[c], bias[c]));
    }
  }
}

// CL = CTAs per cluster along M (1 or 2).  With CL = 2 the two CTAs of a
// cluster compute vertically adjacent tiles (2 pm and 2 pm + 1) of the same
// 256 columns: each loads its own 128 x 64 slice of A and one half of the
// shared 64 x 256 slice of B, multicast into both CTAs, so every CTA moves
// 32 KB instead of 48 KB per k-block from L2.  A stage may be refilled only
// after the MMAs of both CTAs have read it: each MMA thread commits to the
// stage's empty barrier in both CTAs (count CL).
template <int CL>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bf16_kernel(const __grid_constant__ TcArgs p, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem<1024>(smem_raw);
  TcSmemTail* tail = reinterpret_cast<TcSmemTail*>(smem + STAGES * kStageBytes);
  volatile int* abort_flag = &tail->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int groups_m = (tiles_m + CL - 1) / CL;   // tile rows handled per cluster item
  const int num_items = groups_m * tiles_n;
  const int num_kb = (p.K + BK - 1) / BK;
  const uint32_t rank = (CL > 1) ? cluster_cta_rank() : 0u;
  const int first_item = static_cast<int>(blockIdx.x) / CL;
  const int item_stride = static_cast<int>(gridDim.x) / CL;
  constexpr uint16_t kPeers = static_cast<uint16_t>((1u << CL) - 1u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&tail->full[s], 1);
      mbar_init(&tail->empty[s], CL);
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
  // Peers multicast into this CTA's shared memory and barriers: all barriers
  // of the cluster must be initialised first.
  if (CL > 1) cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = tail->tmem_base;

  if (warp == 0) {
    // -------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = first_item; t < num_items && ok; t += item_stride) {
        int pm, tn;
        tile_coords(t, groups_m, tiles_n, pm, tn);
        const int tm = pm * CL + static_cast<int>(rank);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t round = it / STAGES;
          if (!mbar_wait(&tail->empty[s], (round & 1u) ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * kStageBytes;
          uint8_t* sb = sa + kStageBytesA;
          // all 48 KB arrive here: A from this CTA, B half from each CTA
          mbar_arrive_expect_tx(&tail->full[s], kStageBytes);
          tma_load_2d(sa, &tmA, kb * BK, tm * BM, &tail->full[s]);
          if (CL == 1) {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(sb + j * kBoxBytesB, &tmB, tn * BN + j * 64, kb * BK, &tail->full[s]);
          } else {
#pragma unroll
            for (int jj = 0; jj < BN / 64 / CL; ++jj) {
              const int j = static_cast<int>(rank) * (BN / 64 / CL) + jj;
              tma_load_2d_multicast(sb + j * kBoxBytesB, &tmB, tn * BN + j * 64, kb * BK,
                                    &tail->full[s], kPeers);
            }
          }
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
      for (int t = first_item; t < num_items && ok; t += item_stride, ++j) {
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
          if (CL == 1)
            tc_commit(&tail->empty[s]);
          else
            tc_commit_multicast(&tail->empty[s], kPeers);  // frees the stage in both CTAs
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
    for (int t = first_item; t < num_items; t += item_stride, ++j) {
      int pm, tn;
      tile_coords(t, groups_m, tiles_n, pm, tn);
      const int tm = pm * CL + static_cast<int>(rank);
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
  // No CTA may exit while its peer can still multicast into it.
  if (CL > 1) cluster_sync();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace

cudaError_t launch_tc_bf16(const TcArgs& a, const CUtensorMap* tmA, const CUtensorMap* tmB,
                           int num_sms, cudaStream_t stream) {
  const int tiles_m = (a.M + BM - 1) / BM;
  const int tiles_n = (a.N + BN - 1) / BN;
  if (kClusterM > 1 && tiles_m >= kClusterM) {
    auto kernel = tc_bf16_kernel<kClusterM>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClusterM;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Persistent clusters: as many as can be resident at once, at most one
    // per pair of tiles.
    const int items = ((tiles_m + kClusterM - 1) / kClusterM) * tiles_n;
    int max_clusters = 0;
    cfg.gridDim = dim3(kClusterM * (num_sms / kClusterM));
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kernel, &cfg) != cudaSuccess ||
        max_clusters < 1) {
      cudaGetLastError();
      max_clusters = num_sms / kClusterM;
    }
    const int clusters = items < max_clusters ? items : max_clusters;
    cfg.gridDim = dim3(kClusterM * clusters);
    e = cudaLaunchKernelEx(&cfg, kernel, a, *tmA, *tmB);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  auto kernel = tc_bf16_kernel<1>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int tiles = tiles_m * tiles_n;
  const int grid = tiles < num_sms ? tiles : num_sms;
  kernel<<<grid, kThreads, kSmemBytes, stream>>>(a, *tmA, *tmB);
  return cudaGetLastError();
}

}  // namespace g12
