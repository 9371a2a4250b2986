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
//
// That single-CTA kernel serves M <= 128.  Larger problems run on CTA pairs
// (tc_bf16_pair_kernel below): two SMs share one 256 x 256 tile and one MMA
// stream, which cuts the shared-memory operand bytes each SM's tensor core
// reads per MMA from 12 KB to 8 KB.
//
// Both kernels walk work units instead of tiles: the tiles that would leave
// the last round of the persistent grid partly idle ("A GEMM Kernel, Step by
// Step", "The fringe and the last wave") are cut along k, the split-K of its
// "What is left": each part's partial sums go to a workspace, and the last
// part to finish a tile adds them in part order before the output stage.
#include <cuda_runtime.h>

#include <atomic>
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
// Cost of storing or loading one split part's partial sums, in k-block times
// (see tail_split): a 128 KB partial per CTA moves in about 1.1 us at the
// ~120 GB/s one SM gets from L2, some 3 k-blocks of the tensor core.
#ifndef G12_TC_PART_COST
#define G12_TC_PART_COST 3.0
#endif
constexpr int STAGES = G12_TC_STAGES;
constexpr int kStageBytesA = BM * BK * 2;            // 16 KB
constexpr int kStageBytesB = BK * BN * 2;            // 32 KB
constexpr int kBoxBytesB = BK * 64 * 2;              // one 64-column box, 8 KB
constexpr int kStageBytes = kStageBytesA + kStageBytesB;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr uint32_t kTmemCols = 512;
constexpr int kGroupM = G12_TC_GROUP_M;  // raster group height (tile rows or row pairs)
constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN, /*A MN-major*/ 0, /*B MN-major*/ 1);
// Named barriers of the epilogue warps (0 is __syncthreads).
constexpr uint32_t kEpiBarSync = 1, kEpiBarAny = 2;
// Partial sums of one split part of one CTA's 128 x 256 tile.
constexpr int64_t kPartFloats = static_cast<int64_t>(BM) * BN;

struct __align__(8) TcSmemTail {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int last_flag;
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

// One work unit: item (tile or pair tile), its k-block range and, for a
// split item, its part index and tail index (part = -1 for a whole item).
struct Unit {
  int item, kb0, kb1, part, tail;
};

__device__ __forceinline__ int num_units(const TcArgs& p, int num_items) {
  return p.full_items + (num_items - p.full_items) * p.split;
}

__device__ __forceinline__ Unit unit_of(const TcArgs& p, int u, int num_kb) {
  Unit w;
  if (u < p.full_items) {
    w.item = u;
    w.kb0 = 0;
    w.kb1 = num_kb;
    w.part = -1;
    w.tail = -1;
    return w;
  }
  const int v = u - p.full_items;
  w.tail = v / p.split;
  w.part = v - w.tail * p.split;
  w.item = p.full_items + w.tail;
  w.kb0 = w.part * num_kb / p.split;
  w.kb1 = (w.part + 1) * num_kb / p.split;
  return w;
}

// One 32-column chunk of an accumulator row through the output stage (see
// epilogue.cuh).  Old C, bias and residual values are all loaded before the
// first store, so the loads overlap (interleaved load/store pairs to possibly
// aliasing addresses would cost a memory round trip each).  amax_acc: this
// thread's running max |v|.
__device__ __forceinline__ void store_row_chunk(const TcArgs& p, int row, int col0,
                                                const uint32_t (&r)[32], float& amax_acc) {
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
    float bias[32], res[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      bias[c] = epi_bias(e, col0 + c);
      res[c] = epi_residual(e, row, col0 + c);
    }
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      float v[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        v[c] = epi_value(e, __uint_as_float(r[8 * h + c]), read_c ? old[8 * h + c] : 0.0f,
                         bias[8 * h + c], res[8 * h + c]);
        epi_track(e, amax_acc, v[c]);
      }
      if (e.d_vec) {
        epi_store8(e, row, col0 + 8 * h, v);
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) epi_store1(e, row, col0 + 8 * h + c, v[c]);
      }
    }
  } else {
    // ragged right edge
    float old[32], bias[32], res[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const bool in = col0 + c < p.N;
      old[c] = (read_c && in) ? c_row[col0 + c] : 0.0f;
      bias[c] = in ? epi_bias(e, col0 + c) : 0.0f;
      res[c] = in ? epi_residual(e, row, col0 + c) : 0.0f;
    }
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const int col = col0 + c;
      if (col < p.N) {
        const float v = epi_value(e, __uint_as_float(r[c]), old[c], bias[c], res[c]);
        epi_track(e, amax_acc, v);
        epi_store1(e, row, col, v);
      }
    }
  }
}

__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync %0, %1;" ::"n"(kEpiBarSync), "n"(kEpiThreads) : "memory");
}

// Output stage of one work unit, run by the 4 epilogue warps of a CTA (thread
// et = TMEM lane et = row et of the CTA's 128-row tile).  taddr: this warp's
// lanes of the accumulator.  slot: this CTA's index among the split items'
// counters (-1 for a whole item).
//
// A split part stores its partial sums (thread-major float4s, coalesced per
// warp), then counts its arrival; the last of the `split` parts re-reads its
// own accumulator and adds all parts in part order -- a fixed order, so the
// result does not depend on which part finishes last -- and writes D.
__device__ __forceinline__ void epilogue_unit(const TcArgs& p, uint32_t taddr, int row, int tn,
                                              int slot, int part, int et, int* last_flag,
                                              float& amax_acc) {
  if (slot < 0) {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(taddr + c * 32, r);
      tc_wait_ld();
      if (row < p.M) store_row_chunk(p, row, tn * BN + c * 32, r, amax_acc);
    }
    return;
  }
  float4* const ws4 = reinterpret_cast<float4*>(p.ws);
  const int64_t slot_base = static_cast<int64_t>(slot) * p.split;  // in parts
  {
    float4* mine = ws4 + (slot_base + part) * (kPartFloats / 4);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(taddr + c * 32, r);
      tc_wait_ld();
#pragma unroll
      for (int q = 0; q < 8; ++q)
        __stcg(mine + (c * 8 + q) * kEpiThreads + et,
               make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                           __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])));
    }
  }
  epi_bar();
  if (et == 0) {
    __threadfence();  // publish the whole CTA's partial before arriving
    const uint32_t before = atomicAdd(p.counters + slot, 1u);
    *last_flag = (before == static_cast<uint32_t>(p.split - 1)) ? 1 : 0;
  }
  epi_bar();
  if (*reinterpret_cast<volatile int*>(last_flag)) {
    __threadfence();
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(taddr + c * 32, r);
      tc_wait_ld();
      float sum[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) sum[i] = 0.0f;
      for (int q_part = 0; q_part < p.split; ++q_part) {
        if (q_part == part) {
#pragma unroll
          for (int i = 0; i < 32; ++i) sum[i] += __uint_as_float(r[i]);
        } else {
          const float4* src = ws4 + (slot_base + q_part) * (kPartFloats / 4);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 v = __ldcg(src + (c * 8 + q) * kEpiThreads + et);
            sum[4 * q] += v.x;
            sum[4 * q + 1] += v.y;
            sum[4 * q + 2] += v.z;
            sum[4 * q + 3] += v.w;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(sum[i]);
      if (row < p.M) store_row_chunk(p, row, tn * BN + c * 32, r, amax_acc);
    }
    if (et == 0) p.counters[slot] = 0u;
  }
  epi_bar();  // last_flag is rewritten by the next split unit
}

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
  const int num_kb = (p.K + BK - 1) / BK;
  const int units = num_units(p, tiles_m * tiles_n);

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
    tail->last_flag = 0;
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
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit w = unit_of(p, u, num_kb);
        int tm, tn;
        tile_coords(w.item, tiles_m, tiles_n, tm, tn);
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
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
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++j) {
        const Unit w = unit_of(p, u, num_kb);
        const uint32_t ab = j & 1u, ar = j >> 1;
        if (!mbar_wait(&tail->tmem_empty[ab], (ar & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + ab * BN;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
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
            tc_mma_f16(d_tmem, adesc, bdesc, kIdesc, (kb != w.kb0 || kk != 0) ? 1u : 0u);
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
    const int et = quarter * 32 + lane;
    float amax_acc = 0.0f;
    uint32_t j = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++j) {
      const Unit w = unit_of(p, u, num_kb);
      int tm, tn;
      tile_coords(w.item, tiles_m, tiles_n, tm, tn);
      const uint32_t ab = j & 1u, ar = j >> 1;
      const bool ok = mbar_wait(&tail->tmem_full[ab], ar & 1u, abort_flag, p.err);
      // Leave together if a wait ran out anywhere (see named_bar_any).
      if (named_bar_any(kEpiBarAny, kEpiThreads, !ok)) break;
      tc_fence_after_sync();
      const int row = tm * BM + et;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + ab * BN;
      epilogue_unit(p, taddr, row, tn, w.tail, w.part, et, &tail->last_flag, amax_acc);
      tc_fence_before_sync();
      mbar_arrive(&tail->tmem_empty[ab]);
    }
    epi_flush_amax(p.epi, amax_acc);
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ------------------------------------------------------------------------
// CTA-pair kernel (cta_group::2): the two CTAs of a cluster compute one
// 256 x 256 tile with a single stream of M=256, N=256, K=16 MMAs issued by the
// even CTA.  Each CTA holds its own 128 x 64 slice of A and one 64 x 128 half
// of B (columns rank * 128 ...) per stage, 32 KB instead of 48 KB, and the
// tensor core of each SM reads only that from its own shared memory (the B
// half of the other SM arrives over the pair link).  Each CTA's TMEM holds its
// 128 rows of the tile, so the epilogue is the one above, per CTA.
//
// Barriers (same offsets in both CTAs):
//   full[s]       even CTA only: one arrival (its producer, announcing the
//                 bytes of both CTAs) + the transaction bytes of both CTAs'
//                 copies, which signal it from either CTA;
//   empty[s]      in each CTA, one arrival from the MMA commit, multicast to
//                 both when the MMAs have read the stage;
//   tmem_full[b]  in each CTA, from the commit after a tile's last k-block;
//   tmem_empty[b] even CTA only: one arrival per epilogue warp of both CTAs.
#ifndef G12_TC_PAIR_STAGES
#define G12_TC_PAIR_STAGES 6
#endif
constexpr int PS = G12_TC_PAIR_STAGES;
constexpr int kPairBN = BN / 2;                         // B columns held per CTA
constexpr int kPairStageBytesA = BM * BK * 2;           // 16 KB
constexpr int kPairStageBytesB = BK * kPairBN * 2;      // 16 KB
constexpr int kPairStageBytes = kPairStageBytesA + kPairStageBytesB;
constexpr uint16_t kPairMask = 0x3;
constexpr uint32_t kPairIdesc = idesc_bf16_f32(2 * BM, BN, /*A MN-major*/ 0, /*B MN-major*/ 1);

struct __align__(8) PairSmemTail {
  uint64_t full[PS];
  uint64_t empty[PS];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int last_flag;
};

constexpr size_t kPairSmemBytes = 1024 + PS * kPairStageBytes + sizeof(PairSmemTail);
static_assert(kPairSmemBytes <= 227 * 1024, "pair kernel shared memory");

__global__ void __launch_bounds__(kThreads, 1)
    tc_bf16_pair_kernel(const __grid_constant__ TcArgs p, const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem<1024>(smem_raw);
  PairSmemTail* tail = reinterpret_cast<PairSmemTail*>(smem + PS * kPairStageBytes);
  volatile int* abort_flag = &tail->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int pairs_m = (tiles_m + 1) / 2;
  const int units = num_units(p, pairs_m * tiles_n);
  const int num_kb = (p.K + BK - 1) / BK;
  const uint32_t rank = cluster_cta_rank() & 1u;
  const bool even = (rank == 0);
  const int first_item = static_cast<int>(blockIdx.x) / 2;
  const int item_stride = static_cast<int>(gridDim.x) / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < PS; ++s) {
      mbar_init(&tail->full[s], 1);
      mbar_init(&tail->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tail->tmem_full[b], 1);
      mbar_init(&tail->tmem_empty[b], 2 * kEpiWarps);
    }
    mbar_init(&tail->drain, 1);
    tail->abort_flag = 0;
    tail->last_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(&tail->tmem_base, kTmemCols);
    tmem_relinquish_alloc_permit_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  // Both CTAs signal barriers of the even CTA: all must be initialised first.
  cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = tail->tmem_base;

  if (warp == 0) {
    // -------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint32_t full0 = mapa_shared(smem_u32(&tail->full[0]), 0);
      uint32_t it = 0;
      bool ok = true;
      for (int u = first_item; u < units && ok; u += item_stride) {
        const Unit w = unit_of(p, u, num_kb);
        int pm, tn;
        tile_coords(w.item, pairs_m, tiles_n, pm, tn);
        const int tm = pm * 2 + static_cast<int>(rank);
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int s = it % PS;
          const uint32_t round = it / PS;
          if (!mbar_wait(&tail->empty[s], (round & 1u) ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * kPairStageBytes;
          uint8_t* sb = sa + kPairStageBytesA;
          const uint32_t full = full0 + static_cast<uint32_t>(s * sizeof(uint64_t));
          if (even) mbar_arrive_expect_tx(&tail->full[s], 2 * kPairStageBytes);
          tma_load_2d_pair(sa, &tmA, kb * BK, tm * BM, full);
#pragma unroll
          for (int j = 0; j < kPairBN / 64; ++j)
            tma_load_2d_pair(sb + j * kBoxBytesB, &tmB,
                             tn * BN + static_cast<int>(rank) * kPairBN + j * 64, kb * BK, full);
        }
      }
      // Leave only after the MMAs have read every stage this CTA filled: then
      // all of its copies have landed and every commit aimed at its barriers
      // has arrived.  After an abort the stages may never be read; the wait
      // then gives up at the time limit, long after any copy has landed.
      const uint64_t t0 = globaltimer_ns();
      for (uint32_t j = it > PS ? it - PS : 0u; j < it; ++j) {
        while (!mbar_try_wait(&tail->empty[j % PS], (j / PS) & 1u)) {
          if (globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------- MMA issuer (even CTA only)
    if (even && lane == 0) {
      uint32_t it = 0;
      uint32_t j = 0;
      bool ok = true;
      bool issued = false;
      for (int u = first_item; u < units && ok; u += item_stride, ++j) {
        const Unit w = unit_of(p, u, num_kb);
        const uint32_t ab = j & 1u, ar = j >> 1;
        if (!mbar_wait(&tail->tmem_empty[ab], (ar & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + ab * BN;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int s = it % PS;
          const uint32_t round = it / PS;
          if (!mbar_wait(&tail->full[s], round & 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sa = smem_u32(smem + s * kPairStageBytes);
          const uint32_t sb = sa + kPairStageBytesA;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t adesc = smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bdesc = smem_desc_sw128(sb + kk * 2048, kBoxBytesB, 1024);
            tc_mma_f16_pair(d_tmem, adesc, bdesc, kPairIdesc, (kb != w.kb0 || kk != 0) ? 1u : 0u);
          }
          issued = true;
          tc_commit_pair_multicast(&tail->empty[s], kPairMask);
        }
        if (!ok) break;
        tc_commit_pair_multicast(&tail->tmem_full[ab], kPairMask);
      }
      if (ok) {
        // Wait for both CTAs' epilogues to release the last accumulators, so
        // that no arrival from the odd CTA is still on its way at exit.
        for (uint32_t jj = j > 2 ? j - 2 : 0u; jj < j; ++jj)
          if (!mbar_wait(&tail->tmem_empty[jj & 1u], (jj >> 1) & 1u, abort_flag, p.err)) break;
      } else if (issued) {
        // Let every MMA this thread issued finish before TMEM is released.
        tc_commit_pair(&tail->drain);
        mbar_drain_wait(&tail->drain, 0);
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int et = quarter * 32 + lane;
    float amax_acc = 0.0f;
    const uint32_t tmem_empty0 = mapa_shared(smem_u32(&tail->tmem_empty[0]), 0);
    uint32_t j = 0;
    for (int u = first_item; u < units; u += item_stride, ++j) {
      const Unit w = unit_of(p, u, num_kb);
      int pm, tn;
      tile_coords(w.item, pairs_m, tiles_n, pm, tn);
      const int tm = pm * 2 + static_cast<int>(rank);
      const uint32_t ab = j & 1u, ar = j >> 1;
      const bool ok = mbar_wait(&tail->tmem_full[ab], ar & 1u, abort_flag, p.err);
      if (named_bar_any(kEpiBarAny, kEpiThreads, !ok)) break;
      tc_fence_after_sync();
      const int row = tm * BM + et;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + ab * BN;
      // each CTA of the pair owns the counter and partials of its 128 rows
      const int slot = w.tail < 0 ? -1 : w.tail * 2 + static_cast<int>(rank);
      epilogue_unit(p, taddr, row, tn, slot, w.part, et, &tail->last_flag, amax_acc);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tmem_empty0 + ab * static_cast<uint32_t>(sizeof(uint64_t)));
    }
    epi_flush_amax(p.epi, amax_acc);
  }

  tc_fence_before_sync();
  __syncthreads();
  // Neither CTA releases TMEM or exits while the pair's MMAs or copies can
  // still touch it.
  cluster_sync();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

}  // namespace

// Clusters of the pair kernel that can be resident at once on the current
// device (one query per device).
static int pair_max_clusters(int num_sms) {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return num_sms / 2;
  }
  const int known = cache[dev].load(std::memory_order_relaxed);
  if (known > 0) return known;
  int clusters = 0;
  auto kernel = tc_bf16_pair_kernel;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kPairSmemBytes)) == cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (num_sms / 2));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kPairSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) clusters = 0;
  }
  cudaGetLastError();
  if (clusters < 1) clusters = num_sms / 2;
  cache[dev].store(clusters, std::memory_order_relaxed);
  return clusters;
}

TcPlan tc_plan(int M, int N, int K, int num_sms) {
  TcPlan pl{};
  const int tiles_m = (M + BM - 1) / BM;
  const int tiles_n = (N + BN - 1) / BN;
  const int num_kb = (K + BK - 1) / BK;
  pl.pair = tiles_m >= 2;
  const int ctas_per_item = pl.pair ? 2 : 1;
  const int items = pl.pair ? ((tiles_m + 1) / 2) * tiles_n : tiles_m * tiles_n;
  const int workers = pl.pair ? pair_max_clusters(num_sms) : num_sms;
  pl.split = tail_split(items, num_kb, workers, G12_TC_PART_COST);
  const int tail = pl.split > 1 ? (items >= workers ? items % workers : items) : 0;
  pl.full_items = items - tail;
  const int units = pl.full_items + tail * pl.split;
  pl.grid = ctas_per_item * (units < workers ? units : workers);
  pl.ws_floats = static_cast<int64_t>(tail) * pl.split * ctas_per_item * kPartFloats;
  pl.counters = static_cast<int64_t>(tail) * ctas_per_item;
  return pl;
}

cudaError_t launch_tc_bf16(const TcArgs& a, const TcPlan& plan, const CUtensorMap* tmA,
                           const CUtensorMap* tmB, cudaStream_t stream) {
  if (plan.grid < 1) return cudaSuccess;
  if (plan.pair) {
    auto kernel = tc_bf16_pair_kernel;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kPairSmemBytes));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kPairSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, a, *tmA, *tmB);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  auto kernel = tc_bf16_kernel;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  kernel<<<plan.grid, kThreads, kSmemBytes, stream>>>(a, *tmA, *tmB);
  return cudaGetLastError();
}

}  // namespace g12
