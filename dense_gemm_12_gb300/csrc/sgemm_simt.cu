// sgemm_simt.cu -- fp32 GEMM on the CUDA cores (FFMA), C = alpha*A*B + beta*C.
//
// Structure (the register-tiled scheme of "Tiled matrix multiplication",
// "How it works", and of "A GEMM Kernel, Step by Step", rungs four to six and
// "The last rung", rebuilt for sm_103a):
//   * persistent CTAs walk 128 x 128 output tiles in a grouped raster order so
//     CTAs running at the same time share A row-panels and B column-panels in
//     L2 ("Tiled matrix multiplication", "Complexity and constants");
//   * a producer warp streams 128 x 32 slices of A and 32 x 128 slices of B
//     into a STAGES-deep shared-memory ring with TMA (cp.async.bulk.tensor),
//     completion tracked by full/empty mbarriers -- the multi-buffered copy
//     pipeline the pages name for Hopper, which also frees the compute warps
//     from issuing any load instruction to global memory;
//   * 8 compute warps each own a 32 x 64 warp tile, every lane an 8 x 8
//     register micro-tile; per k the lane reads 8 A values and 8 B values from
//     shared memory with 128-bit loads and issues 64 FFMAs;
//   * the A slice stays k-contiguous (TMA cannot transpose fp32); the 128-byte
//     TMA swizzle plus a lane->row map of stride 4 keeps the 128-bit reads of
//     four k values at once free of bank conflicts, which replaces the pages'
//     transposed-and-padded A tile;
//   * TMA zero-fills rows and columns past M, N, K, so ragged edges need no
//     predicate in the hot loop; the epilogue applies alpha/beta and masks.
// Operands TMA cannot describe (unaligned base or pitch, or bf16 to be widened)
// are loaded by four producer warps with cp.async / plain loads into the same
// shared-memory layout, so the compute warps are identical in every variant.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace g12 {
namespace {

constexpr int BM = kSimtBM, BN = kSimtBN, BK = kSimtBK;
#ifndef G12_SIMT_KQ_UNROLL
#define G12_SIMT_KQ_UNROLL 8
#endif
#ifndef G12_SIMT_STAGES
#define G12_SIMT_STAGES 4
#endif
constexpr int STAGES = G12_SIMT_STAGES;
constexpr int kKqUnroll = G12_SIMT_KQ_UNROLL;  // unroll depth of the 4-k-step loop
// The block is launched with 384 threads x 168 registers = 64512.
constexpr int kLaunchRegs = 168;
constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kStageBytesA = BM * BK * 4;  // 16 KB, rows of 128 B, 128-B swizzled
constexpr int kStageBytesB = BK * BN * 4;  // 16 KB, rows of 512 B, not swizzled
constexpr int kStageBytes = kStageBytesA + kStageBytesB;

struct __align__(8) SimtSmemTail {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  int abort_flag;
  int last_flag;
};

// Tile and k-range of work item i (see SimtArgs).
struct SimtItem {
  int tm, tn;
  int kb0, kb1;    // k-blocks [kb0, kb1)
  int split_tile;  // -1 for a whole tile, else the index of the split tile
  int part;        // which of the split k-ranges
};

constexpr size_t kSmemBytes = 1024 /*alignment slack*/ + STAGES * kStageBytes +
                              sizeof(SimtSmemTail);

// Grouped raster: tiles walk column by column through groups of group_m
// tile rows, so neighbouring CTAs share A row panels and B column panels in L2.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m, int& tm,
                                            int& tn) {
  const int per_group = group_m * tiles_n;
  const int g = t / per_group;
  const int first_m = g * group_m;
  const int rows = min(tiles_m - first_m, group_m);
  const int local = t - g * per_group;
  tm = first_m + local % rows;
  tn = local / rows;
}

__device__ __forceinline__ SimtItem simt_item(const SimtArgs& p, int i, int tiles_m, int tiles_n,
                                              int num_kb) {
  SimtItem it;
  int tile;
  if (i < p.full_items) {
    tile = i;
    it.kb0 = 0;
    it.kb1 = num_kb;
    it.split_tile = -1;
    it.part = 0;
  } else {
    const int j = i - p.full_items;
    it.split_tile = j / p.split;
    it.part = j - it.split_tile * p.split;
    tile = p.full_items + it.split_tile;
    it.kb0 = static_cast<int>(static_cast<int64_t>(it.part) * num_kb / p.split);
    it.kb1 = static_cast<int>(static_cast<int64_t>(it.part + 1) * num_kb / p.split);
  }
  tile_coords(tile, tiles_m, tiles_n, p.group_m, it.tm, it.tn);
  return it;
}

// Byte offset of A element (m, k) inside a stage: 128-byte rows, the 16-byte
// chunk index XOR-ed with (m mod 8) -- the layout TMA's 128-byte swizzle
// writes into a 1024-byte aligned buffer.
__device__ __forceinline__ uint32_t a_smem_offset(int m, int k) {
  return static_cast<uint32_t>(m * 128 + ((((k >> 2) ^ (m & 7)) << 4)) + ((k & 3) << 2));
}

// Barrier among the 256 compute threads only (the producer warps never join).
__device__ __forceinline__ void compute_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kComputeThreads) : "memory");
}

template <int MODE_A, int MODE_B>
struct SimtTraits {
  static constexpr bool kAnyGeneric = (MODE_A != kLoadTma) || (MODE_B != kLoadTma);
  static constexpr bool kAnyTma = (MODE_A == kLoadTma) || (MODE_B == kLoadTma);
  // Always a full producer warpgroup, so the register split below works on
  // whole warpgroups (only one lane issues TMA when both operands use it).
  static constexpr int kProducerWarps = 4;
  static constexpr int kThreads = kComputeThreads + kProducerWarps * 32;
  // Arrivals that complete one phase of a full barrier: every generic
  // producer thread arrives once, the TMA issuer once (with the byte count).
  static constexpr uint32_t kFullCount = (kAnyGeneric ? 128u : 0u) + (kAnyTma ? 1u : 0u);
  // Per-thread register split between the two compute warpgroups and the
  // producer warpgroup; producers that widen bf16 keep more registers.
  static constexpr bool kConvert = (MODE_A == kLoadConvertBf16) || (MODE_B == kLoadConvertBf16);
  static constexpr int kProducerRegs = kConvert ? 72 : 56;
  static constexpr int kComputeRegs = kConvert ? 216 : 224;
  static_assert(256 * kComputeRegs + 128 * kProducerRegs <= 384 * kLaunchRegs,
                "register split exceeds the launch allocation");
  static constexpr uint32_t kTmaBytes =
      (MODE_A == kLoadTma ? kStageBytesA : 0) + (MODE_B == kLoadTma ? kStageBytesB : 0);
};

// ------------------------------------------------------------------ loaders
// Generic fp32 A slice: 128 rows x 32 k, 32 elements per producer thread,
// consecutive threads on consecutive k (coalesced reads of row-major A).
__device__ __forceinline__ void load_a_cpasync(uint8_t* sA, const float* A, int64_t lda, int M,
                                               int K, int m0, int k0, int ptid) {
#pragma unroll 8
  for (int q = 0; q < (BM * BK) / 128; ++q) {
    const int e = ptid + q * 128;
    const int m = e >> 5, k = e & 31;
    const int gm = m0 + m, gk = k0 + k;
    const bool in = (gm < M) && (gk < K);
    const float* src = in ? (A + static_cast<int64_t>(gm) * lda + gk) : A;
    cp_async_4(sA + a_smem_offset(m, k), src, in ? 4u : 0u);
  }
}

// Generic fp32 B slice: 32 k-rows x 128 n, consecutive threads on consecutive n.
__device__ __forceinline__ void load_b_cpasync(uint8_t* sB, const float* B, int64_t ldb, int N,
                                               int K, int n0, int k0, int ptid) {
#pragma unroll 8
  for (int q = 0; q < (BK * BN) / 128; ++q) {
    const int e = ptid + q * 128;
    const int k = e >> 7, n = e & 127;
    const int gk = k0 + k, gn = n0 + n;
    const bool in = (gk < K) && (gn < N);
    const float* src = in ? (B + static_cast<int64_t>(gk) * ldb + gn) : B;
    cp_async_4(sB + (k * BN + n) * 4, src, in ? 4u : 0u);
  }
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// bf16 A slice widened to fp32 (exact), same layout as the fp32 A slice.
// Parts stay rolled: each issues its 8 loads before its 8 stores, and the
// producer keeps few registers (the compute warps hold the rest).
__device__ __forceinline__ void load_a_bf16(uint8_t* sA, const uint16_t* A, int64_t lda, int M,
                                            int K, int m0, int k0, int ptid) {
#pragma unroll 1
  for (int part = 0; part < 4; ++part) {
    uint16_t v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = ptid + (part * 8 + q) * 128;
      const int m = e >> 5, k = e & 31;
      const int gm = m0 + m, gk = k0 + k;
      v[q] = (gm < M && gk < K) ? __ldg(A + static_cast<int64_t>(gm) * lda + gk) : uint16_t(0);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = ptid + (part * 8 + q) * 128;
      const int m = e >> 5, k = e & 31;
      *reinterpret_cast<float*>(sA + a_smem_offset(m, k)) = bf16_bits_to_f32(v[q]);
    }
  }
}

__device__ __forceinline__ void load_b_bf16(uint8_t* sB, const uint16_t* B, int64_t ldb, int N,
                                            int K, int n0, int k0, int ptid) {
#pragma unroll 1
  for (int part = 0; part < 4; ++part) {
    uint16_t v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = ptid + (part * 8 + q) * 128;
      const int k = e >> 7, n = e & 127;
      const int gk = k0 + k, gn = n0 + n;
      v[q] = (gk < K && gn < N) ? __ldg(B + static_cast<int64_t>(gk) * ldb + gn) : uint16_t(0);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = ptid + (part * 8 + q) * 128;
      const int k = e >> 7, n = e & 127;
      *reinterpret_cast<float*>(sB + (k * BN + n) * 4) = bf16_bits_to_f32(v[q]);
    }
  }
}

// ------------------------------------------------------- packed fp32 pairs
// sm_100-class GPUs execute two independent fp32 FMAs per lane from one
// fma.rn.f32x2 instruction (each lane-half rounds exactly like fmaf).  One
// issue slot then covers two FMA-pipe cycles, leaving slots free for the
// shared loads and address arithmetic of the micro-tile loop.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// ------------------------------------------------------------------ compute
// One stage (BK = 32 values of k) of the 8 x 8 outer-product accumulation.
// Lane layout inside the 32 x 64 warp tile: rg = lane / 8 picks rows
// {rg, rg+4, ..., rg+28}; cg = lane % 8 picks columns {4cg..4cg+3} and
// {32+4cg..32+4cg+3}.  A is read four k values at a time (one 128-bit load
// per row), B one k row at a time as two 128-bit loads.  The accumulators
// are fp32 pairs: acc2[i][q] holds the thread's columns 2q and 2q+1 of row i,
// updated with fma.rn.f32x2 (A value duplicated into both halves).
__device__ __forceinline__ void compute_stage_x2(const uint8_t* sA, const uint8_t* sB,
                                                 uint64_t (&acc2)[8][4], int wm, int wn,
                                                 int rg, int cg) {
  const uint8_t* a_row0 = sA + (wm * 32 + rg) * 128;
  const float* b_base = reinterpret_cast<const float*>(sB) + wn * 64 + cg * 4;
  const int x_even = rg;
  const int x_odd = rg + 4;
#pragma unroll kKqUnroll
  for (int kq = 0; kq < BK / 4; ++kq) {
    float4 a[8];
    const int off_even = (kq ^ x_even) << 4;
    const int off_odd = (kq ^ x_odd) << 4;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint8_t* p = a_row0 + i * 4 * 128 + ((i & 1) ? off_odd : off_even);
      a[i] = *reinterpret_cast<const float4*>(p);
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int k = kq * 4 + kk;
      const ulonglong2 b0 = *reinterpret_cast<const ulonglong2*>(b_base + k * BN);
      const ulonglong2 b1 = *reinterpret_cast<const ulonglong2*>(b_base + k * BN + 32);
      const uint64_t bv[4] = {b0.x, b0.y, b1.x, b1.y};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
        const uint64_t a2 = pack2(av, av);
#pragma unroll
        for (int q = 0; q < 4; ++q) acc2[i][q] = ffma2(a2, bv[q], acc2[i][q]);
      }
    }
  }
}

// C = alpha * acc + beta * C for the thread's 8 x 8 micro-tile.  For each
// 4-column half the old values of all 8 rows are loaded before any store, so
// the loads overlap; interleaved load/store pairs to possibly aliasing rows
// would serialise a memory round trip per row.
__device__ __forceinline__ void epilogue(const SimtArgs& p, const float (&acc)[8][8], int tm,
                                         int tn, int wm, int wn, int rg, int cg) {
  const bool read_c = (p.beta != 0.0f);
  const int row0 = tm * BM + wm * 32 + rg;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int col = tn * BN + wn * 64 + h * 32 + cg * 4;
    if (p.c_vec4 && col + 3 < p.N) {
      float4 old[8];
      if (read_c) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int row = row0 + 4 * i;
          old[i] = row < p.M ? *reinterpret_cast<const float4*>(
                                   p.C + static_cast<int64_t>(row) * p.ldc + col)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int row = row0 + 4 * i;
        if (row >= p.M) continue;
        float4 v = make_float4(acc[i][h * 4 + 0], acc[i][h * 4 + 1], acc[i][h * 4 + 2],
                               acc[i][h * 4 + 3]);
        if (read_c) {
          v.x = fmaf(p.alpha, v.x, p.beta * old[i].x);
          v.y = fmaf(p.alpha, v.y, p.beta * old[i].y);
          v.z = fmaf(p.alpha, v.z, p.beta * old[i].z);
          v.w = fmaf(p.alpha, v.w, p.beta * old[i].w);
        } else {
          v.x *= p.alpha;
          v.y *= p.alpha;
          v.z *= p.alpha;
          v.w *= p.alpha;
        }
        *reinterpret_cast<float4*>(p.C + static_cast<int64_t>(row) * p.ldc + col) = v;
      }
    } else {
      float old[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int row = row0 + 4 * i;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          old[i][c] = (read_c && row < p.M && col + c < p.N)
                          ? p.C[static_cast<int64_t>(row) * p.ldc + col + c]
                          : 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int row = row0 + 4 * i;
        if (row >= p.M) continue;
        float* c_row = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (col + c < p.N) {
            const float r = acc[i][h * 4 + c];
            c_row[col + c] = read_c ? fmaf(p.alpha, r, p.beta * old[i][c]) : p.alpha * r;
          }
        }
      }
    }
  }
}

template <int MODE_A, int MODE_B>
__global__ void __launch_bounds__(SimtTraits<MODE_A, MODE_B>::kThreads, 1)
    simt_gemm_kernel(const SimtArgs p, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB) {
  using T = SimtTraits<MODE_A, MODE_B>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem<1024>(smem_raw);
  SimtSmemTail* tail = reinterpret_cast<SimtSmemTail*>(smem + STAGES * kStageBytes);
  auto stage_a = [&](int s) { return smem + s * kStageBytes; };
  auto stage_b = [&](int s) { return smem + s * kStageBytes + kStageBytesA; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int num_tiles = tiles_m * tiles_n;
  const int num_kb = (p.K + BK - 1) / BK;
  const int num_items = p.full_items + (num_tiles - p.full_items) * p.split;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&tail->full[s], T::kFullCount);
      mbar_init(&tail->empty[s], kComputeThreads);
    }
    tail->abort_flag = 0;
    tail->last_flag = 0;
    fence_barrier_init();
  }
  if (MODE_A == kLoadTma && threadIdx.x == kComputeThreads) tma_prefetch_desc(&tmA);
  if (MODE_B == kLoadTma && threadIdx.x == kComputeThreads) tma_prefetch_desc(&tmB);
  __syncthreads();
  volatile int* abort_flag = &tail->abort_flag;
  // Launched with programmatic stream serialization: the set-up above touches
  // no global memory and may overlap the previous kernel's last CTAs; both
  // roles wait for its completion (grid_dependency_wait) before their first
  // global access.

  if (warp >= kComputeWarps) {
    // ------------------------------------------------------------ producers
    // Hand registers to the compute warpgroups (see SimtTraits: the split
    // never exceeds the 384 x 168 the block is launched with).
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(T::kProducerRegs));
    grid_dependency_wait();
    const int ptid = threadIdx.x - kComputeThreads;
    const bool tma_issuer = (ptid == 0) && T::kAnyTma;
    if (!T::kAnyGeneric && ptid != 0) return;
    uint32_t it = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < num_items && ok; i += gridDim.x) {
      const SimtItem w = simt_item(p, i, tiles_m, tiles_n, num_kb);
      const int tm = w.tm, tn = w.tn;
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t round = it / STAGES;
        if (!mbar_wait(&tail->empty[s], (round & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        if (tma_issuer) {
          mbar_arrive_expect_tx(&tail->full[s], T::kTmaBytes);
          if (MODE_A == kLoadTma) tma_load_2d(stage_a(s), &tmA, kb * BK, tm * BM, &tail->full[s]);
          if (MODE_B == kLoadTma) tma_load_2d(stage_b(s), &tmB, tn * BN, kb * BK, &tail->full[s]);
        }
        if (T::kAnyGeneric) {
          if (MODE_A == kLoadCpAsyncF32)
            load_a_cpasync(stage_a(s), static_cast<const float*>(p.A), p.lda, p.M, p.K, tm * BM,
                           kb * BK, ptid);
          if (MODE_B == kLoadCpAsyncF32)
            load_b_cpasync(stage_b(s), static_cast<const float*>(p.B), p.ldb, p.N, p.K, tn * BN,
                           kb * BK, ptid);
          if (MODE_A == kLoadConvertBf16)
            load_a_bf16(stage_a(s), static_cast<const uint16_t*>(p.A), p.lda, p.M, p.K, tm * BM,
                        kb * BK, ptid);
          if (MODE_B == kLoadConvertBf16)
            load_b_bf16(stage_b(s), static_cast<const uint16_t*>(p.B), p.ldb, p.N, p.K, tn * BN,
                        kb * BK, ptid);
          if (MODE_A == kLoadCpAsyncF32 || MODE_B == kLoadCpAsyncF32)
            cp_async_mbar_arrive_noinc(&tail->full[s]);
          else
            mbar_arrive(&tail->full[s]);
        }
      }
    }
    if (!ok) {
      // Drain this CTA's own copies still in flight before it may exit.
      if (T::kAnyGeneric) cp_async_wait_all();
      if (tma_issuer) {
        const uint32_t first = it > STAGES ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j) mbar_drain_wait(&tail->full[j % STAGES], (j / STAGES) & 1u);
      }
    }
    return;
  }

  // -------------------------------------------------------------- compute
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(T::kComputeRegs));
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int wm = warp >> 1, wn = warp & 1;
  const int rg = lane >> 3, cg = lane & 7;
  const int ctid = threadIdx.x;  // 0..255
  uint32_t it = 0;
  for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
    const SimtItem w = simt_item(p, item, tiles_m, tiles_n, num_kb);
    uint64_t acc2[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc2[i][q] = 0ull;
    bool failed = false;
    for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
      const int s = it % STAGES;
      const uint32_t round = it / STAGES;
      if (!mbar_wait(&tail->full[s], round & 1u, abort_flag, p.err)) {
        failed = true;
        break;
      }
      compute_stage_x2(stage_a(s), stage_b(s), acc2, wm, wn, rg, cg);
      mbar_arrive(&tail->empty[s]);
    }
    // Leave together if a wait ran out anywhere (see named_bar_any).
    if (named_bar_any(1, kComputeThreads, failed)) return;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) unpack2(acc2[i][q], acc[i][2 * q], acc[i][2 * q + 1]);
    if (w.split_tile < 0) {
      epilogue(p, acc, w.tm, w.tn, wm, wn, rg, cg);
      continue;
    }
    // Split tile: publish this k-range's partial sums (64 per thread, stored
    // contiguously per thread), then count the arrival; the last of the
    // tile's `split` parts adds all partials in part order -- a fixed order,
    // so the result does not depend on which part finishes last.
    float* mine = p.ws + (static_cast<int64_t>(w.split_tile * p.split + w.part) *
                              kComputeThreads + ctid) * 64;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      __stcg(reinterpret_cast<float4*>(mine + 8 * i),
             make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
      __stcg(reinterpret_cast<float4*>(mine + 8 * i + 4),
             make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]));
    }
    compute_bar();
    if (ctid == 0) {
      const uint32_t before = atomic_add_acq_rel_gpu(p.counters + w.split_tile, 1u);
      tail->last_flag = (before == static_cast<uint32_t>(p.split - 1)) ? 1 : 0;
    }
    compute_bar();
    const int last = tail->last_flag;
    if (last) {
      float sum[8][8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) sum[i][j] = 0.0f;
      // Parts are added in part order.  The variants whose producers widen
      // bf16 leave the compute warps fewer registers: there this thread's own
      // partial is read back from the workspace like the others (same
      // values, same order) so that its accumulators need not stay live;
      // elsewhere it comes from the accumulators, one round trip fewer.
      for (int part = 0; part < p.split; ++part) {
        const float* src = p.ws + (static_cast<int64_t>(w.split_tile * p.split + part) *
                                       kComputeThreads + ctid) * 64;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float v[8];
          if (!T::kConvert && part == w.part) {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = acc[i][j];
          } else {
            const float4 lo = __ldcg(reinterpret_cast<const float4*>(src + 8 * i));
            const float4 hi = __ldcg(reinterpret_cast<const float4*>(src + 8 * i + 4));
            v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w;
            v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) sum[i][j] += v[j];
        }
      }
      epilogue(p, sum, w.tm, w.tn, wm, wn, rg, cg);
      if (ctid == 0) p.counters[w.split_tile] = 0u;
    }
    compute_bar();  // last_flag is rewritten by the next split item
  }
}

template <int MODE_A, int MODE_B>
cudaError_t launch_variant(const SimtArgs& a, const CUtensorMap* tmA, const CUtensorMap* tmB,
                           int num_sms, cudaStream_t stream) {
  using T = SimtTraits<MODE_A, MODE_B>;
  auto kernel = simt_gemm_kernel<MODE_A, MODE_B>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
  const int num_items = a.full_items + (tiles - a.full_items) * a.split;
  const int grid = num_items < num_sms ? num_items : num_sms;
  CUtensorMap dummy{};
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(T::kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, a, tmA ? *tmA : dummy, tmB ? *tmB : dummy);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

SimtPlan simt_plan(int tiles, int num_kb, int num_sms, const TileConfig* fixed) {
  const int group_m = (fixed != nullptr && fixed->group_m > 0) ? fixed->group_m : 8;
  SimtPlan pl{tiles, 1, tiles < num_sms ? tiles : num_sms, group_m, 0, 0};
  if (tiles <= 0 || num_sms <= 0) return pl;
  // Tiles beyond the last full wave (all of them when there are fewer tiles
  // than SMs) are split along k when that shortens the last wave.
  // Measured split overhead: about 2 k-block times (2.6 us each) per part
  // and round.  A pinned split is capped at one k-block per part.
  int best_s = (fixed != nullptr && fixed->split > 0) ? fixed->split
                                                      : tail_split(tiles, num_kb, num_sms, 2.0);
  if (best_s > num_kb) best_s = num_kb;
  const int tail = tiles >= num_sms ? tiles % num_sms : tiles;
  if (best_s <= 1 || tail == 0) return pl;
  pl.full_items = tiles - tail;
  pl.split = best_s;
  const int items = pl.full_items + tail * best_s;
  pl.grid = items < num_sms ? items : num_sms;
  pl.ws_floats = static_cast<int64_t>(tail) * best_s * kComputeThreads * 64;
  pl.counters = tail;
  return pl;
}

cudaError_t launch_simt(const SimtArgs& a, LoadMode mode_a, LoadMode mode_b,
                        const CUtensorMap* tmA, const CUtensorMap* tmB, int num_sms,
                        cudaStream_t stream) {
  if (mode_a == kLoadTma && mode_b == kLoadTma)
    return launch_variant<kLoadTma, kLoadTma>(a, tmA, tmB, num_sms, stream);
  if (mode_a == kLoadCpAsyncF32 && mode_b == kLoadTma)
    return launch_variant<kLoadCpAsyncF32, kLoadTma>(a, tmA, tmB, num_sms, stream);
  if (mode_a == kLoadTma && mode_b == kLoadCpAsyncF32)
    return launch_variant<kLoadTma, kLoadCpAsyncF32>(a, tmA, tmB, num_sms, stream);
  if (mode_a == kLoadCpAsyncF32 && mode_b == kLoadCpAsyncF32)
    return launch_variant<kLoadCpAsyncF32, kLoadCpAsyncF32>(a, tmA, tmB, num_sms, stream);
  if (mode_a == kLoadConvertBf16 && mode_b == kLoadConvertBf16)
    return launch_variant<kLoadConvertBf16, kLoadConvertBf16>(a, tmA, tmB, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace g12
