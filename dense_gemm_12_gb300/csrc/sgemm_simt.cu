// sgemm_simt.cu -- fp32 GEMM on the CUDA cores (FFMA), C = alpha*A*B + beta*C.
//
// Structure (the register-tiled scheme of "Tiled matrix multiplication",
// "How it works", and of "A GEMM Kernel, Step by Step", rungs four to six and
// "The last rung", rebuilt for sm_103a):
//   * persistent CTAs walk 128 x BN output tiles (BN = 128 or 256) in a
//     grouped raster order so CTAs running at the same time share A
//     row-panels and B column-panels in L2 ("Tiled matrix multiplication",
//     "Complexity and constants");
//   * a producer warp streams 128 x 32 slices of A and 32 x BN slices of B
//     into a STAGES-deep shared-memory ring with TMA (cp.async.bulk.tensor),
//     completion tracked by full/empty mbarriers -- the multi-buffered copy
//     pipeline the pages name for Hopper, which also frees the compute warps
//     from issuing any load instruction to global memory;
//   * 8 compute warps each own a 32 x BN/2 warp tile, every lane an 8 x BN/16
//     register micro-tile; per k the lane reads 8 A values and BN/16 B values
//     from shared memory with 128-bit loads and issues 8 x BN/16 FFMAs.  The
//     wide tile (8 x 16 per lane) reads fewer shared-memory bytes per FMA;
//     the narrow one gives twice as many tiles for small problems;
//   * the A slice stays k-contiguous (TMA cannot transpose fp32); the 128-byte
//     TMA swizzle plus a lane->row map of stride 4 keeps the 128-bit reads of
//     four k values at once free of bank conflicts, which replaces the pages'
//     transposed-and-padded A tile;
//   * TMA zero-fills rows and columns past M, N, K, so ragged edges need no
//     predicate in the hot loop; the epilogue applies alpha/beta and masks;
//   * the tiles of the last, partial round are cut along k -- into equal
//     parts, or (stream-K) by dealing their k-blocks out evenly to all CTAs --
//     so that the last round keeps every SM busy ("A GEMM Kernel, Step by
//     Step", "The fringe and the last wave" and "What is left");
//   * when every tile fits in one round, the k-parts of a tile can instead
//     form a thread-block cluster and add their partial sums through
//     distributed shared memory, with no round trip through global memory.
// Operands TMA cannot describe (unaligned base or pitch, or bf16 to be widened)
// are loaded by four producer warps with cp.async / plain loads into the same
// shared-memory layout, so the compute warps are identical in every variant.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace g12 {
namespace {

constexpr int BM = kSimtBM, BK = kSimtBK;
// Unroll depth of the 4-k-step loop, per tile width (measured: the wide
// tile is 1.3 % faster at 4092^3 with 4 than with 8, the narrow one 3.5 %
// slower at 2048^3).
constexpr int kKqUnrollWide = 4, kKqUnrollNarrow = 8;
constexpr int STAGES = 4;
// The block is launched with 384 threads x 168 registers = 64512.
constexpr int kLaunchRegs = 168;
constexpr int kComputeWarps = 8;
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kStageBytesA = BM * BK * 4;  // 16 KB, rows of 128 B, 128-B swizzled

// Geometry that depends on the tile width BN.
template <int BN>
struct Geom {
  static_assert(BN == 128 || BN == 256, "tile width");
  static constexpr int kColGroups = BN / 64;            // 4-column groups per lane
  static constexpr int kCols = 4 * kColGroups;          // columns per lane
  static constexpr int kAcc = 8 * kCols;                // accumulators per lane
  static constexpr int kStageBytesB = BK * BN * 4;      // rows of BN x 4 B, not swizzled
  static constexpr int kStageBytes = kStageBytesA + kStageBytesB;
  static constexpr int kKqUnroll = BN == 256 ? kKqUnrollWide : kKqUnrollNarrow;
};

struct __align__(8) SimtSmemTail {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t ready;   // cluster fix-up: every CTA's partial sums are stored
  uint64_t done;    // cluster fix-up: every CTA has read this one's
  int abort_flag;
  int last_flag;
};

template <int BN>
constexpr size_t smem_bytes() {
  return 1024 /*alignment slack*/ + STAGES * Geom<BN>::kStageBytes + sizeof(SimtSmemTail);
}

// Tile and k-range of work item i (see SimtArgs).
struct SimtItem {
  int tm, tn;
  int kb0, kb1;    // k-blocks [kb0, kb1); empty items (kb0 == kb1) are skipped
  int tail_tile;   // -1 for a whole tile, else the index of the tail tile
  int part;        // this item's place among the tile's parts, in k order
  int parts;       // number of parts of the tile
  int slot;        // workspace slot of this part's partial sums
};

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

// Workspace slot of part `idx` (k order) of tail tile t.
__device__ __forceinline__ int part_slot(const SimtArgs& p, int t, int idx, int num_kb,
                                         int64_t W) {
  if (p.sk_workers == 0) return t * p.split + idx;
  const int64_t G = p.sk_workers;
  const int64_t first = sk_worker(static_cast<int64_t>(t) * num_kb, W, G);
  const int64_t j = first + idx;
  return static_cast<int>(2 * j + (sk_lo(j, W, G) < static_cast<int64_t>(t) * num_kb ? 1 : 0));
}

__device__ __forceinline__ SimtItem simt_item(const SimtArgs& p, int i, int tiles_m, int tiles_n,
                                              int num_kb) {
  SimtItem it;
  int tile;
  it.tail_tile = -1;
  it.part = 0;
  it.parts = 1;
  it.slot = 0;
  if (i < p.full_items) {
    tile = i;
    it.kb0 = 0;
    it.kb1 = num_kb;
  } else if (p.sk_workers == 0) {
    const int j = i - p.full_items;
    it.tail_tile = j / p.split;
    it.part = j - it.tail_tile * p.split;
    it.parts = p.split;
    it.slot = j;
    tile = p.full_items + it.tail_tile;
    it.kb0 = static_cast<int>(static_cast<int64_t>(it.part) * num_kb / p.split);
    it.kb1 = static_cast<int>(static_cast<int64_t>(it.part + 1) * num_kb / p.split);
  } else {
    // Stream-K: items full_items + s * gridDim.x + w are segment s of worker w.
    const int j = i - p.full_items;
    const int s = j / static_cast<int>(gridDim.x);
    const int w = j - s * static_cast<int>(gridDim.x);
    const int64_t G = p.sk_workers;
    const int64_t W = static_cast<int64_t>(tiles_m * tiles_n - p.full_items) * num_kb;
    it.kb0 = it.kb1 = 0;
    it.tm = it.tn = 0;
    if (w >= G) return it;
    const int64_t lo = sk_lo(w, W, G), hi = sk_lo(w + 1, W, G);
    int64_t t = lo / num_kb;
    int64_t a = lo - t * num_kb, b = min(hi - t * num_kb, static_cast<int64_t>(num_kb));
    if (s == 1) {
      if (hi <= (t + 1) * num_kb) return it;
      ++t;
      a = 0;
      b = hi - t * num_kb;
    }
    it.tail_tile = static_cast<int>(t);
    it.kb0 = static_cast<int>(a);
    it.kb1 = static_cast<int>(b);
    const int64_t first = sk_worker(t * num_kb, W, G);
    const int64_t last = sk_worker((t + 1) * num_kb - 1, W, G);
    it.part = static_cast<int>(w - first);
    it.parts = static_cast<int>(last - first + 1);
    it.slot = 2 * w + s;
    tile = p.full_items + it.tail_tile;
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

// Generic fp32 B slice: 32 k-rows x BN n, consecutive threads on consecutive n.
template <int BN>
__device__ __forceinline__ void load_b_cpasync(uint8_t* sB, const float* B, int64_t ldb, int N,
                                               int K, int n0, int k0, int ptid) {
#pragma unroll 8
  for (int q = 0; q < (BK * BN) / 128; ++q) {
    const int e = ptid + q * 128;
    const int k = e / BN, n = e % BN;
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
  for (int part = 0; part < (BM * BK) / 1024; ++part) {
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

template <int BN>
__device__ __forceinline__ void load_b_bf16(uint8_t* sB, const uint16_t* B, int64_t ldb, int N,
                                            int K, int n0, int k0, int ptid) {
#pragma unroll 1
  for (int part = 0; part < (BK * BN) / 1024; ++part) {
    uint16_t v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = ptid + (part * 8 + q) * 128;
      const int k = e / BN, n = e % BN;
      const int gk = k0 + k, gn = n0 + n;
      v[q] = (gk < K && gn < N) ? __ldg(B + static_cast<int64_t>(gk) * ldb + gn) : uint16_t(0);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int e = ptid + (part * 8 + q) * 128;
      const int k = e / BN, n = e % BN;
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
// One stage (BK = 32 values of k) of the 8 x kCols outer-product
// accumulation.  Lane layout inside the 32 x BN/2 warp tile: rg = lane / 8
// picks rows {rg, rg+4, ..., rg+28}; cg = lane % 8 picks the columns
// {32j + 4cg .. 32j + 4cg + 3}, j < kColGroups.  A is read four k values at a
// time (one 128-bit load per row), B one k row at a time as kColGroups
// 128-bit loads.  The accumulators are fp32 pairs: acc2[i][2j + h] holds
// columns 32j + 4cg + 2h and +1 of row i, updated with fma.rn.f32x2 (the A
// value duplicated into both halves).
template <int BN>
__device__ __forceinline__ void compute_stage_x2(const uint8_t* sA, const uint8_t* sB,
                                                 uint64_t (&acc2)[8][Geom<BN>::kCols / 2],
                                                 int wm, int wn, int rg, int cg) {
  constexpr int kGroups = Geom<BN>::kColGroups;
  const uint8_t* a_row0 = sA + (wm * 32 + rg) * 128;
  const float* b_base = reinterpret_cast<const float*>(sB) + wn * (BN / 2) + cg * 4;
  const int x_even = rg;
  const int x_odd = rg + 4;
#pragma unroll Geom<BN>::kKqUnroll
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
      uint64_t bv[2 * kGroups];
#pragma unroll
      for (int j = 0; j < kGroups; ++j) {
        const ulonglong2 b = *reinterpret_cast<const ulonglong2*>(b_base + k * BN + 32 * j);
        bv[2 * j] = b.x;
        bv[2 * j + 1] = b.y;
      }
      uint64_t a2[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
        a2[i] = pack2(av, av);
      }
      // Column pairs outermost, rows in a snake (0..7, then 7..0): each FMA
      // shares its B pair with the previous one, and at a turn also its A
      // pair.  Measured against rows outermost (the same FMAs in another
      // order, bitwise the same sums): 2.080 vs 2.135 ms at 4092^3.
#pragma unroll
      for (int q = 0; q < 2 * kGroups; ++q)
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int i = (q & 1) ? 7 - r : r;
          acc2[i][q] = ffma2(a2[i], bv[q], acc2[i][q]);
        }
    }
  }
}

// C = alpha * acc + beta * C for the thread's 8 x kCols micro-tile, kRows rows
// at a time: the old values of a chunk's rows are all loaded before any of
// them is stored, so their round trips overlap (a load issued after a store
// to a possibly aliasing address would wait for it).  Batch sizes below.
template <int BN>
__device__ __forceinline__ void epilogue(const SimtArgs& p, const float (&acc)[8][Geom<BN>::kCols],
                                         int tm, int tn, int wm, int wn, int rg, int cg) {
  constexpr int kGroups = Geom<BN>::kColGroups;
  const bool read_c = (p.beta != 0.0f);
  const int row0 = tm * BM + wm * 32 + rg;
  const int col0 = tn * BN + wn * (BN / 2) + cg * 4;
  const bool vec = p.c_vec4 && col0 + 32 * (kGroups - 1) + 3 < p.N;
  if (vec) {
    // Rows in flight per batch: all 8 on the narrow tile; 2 on the wide one,
    // whose 128 accumulators leave room for 32 old values but not 64 (4 rows
    // spilled, and made the k loop 1.5 % slower; 1 row left 8 serial round
    // trips to memory: 2 rows took 4092^3 with beta != 0 from 2.055 to
    // 2.044 ms).  A running row pointer keeps the addresses in two registers.
    constexpr int kRows = BN == 128 ? 8 : 2;
    const int64_t row_step = 4 * p.ldc;
    float* c_next = p.C + static_cast<int64_t>(row0) * p.ldc + col0;
#pragma unroll
    for (int i0 = 0; i0 < 8; i0 += kRows) {
      float4 old[kRows][kGroups];
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const int row = row0 + 4 * (i0 + r);
        const float* c_row = c_next + r * row_step;
#pragma unroll
        for (int h = 0; h < kGroups; ++h)
          old[r][h] = (read_c && row < p.M) ? *reinterpret_cast<const float4*>(c_row + 32 * h)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        const int i = i0 + r;
        const int row = row0 + 4 * i;
        if (row >= p.M) continue;
        float* c_row = c_next + r * row_step;
#pragma unroll
        for (int h = 0; h < kGroups; ++h) {
          float4 v = make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2],
                                 acc[i][4 * h + 3]);
          if (read_c) {
            v.x = fmaf(p.alpha, v.x, p.beta * old[r][h].x);
            v.y = fmaf(p.alpha, v.y, p.beta * old[r][h].y);
            v.z = fmaf(p.alpha, v.z, p.beta * old[r][h].z);
            v.w = fmaf(p.alpha, v.w, p.beta * old[r][h].w);
          } else {
            v.x *= p.alpha;
            v.y *= p.alpha;
            v.z *= p.alpha;
            v.w *= p.alpha;
          }
          *reinterpret_cast<float4*>(c_row + 32 * h) = v;
        }
      }
      c_next += kRows * row_step;
    }
    return;
  }
  // Edge tiles and C rows without float4 alignment: element by element.
  constexpr int kRows = BN == 128 ? 8 : 1;
#pragma unroll
  for (int i0 = 0; i0 < 8; i0 += kRows) {
    float old[kRows][4 * kGroups];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int row = row0 + 4 * (i0 + r);
      const float* c_row = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
      for (int h = 0; h < kGroups; ++h)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int col = col0 + 32 * h + c;
          old[r][4 * h + c] = (read_c && row < p.M && col < p.N) ? c_row[col] : 0.0f;
        }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int i = i0 + r;
      const int row = row0 + 4 * i;
      if (row >= p.M) continue;
      float* c_row = p.C + static_cast<int64_t>(row) * p.ldc;
#pragma unroll
      for (int h = 0; h < kGroups; ++h)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int col = col0 + 32 * h + c;
          if (col < p.N) {
            const float x = acc[i][4 * h + c];
            c_row[col] = read_c ? fmaf(p.alpha, x, p.beta * old[r][4 * h + c]) : p.alpha * x;
          }
        }
    }
  }
}

// ------------------------------------------------- cluster fix-up (split)
// The cluster handshake.  Every thread arrives once on the cluster barrier
// right after the mbarriers are initialised (non-blocking), so the idle
// producer threads can exit at once, as in the unclustered kernel -- idle
// warps left resident through the k loop, even asleep, measured 4-5 % slower
// k loops.  The compute warps wait on that one phase before their first
// access to another CTA; the later steps use the `ready` and `done`
// mbarriers, arrived on from every CTA of the cluster (release at cluster
// scope) and waited on with a bound.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait with acquire at cluster scope; as mbar_wait when `abort_flag`
// is given, else with the limit alone and no record.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag, uint32_t* err_word,
                                                  uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (abort_flag != nullptr && *abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      if (abort_flag != nullptr) {
        *abort_flag = 1;
        atomicOr(err_word, kErrWaitTimeout);
      }
      return false;
    }
  }
  return true;
}

// Arrive on mbarrier `bar` (same offset) in every CTA of the cluster: thread
// r < S of the calling threads arrives on CTA r's, all in one instruction.
// Called after a barrier of the compute threads, so each arrival (a release
// at cluster scope) also covers the other threads' earlier accesses.
__device__ __forceinline__ void mbar_arrive_all(uint64_t* bar, int S, int ctid) {
  if (ctid < S) mbar_arrive_cluster(mapa_shared(smem_u32(bar), static_cast<uint32_t>(ctid)));
}

// Float4 groups of the 128 x 128 tile one compute thread reduces in a
// cluster of S >= 2 CTAs: at most 4096 / (2 * 256).
constexpr int kClusterMaxGroups = (BM * 128 / 4) / (2 * kComputeThreads);

// The partial sums of the cluster's S k-parts of one 128 x 128 tile lie in
// each CTA's shared memory as a row-major tile (`part_u32`: its shared
// address, the same in every CTA).  CTA `rank` takes an S-th of the tile's
// float4 groups (group g of this thread: cluster_group) and adds the S
// partials of each in rank (= k) order starting from zero -- the order of
// the global-memory fix-up, so both give the same bits.  All of a thread's
// loads from one CTA are in flight at once: S round trips in all.
__device__ __forceinline__ int cluster_group(int S, int rank, int ctid, int g, int* q1) {
  constexpr int kGroups = BM * 128 / 4;
  *q1 = static_cast<int>(static_cast<int64_t>(rank + 1) * kGroups / S);
  return static_cast<int>(static_cast<int64_t>(rank) * kGroups / S) + ctid + g * kComputeThreads;
}

__device__ __forceinline__ void cluster_gather(uint32_t part_u32, int S, int rank, int ctid,
                                               float4 (&sum)[kClusterMaxGroups]) {
  constexpr int G = kClusterMaxGroups;
#pragma unroll
  for (int g = 0; g < G; ++g) sum[g] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r = 0; r < S; ++r) {
    float4 v[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      int q1;
      const int q = cluster_group(S, rank, ctid, g, &q1);
      v[g] = q < q1 ? ld_shared_cluster_v4(mapa_shared(part_u32 + static_cast<uint32_t>(q) * 16u,
                                                       static_cast<uint32_t>(r)))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      sum[g].x += v[g].x;
      sum[g].y += v[g].y;
      sum[g].z += v[g].z;
      sum[g].w += v[g].w;
    }
  }
}

// C = alpha * sum + beta * C for the groups of cluster_gather, with the
// edge masks.  All old C values are loaded before any store (a load after a
// store to C would wait for it): one round trip to memory.
__device__ __forceinline__ void cluster_store(const SimtArgs& p, int S, int rank, int tm, int tn,
                                              int ctid, const float4 (&sum)[kClusterMaxGroups]) {
  constexpr int G = kClusterMaxGroups;
  const bool read_c = (p.beta != 0.0f);
  float old[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    int q1;
    const int q = cluster_group(S, rank, ctid, g, &q1);
    const int row = tm * BM + (q >> 5);
    const int col = tn * 128 + (q & 31) * 4;
    const float* c_row = p.C + static_cast<int64_t>(row) * p.ldc;
    const bool live = read_c && q < q1 && row < p.M;
    if (live && p.c_vec4 && col + 3 < p.N) {
      const float4 o = *reinterpret_cast<const float4*>(c_row + col);
      old[g][0] = o.x;
      old[g][1] = o.y;
      old[g][2] = o.z;
      old[g][3] = o.w;
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) old[g][c] = (live && col + c < p.N) ? c_row[col + c] : 0.0f;
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    int q1;
    const int q = cluster_group(S, rank, ctid, g, &q1);
    const int row = tm * BM + (q >> 5);
    const int col = tn * 128 + (q & 31) * 4;
    if (q >= q1 || row >= p.M) continue;
    float* c_row = p.C + static_cast<int64_t>(row) * p.ldc;
    const float x[4] = {sum[g].x, sum[g].y, sum[g].z, sum[g].w};
    float y[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) y[c] = read_c ? fmaf(p.alpha, x[c], p.beta * old[g][c]) : p.alpha * x[c];
    if (p.c_vec4 && col + 3 < p.N) {
      *reinterpret_cast<float4*>(c_row + col) = make_float4(y[0], y[1], y[2], y[3]);
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (col + c < p.N) c_row[col + c] = y[c];
    }
  }
}

// CLUSTER: the launch is a grid of clusters of p.cluster CTAs, one per k-part
// of a tile (full_items = 0, split = p.cluster, one item per CTA); the parts
// are added through distributed shared memory instead of the workspace.
template <int MODE_A, int MODE_B, int BN, bool CLUSTER>
__global__ void __launch_bounds__(SimtTraits<MODE_A, MODE_B>::kThreads, 1)
    simt_gemm_kernel(const SimtArgs p, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB) {
  static_assert(!CLUSTER || BN == 128, "the cluster fix-up is written for 128 x 128 tiles");
  using T = SimtTraits<MODE_A, MODE_B>;
  using Gm = Geom<BN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem<1024>(smem_raw);
  SimtSmemTail* tail = reinterpret_cast<SimtSmemTail*>(smem + STAGES * Gm::kStageBytes);
  auto stage_a = [&](int s) { return smem + s * Gm::kStageBytes; };
  auto stage_b = [&](int s) { return smem + s * Gm::kStageBytes + kStageBytesA; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int num_tiles = tiles_m * tiles_n;
  const int num_kb = (p.K + BK - 1) / BK;
  const int num_items = p.sk_workers > 0
                            ? p.full_items + 2 * static_cast<int>(gridDim.x)
                            : p.full_items + (num_tiles - p.full_items) * p.split;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&tail->full[s], T::kFullCount);
      mbar_init(&tail->empty[s], kComputeWarps);
    }
    mbar_init(&tail->ready, CLUSTER ? static_cast<uint32_t>(p.cluster) : 1u);
    mbar_init(&tail->done, CLUSTER ? static_cast<uint32_t>(p.cluster) : 1u);
    tail->abort_flag = 0;
    tail->last_flag = 0;
    fence_barrier_init();
  }
  if (MODE_A == kLoadTma && threadIdx.x == kComputeThreads) tma_prefetch_desc(&tmA);
  if (MODE_B == kLoadTma && threadIdx.x == kComputeThreads) tma_prefetch_desc(&tmB);
  __syncthreads();
  if (CLUSTER) cluster_arrive_release();  // this CTA's barriers are initialised
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
          constexpr uint32_t kTmaBytes = (MODE_A == kLoadTma ? kStageBytesA : 0) +
                                         (MODE_B == kLoadTma ? Gm::kStageBytesB : 0);
          mbar_arrive_expect_tx(&tail->full[s], kTmaBytes);
          if (MODE_A == kLoadTma) tma_load_2d(stage_a(s), &tmA, kb * BK, tm * BM, &tail->full[s]);
          if (MODE_B == kLoadTma) tma_load_2d(stage_b(s), &tmB, tn * BN, kb * BK, &tail->full[s]);
        }
        if (T::kAnyGeneric) {
          if (MODE_A == kLoadCpAsyncF32)
            load_a_cpasync(stage_a(s), static_cast<const float*>(p.A), p.lda, p.M, p.K, tm * BM,
                           kb * BK, ptid);
          if (MODE_B == kLoadCpAsyncF32)
            load_b_cpasync<BN>(stage_b(s), static_cast<const float*>(p.B), p.ldb, p.N, p.K,
                               tn * BN, kb * BK, ptid);
          if (MODE_A == kLoadConvertBf16)
            load_a_bf16(stage_a(s), static_cast<const uint16_t*>(p.A), p.lda, p.M, p.K, tm * BM,
                        kb * BK, ptid);
          if (MODE_B == kLoadConvertBf16)
            load_b_bf16<BN>(stage_b(s), static_cast<const uint16_t*>(p.B), p.ldb, p.N, p.K,
                            tn * BN, kb * BK, ptid);
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
  const int64_t tail_kb = static_cast<int64_t>(num_tiles - p.full_items) * num_kb;
  uint32_t it = 0;
  for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
    const SimtItem w = simt_item(p, item, tiles_m, tiles_n, num_kb);
    if (!CLUSTER && w.kb0 == w.kb1) continue;  // an empty stream-K segment
    uint64_t acc2[8][Gm::kCols / 2];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int q = 0; q < Gm::kCols / 2; ++q) acc2[i][q] = 0ull;
    bool failed = false;
    for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
      const int s = it % STAGES;
      const uint32_t round = it / STAGES;
      if (!mbar_wait(&tail->full[s], round & 1u, abort_flag, p.err)) {
        failed = true;
        break;
      }
      compute_stage_x2<BN>(stage_a(s), stage_b(s), acc2, wm, wn, rg, cg);
      // One arrival per warp, after all its lanes' shared-memory reads.
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->empty[s]);
    }
    // Leave together if a wait ran out anywhere (see named_bar_any).
    const bool any_failed = named_bar_any(1, kComputeThreads, failed);
    if (CLUSTER) {
      // Every compute warp is past its last stage (the barrier above), so
      // the ring is free: the partial sums go to its first 64 KB as a
      // row-major 128 x 128 tile.  After a wait ran out the ring may still
      // be receiving copies: nothing is written or read, but the CTA still
      // arrives on every barrier its peers wait for.
      if (!any_failed) {
        float* part = reinterpret_cast<float*>(smem);
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int q = 0; q < Gm::kCols / 2; q += 2) {
            float4 v;
            unpack2(acc2[i][q], v.x, v.y);
            unpack2(acc2[i][q + 1], v.z, v.w);
            const int row = wm * 32 + rg + 4 * i;
            const int col = wn * 64 + cg * 4 + 32 * (q / 2);
            *reinterpret_cast<float4*>(part + row * 128 + col) = v;
          }
      }
      cluster_wait_acquire();  // every CTA of the cluster has its barriers
      compute_bar();           // this CTA's partial sums are all stored
      mbar_arrive_all(&tail->ready, p.cluster, ctid);
      if (ctid == 0)
        tail->last_flag =
            mbar_wait_cluster(&tail->ready, 0, abort_flag, p.err, kWaitLimitNs) ? 1 : 0;
      compute_bar();
      const bool reduce = tail->last_flag && !any_failed;
      const int rank = static_cast<int>(cluster_cta_rank());
      float4 sum[kClusterMaxGroups];
      if (reduce) cluster_gather(smem_u32(smem), p.cluster, rank, ctid, sum);
      compute_bar();  // this CTA's reads of the other CTAs are done
      mbar_arrive_all(&tail->done, p.cluster, ctid);
      if (reduce) cluster_store(p, p.cluster, rank, w.tm, w.tn, ctid, sum);
      // The CTA (its shared memory) stays until every CTA has read it.  The
      // wait ignores this CTA's abort flag and outlasts a peer's bounded wait
      // on `ready`, after which that peer arrives here too.
      if (ctid == 0) mbar_wait_cluster(&tail->done, 0, nullptr, nullptr, 2 * kWaitLimitNs);
      return;
    }
    if (any_failed) return;
    float acc[8][Gm::kCols];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int q = 0; q < Gm::kCols / 2; ++q) unpack2(acc2[i][q], acc[i][2 * q], acc[i][2 * q + 1]);
    if (w.tail_tile < 0) {
      epilogue<BN>(p, acc, w.tm, w.tn, wm, wn, rg, cg);
      continue;
    }
    // Part of a tail tile: publish this k-range's partial sums, then count
    // the arrival; the last of the tile's parts adds all partials in k order
    // -- a fixed order, so the result does not depend on which part finishes
    // last.  Float4 q of thread t of a part lies at q * 256 + t, so a warp's
    // stores and loads cover whole lines (each thread's partial stored
    // contiguously left a warp's 16-byte loads on 32 lines: 4092^3 2.045 ->
    // 2.024 ms, 2048^3 287 -> 269 us, 3000 x 5000 x 1999 992 -> 966 us).
    constexpr int Q = Gm::kAcc / 4;  // float4s per thread and part
    float4* const ws4 = reinterpret_cast<float4*>(p.ws);
    auto part_base = [&](int slot) {
      return ws4 + static_cast<int64_t>(slot) * Q * kComputeThreads + ctid;
    };
    {
      float4* mine = part_base(w.slot);
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int h = 0; h < Gm::kColGroups; ++h)
          __stcg(mine + (Gm::kColGroups * i + h) * kComputeThreads,
                 make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]));
    }
    compute_bar();
    if (ctid == 0) {
      const uint32_t before = atomic_add_acq_rel_gpu(p.counters + w.tail_tile, 1u);
      tail->last_flag = (before == static_cast<uint32_t>(w.parts - 1)) ? 1 : 0;
    }
    compute_bar();
    const int last = tail->last_flag;
    if (last) {
      float sum[8][Gm::kCols];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < Gm::kCols; ++j) sum[i][j] = 0.0f;
      // Parts are added in k order.  This thread's own partial comes from
      // its accumulators where registers allow (the narrow tile with fp32
      // producers), else it is read back from the workspace like the others
      // (same values, same order), so that the accumulators need not stay
      // live next to the sums.  (Adding the parts two at a time, two rows at
      // a time, each pair of rows straight through the output stage, cut the
      // loads' round trips but made the wide tile's k loop ~1 % slower.)
      constexpr bool kKeepOwn = (Gm::kAcc <= 64) && !T::kConvert;
      for (int part = 0; part < w.parts; ++part) {
        const float4* src = part_base(part_slot(p, w.tail_tile, part, num_kb, tail_kb));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float v[Gm::kCols];
          if (kKeepOwn && part == w.part) {
#pragma unroll
            for (int j = 0; j < Gm::kCols; ++j) v[j] = acc[i][j];
          } else {
#pragma unroll
            for (int h = 0; h < Gm::kColGroups; ++h) {
              const float4 q = __ldcg(src + (Gm::kColGroups * i + h) * kComputeThreads);
              v[4 * h] = q.x;
              v[4 * h + 1] = q.y;
              v[4 * h + 2] = q.z;
              v[4 * h + 3] = q.w;
            }
          }
#pragma unroll
          for (int j = 0; j < Gm::kCols; ++j) sum[i][j] += v[j];
        }
      }
      epilogue<BN>(p, sum, w.tm, w.tn, wm, wn, rg, cg);
    }
    if (last && ctid == 0) p.counters[w.tail_tile] = 0u;
    compute_bar();  // last_flag is rewritten by the next tail item
  }
}

template <int MODE_A, int MODE_B, int BN, bool CLUSTER = false>
cudaError_t launch_variant(const SimtArgs& a, int grid, const CUtensorMap* tmA,
                           const CUtensorMap* tmB, cudaStream_t stream) {
  using T = SimtTraits<MODE_A, MODE_B>;
  constexpr size_t kSmem = smem_bytes<BN>();
  auto kernel = simt_gemm_kernel<MODE_A, MODE_B, BN, CLUSTER>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmem));
  if (e != cudaSuccess) return e;
  CUtensorMap dummy{};
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CLUSTER ? static_cast<unsigned>(a.cluster) : 1u;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(T::kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = CLUSTER ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kernel, a, tmA ? *tmA : dummy, tmB ? *tmB : dummy);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BN>
cudaError_t launch_width(const SimtArgs& a, int grid, LoadMode mode_a, LoadMode mode_b,
                         const CUtensorMap* tmA, const CUtensorMap* tmB, cudaStream_t stream) {
  if (mode_a == kLoadTma && mode_b == kLoadTma)
    return launch_variant<kLoadTma, kLoadTma, BN>(a, grid, tmA, tmB, stream);
  if (mode_a == kLoadCpAsyncF32 && mode_b == kLoadTma)
    return launch_variant<kLoadCpAsyncF32, kLoadTma, BN>(a, grid, tmA, tmB, stream);
  if (mode_a == kLoadTma && mode_b == kLoadCpAsyncF32)
    return launch_variant<kLoadTma, kLoadCpAsyncF32, BN>(a, grid, tmA, tmB, stream);
  if (mode_a == kLoadCpAsyncF32 && mode_b == kLoadCpAsyncF32)
    return launch_variant<kLoadCpAsyncF32, kLoadCpAsyncF32, BN>(a, grid, tmA, tmB, stream);
  if (mode_a == kLoadConvertBf16 && mode_b == kLoadConvertBf16)
    return launch_variant<kLoadConvertBf16, kLoadConvertBf16, BN>(a, grid, tmA, tmB, stream);
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------- planning
// Measured cost of cutting a tile into parts through the workspace, in
// k-blocks of the tile's own width per part (storing its partial sums, and
// for the last part reading the others and writing the tile): per-CTA
// timestamps put the end of the last part 7.4, 11 and 19 us after the end of
// the k loops for 2, 4 and 8 parts (k-blocks of ~2.5 us): 1.0-1.5 per part,
// with each thread's partial stored contiguously.  Stored warp-coalesced it
// costs less; 0.8 leaves the fewest sweep classes whose fastest plan the
// model misses (26 of 216 with the stream-K constants below; 0.3, closer to
// the ~0.2 per part of 16 tiles of 64 k-blocks -- 8 parts through the
// workspace 31.6 us, 6 in clusters 38.1 us -- left 34: it over-picks the
// 128 x 256 tile with equal splits where narrow stream-K tails win).
constexpr double kSplitFixupKb = 0.8;
// A k-block of a 128 x 256 tile costs about 1.86 k-blocks of a 128 x 128 tile
// (twice the FMAs at ~7 % better FMA-pipe use: fewer shared-memory reads per
// FMA, and the 4-fold unroll of its k loop).  Measured on shapes that both
// widths cover in whole rounds (2432 x {2048, 4096, 8192} x {1024, 2048,
// 4096}): 1.845-1.867.
constexpr double kWideKbCost = 1.86;
// Least k-blocks per stream-K range the cost model picks (a pinned stream-K
// tail goes down to one).
constexpr int kStreamMinKb = 4;
// Stream-K overhead in k-blocks: a fixed cost per segment (a worker runs up
// to two: storing its partial tile, the arrival, restarting the k loop) and a
// cost per partial tile the finishing worker reads.  Refitted after the
// partials were stored warp-coalesced (before: 0.67 per part): 256 x 256 x
// 8192, 128 x 256 x 8192, 256 x 512 x 4092 and 1024 x 1024 x 2048 on 152
// workers (39, 77, 20 and 4 parts per tile) ran in 53.4, 71, 40.2 and 81.4
// us, k-blocks of ~2.5 us: 0.25-0.4 per part beyond the k loop.
constexpr double kStreamSegmentKb = 2.0;
constexpr double kStreamPartKb = 0.27;

// Measured cost of the cluster fix-up per part, in k-blocks: 256^3 runs in
// 16.3, 12.4 and 10.8 us cut into 2, 4 and 8 parts (one k-block of a part
// there ~2.2 us, each part's share of the fix-up ~0.2 us).
constexpr double kClusterFixupKb = 0.15;

struct TailChoice {
  int split;        // equal parts per tail tile (1 = none)
  int sk_workers;   // > 0: stream-K instead
  double cost;      // in k-blocks of this tile width
};

// Cost, in k-blocks, of `tiles` 128-wide tiles cut into S parts that all run
// at once as clusters of S: the longest part plus the fix-up.
double cluster_cost(int num_kb, int S) {
  return static_cast<double>((num_kb + S - 1) / S) + kClusterFixupKb * S;
}

// The cheapest number of parts S (2..8, at most one per k-block) into which
// `tiles` 128-wide tiles can be cut so that all S x tiles CTAs run at once as
// clusters of S (see simt_use_cluster), or 1 if there is none.
int cluster_parts(int tiles, int num_kb, int num_sms) {
  int best = 1;
  for (int S = 2; S <= kSimtMaxCluster && S <= num_kb; ++S)
    if (static_cast<int64_t>(tiles) * S <= num_sms && tiles <= simt_max_clusters(S) &&
        (best == 1 || cluster_cost(num_kb, S) < cluster_cost(num_kb, best)))
      best = S;
  return best;
}

// Cost, in k-blocks, of the tail of `tail` tiles cut into S equal parts
// each, run R = ceil(tail S / workers) rounds deep.
double split_cost(int tail, int S, int num_kb, int workers) {
  const int R = (tail * S + workers - 1) / workers;
  if (S <= 1) return static_cast<double>(R) * num_kb;
  const double per_part = static_cast<double>(num_kb) / S;
  return R * (per_part + S * kSplitFixupKb);
}

// Stream-K tail over G workers: each runs ceil(W / G) k-blocks in up to two
// segments and, when it finishes a tile, reads up to ceil(G / tail) + 1
// partial tiles.
double stream_cost(int tail, int num_kb, int G) {
  const int64_t W = static_cast<int64_t>(tail) * num_kb;
  const int64_t per = (W + G - 1) / G;
  const int parts = (G + tail - 1) / tail + 1;
  return static_cast<double>(per) + 2 * kStreamSegmentKb + kStreamPartKb * parts;
}

// `cluster`: every tile is in the tail and the cluster fix-up is possible.
TailChoice choose_tail(int tail, int num_kb, int num_sms, const TileConfig* fixed, bool cluster) {
  TailChoice c{1, 0, 0.0};
  if (tail <= 0) return c;
  const int64_t W = static_cast<int64_t>(tail) * num_kb;
  const int pinned = fixed != nullptr ? fixed->split : 0;
  if (pinned == GEMM_SPLIT_STREAM) {
    c.sk_workers = static_cast<int>(W < num_sms ? W : num_sms);
    c.cost = stream_cost(tail, num_kb, c.sk_workers);
    return c;
  }
  if (pinned > 0) {
    c.split = pinned > num_kb ? num_kb : pinned;
    c.cost = split_cost(tail, c.split, num_kb, num_sms);
    return c;
  }
  c.split = tail_split(tail, num_kb, num_sms, kSplitFixupKb);
  c.cost = split_cost(tail, c.split, num_kb, num_sms);
  if (cluster) {
    const int S = cluster_parts(tail, num_kb, num_sms);
    const double cc = cluster_cost(num_kb, S);
    if (S > 1 && cc < c.cost) {
      c.split = S;
      c.cost = cc;
    }
  }
  int G = num_sms;
  if (W / G < kStreamMinKb) G = static_cast<int>(W / kStreamMinKb);
  if (G >= tail && G > 1) {
    const double sc = stream_cost(tail, num_kb, G);
    if (sc < c.cost) {
      c.split = 1;
      c.sk_workers = G;
      c.cost = sc;
    }
  }
  return c;
}

// Estimated time of the whole launch in 128 x 128 k-block units.
// `tma_operands`: both operands on TMA, which the cluster fix-up needs.
double plan_time(int M, int N, int num_kb, int num_sms, bool wide, const TileConfig* fixed,
                 bool tma_operands, TailChoice* tail_out, int* full_out) {
  const int bn = simt_bn(wide);
  const int tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
  const int tail = tiles >= num_sms ? tiles % num_sms : tiles;
  const int full = tiles - tail;
  const TailChoice t =
      choose_tail(tail, num_kb, num_sms, fixed, tma_operands && !wide && full == 0);
  *tail_out = t;
  *full_out = full;
  const double kb = (static_cast<double>(full) / num_sms) * num_kb + t.cost;
  return kb * (wide ? kWideKbCost : 1.0);
}

}  // namespace

SimtPlan simt_plan(int M, int N, int K, int num_sms, const TileConfig* fixed, bool allow_wide) {
  SimtPlan pl{};
  pl.group_m = (fixed != nullptr && fixed->group_m > 0) ? fixed->group_m : 8;
  pl.split = 1;
  if (M <= 0 || N <= 0 || K <= 0 || num_sms <= 0) {
    pl.grid = 1;
    return pl;
  }
  const int num_kb = (K + BK - 1) / BK;
  const int pinned_kernel = fixed != nullptr ? fixed->kernel : GEMM_KERNEL_AUTO;
  TailChoice tn{}, tw{};
  int full_n = 0, full_w = 0;
  const double time_n = plan_time(M, N, num_kb, num_sms, false, fixed, allow_wide, &tn, &full_n);
  bool wide = allow_wide && pinned_kernel == GEMM_KERNEL_WIDE;
  if (allow_wide && pinned_kernel == GEMM_KERNEL_AUTO) {
    const double time_w = plan_time(M, N, num_kb, num_sms, true, fixed, true, &tw, &full_w);
    wide = time_w < time_n;
  } else if (wide) {
    plan_time(M, N, num_kb, num_sms, true, fixed, true, &tw, &full_w);
  }
  const TailChoice& t = wide ? tw : tn;
  const int bn = simt_bn(wide);
  const int tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
  const int tail = tiles - (wide ? full_w : full_n);
  pl.wide = wide;
  pl.full_items = tiles;
  pl.grid = tiles < num_sms ? tiles : num_sms;
  if (tail == 0 || (t.split <= 1 && t.sk_workers == 0)) return pl;
  pl.full_items = tiles - tail;
  const int64_t tile_floats = static_cast<int64_t>(BM) * bn;
  if (t.sk_workers > 0) {
    pl.sk_workers = t.sk_workers;
    pl.grid = num_sms;
    pl.ws_floats = 2 * static_cast<int64_t>(t.sk_workers) * tile_floats;
  } else {
    pl.split = t.split;
    const int items = pl.full_items + tail * t.split;
    pl.grid = items < num_sms ? items : num_sms;
    pl.ws_floats = static_cast<int64_t>(tail) * t.split * tile_floats;
  }
  pl.counters = tail;
  return pl;
}

int simt_max_clusters(int S) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev][kSimtMaxCluster + 1];  // 0 = not yet known
  int dev = 0;
  if (S < 2 || S > kSimtMaxCluster || cudaGetDevice(&dev) != cudaSuccess || dev < 0 ||
      dev >= kMaxDev) {
    cudaGetLastError();
    return 0;
  }
  const int known = cache[dev][S].load(std::memory_order_relaxed);
  if (known != 0) return known;
  using T = SimtTraits<kLoadTma, kLoadTma>;
  constexpr size_t kSmem = smem_bytes<128>();
  auto kernel = simt_gemm_kernel<kLoadTma, kLoadTma, 128, true>;
  int n = 0;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmem)) == cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(S));
    cfg.blockDim = dim3(T::kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  if (n > 0) cache[dev][S].store(n, std::memory_order_relaxed);
  return n;
}

bool simt_use_cluster(SimtPlan& pl, int M, int N) {
  pl.cluster = 0;
  if (pl.wide || pl.sk_workers != 0 || pl.full_items != 0 || pl.split < 2 ||
      pl.split > kSimtMaxCluster)
    return false;
  const int tiles = ((M + BM - 1) / BM) * ((N + 127) / 128);
  if (pl.grid != tiles * pl.split || tiles > simt_max_clusters(pl.split)) return false;
  pl.cluster = pl.split;
  pl.ws_floats = 0;
  pl.counters = 0;
  return true;
}

int simt_plan_max_parts(const SimtPlan& pl, int M, int N, int K) {
  if (pl.sk_workers == 0) return pl.split;
  const int bn = simt_bn(pl.wide);
  const int tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
  const int tail = tiles - pl.full_items;
  const int64_t num_kb = (K + BK - 1) / BK;
  const int64_t W = static_cast<int64_t>(tail) * num_kb, G = pl.sk_workers;
  int most = 1;
  for (int64_t t = 0; t < tail; ++t) {
    const int64_t parts =
        sk_worker((t + 1) * num_kb - 1, W, G) - sk_worker(t * num_kb, W, G) + 1;
    if (parts > most) most = static_cast<int>(parts);
  }
  return most;
}

cudaError_t launch_simt(const SimtArgs& a, const SimtPlan& plan, LoadMode mode_a,
                        LoadMode mode_b, const CUtensorMap* tmA, const CUtensorMap* tmB,
                        cudaStream_t stream) {
  if (a.cluster > 1) {
    // Every CTA must have its one item and its cluster (each waits for the
    // others at the cluster barriers): see simt_use_cluster.
    const int tiles = ((a.M + BM - 1) / BM) * ((a.N + 127) / 128);
    if (plan.wide || mode_a != kLoadTma || mode_b != kLoadTma || a.cluster > kSimtMaxCluster ||
        a.full_items != 0 || a.sk_workers != 0 || a.split != a.cluster ||
        plan.grid != tiles * a.cluster)
      return cudaErrorInvalidValue;
    return launch_variant<kLoadTma, kLoadTma, 128, true>(a, plan.grid, tmA, tmB, stream);
  }
  // The planner picks the wide tile only when both operands are on TMA.
  if (plan.wide) {
    if (mode_a != kLoadTma || mode_b != kLoadTma) return cudaErrorInvalidValue;
    return launch_variant<kLoadTma, kLoadTma, 256>(a, plan.grid, tmA, tmB, stream);
  }
  return launch_width<128>(a, plan.grid, mode_a, mode_b, tmA, tmB, stream);
}

}  // namespace g12
