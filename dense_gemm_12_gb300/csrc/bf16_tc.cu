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
// Split overhead per part and round, in k-block times of the tensor core
// (~0.35 us each; see tail_split): storing a 128 KB partial per CTA, and for a
// tile's last part reading the others and writing the tile, measured at
// roughly 3 us per part.
constexpr double kTcFixupKb = 8.0;
constexpr int STAGES = 4;
constexpr int kStageBytesA = BM * BK * 2;            // 16 KB
constexpr int kStageBytesB = BK * BN * 2;            // 32 KB
constexpr int kBoxBytesB = BK * 64 * 2;              // one 64-column box, 8 KB
constexpr int kStageBytes = kStageBytesA + kStageBytesB;
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr uint32_t kTmemCols = 512;
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

// Output staging per epilogue warp: two 4 KB buffers of 32 rows x 32 fp32
// (the TMA output stage alternates between them; store_chunk uses the first).
constexpr int kEpiWarpStageBytes = 2 * 32 * 32 * 4;
constexpr int kEpiStageBytes = kEpiWarps * kEpiWarpStageBytes;
constexpr size_t kSmemBytes = 1024 + STAGES * kStageBytes + kEpiStageBytes + sizeof(TcSmemTail);
static_assert(kSmemBytes <= 227 * 1024, "single-CTA kernel shared memory");

// Grouped raster: items walk column by column through groups of group_m item
// rows, so neighbouring CTAs share A row panels and B column panels in L2.
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

// One work unit: item (tile or pair tile), its k-block range and, for a
// tail item cut along k, its tail index, its part index among the item's
// parts (k order), the item's number of parts and the unit's own workspace
// slot (tail = -1 for a whole item).  An empty unit (kb0 == kb1: a stream-K
// worker whose range lies inside one item has no second segment) is skipped
// by every role.
struct Unit {
  int item, kb0, kb1, tail, part, parts, slot;
};

// Units of the launch: the whole items, then either `split` parts of every
// tail item (unit full_items + t * split + q), or, with stream-K, two
// segment slots per worker (unit full_items + s * G + j is segment s of
// worker j; see sk_lo).  Workers walk units in strides of G, so worker j
// meets exactly its own segments.
__device__ __forceinline__ int num_units(const TcArgs& p, int num_items) {
  if (p.sk_workers > 0) return p.full_items + 2 * p.sk_workers;
  return p.full_items + (num_items - p.full_items) * p.split;
}

// Workspace slot of part q (k order) of tail item t.
__device__ __forceinline__ int part_slot(const TcArgs& p, int t, int q, int num_kb, int64_t W) {
  if (p.sk_workers == 0) return t * p.split + q;
  const int64_t G = p.sk_workers;
  const int64_t j = sk_worker(static_cast<int64_t>(t) * num_kb, W, G) + q;
  return static_cast<int>(2 * j + (sk_lo(j, W, G) < static_cast<int64_t>(t) * num_kb ? 1 : 0));
}

__device__ __forceinline__ Unit unit_of(const TcArgs& p, int u, int num_kb, int num_items) {
  Unit w;
  w.tail = -1;
  w.part = 0;
  w.parts = 1;
  w.slot = -1;
  if (u < p.full_items) {
    w.item = u;
    w.kb0 = 0;
    w.kb1 = num_kb;
    return w;
  }
  const int v = u - p.full_items;
  if (p.sk_workers == 0) {
    w.tail = v / p.split;
    w.part = v - w.tail * p.split;
    w.parts = p.split;
    w.slot = v;
    w.item = p.full_items + w.tail;
    w.kb0 = w.part * num_kb / p.split;
    w.kb1 = (w.part + 1) * num_kb / p.split;
    return w;
  }
  // Stream-K: the tail's W k-blocks, item after item, in contiguous ranges
  // [sk_lo(j), sk_lo(j + 1)) per worker j; a range touches one or two items.
  const int64_t G = p.sk_workers;
  const int s = v / p.sk_workers;
  const int64_t j = v - s * p.sk_workers;
  const int64_t W = static_cast<int64_t>(num_items - p.full_items) * num_kb;
  const int64_t lo = sk_lo(j, W, G), hi = sk_lo(j + 1, W, G);
  int64_t t = lo / num_kb;
  int64_t a = lo - t * num_kb, b = min(hi - t * num_kb, static_cast<int64_t>(num_kb));
  w.item = p.full_items;
  w.kb0 = w.kb1 = 0;
  if (s == 1) {
    if (hi <= (t + 1) * num_kb) return w;  // the range ends inside its first item
    ++t;
    a = 0;
    b = hi - t * num_kb;
  }
  if (a >= b) return w;
  const int64_t first = sk_worker(t * num_kb, W, G);
  const int64_t last = sk_worker((t + 1) * num_kb - 1, W, G);
  w.tail = static_cast<int>(t);
  w.item = p.full_items + w.tail;
  w.kb0 = static_cast<int>(a);
  w.kb1 = static_cast<int>(b);
  w.part = static_cast<int>(j - first);
  w.parts = static_cast<int>(last - first + 1);
  w.slot = static_cast<int>(2 * j + s);
  return w;
}

// One 32-column chunk of this warp's 32 accumulator rows through the output
// stage (see epilogue.cuh).  tcgen05.ld hands each thread one row (r), so a
// direct store would send each warp instruction to 32 rows in 16-byte pieces.
// The chunk is turned around in the warp's 4 KB of shared memory instead --
// 16-byte pieces XOR-swizzled by row, so that neither the row-wise writes nor
// the column-wise reads conflict on banks -- and then 8 lanes cover one row's
// 128 bytes: C, bias and residual loads and the stores of D move whole
// lines.  The fused inputs of all 8 passes are loaded before the first store
// (a load after a store to a possibly aliasing address could not be issued
// early).  All 32 lanes call this together.  row_base: the warp's first row.
//
// FUSED = false is the plain GEMM output (fp32 D = alpha * acc + beta * C, no
// bias, activation, residual, scaling or amax), compiled without the general
// stage: the general stage unrolled over a chunk is large enough that its
// instruction fetches, not its memory traffic, set the pace.
template <bool FUSED>
__device__ __forceinline__ void store_chunk(const TcArgs& p, float4* stg, int row_base, int col0,
                                            const uint32_t (&r)[32], float& amax_acc) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 8; ++q)
    stg[lane * 8 + (q ^ (lane & 7))] =
        make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                    __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
  __syncwarp();
  const Epilogue& e = p.epi;
  const int ch = lane & 7;              // this lane's 4 columns: col .. col + 3
  const int col = col0 + 4 * ch;
  const bool full = col + 3 < p.N;
  if (!FUSED) {
    float cold[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = row_base + i * 4 + (lane >> 3);
#pragma unroll
      for (int k = 0; k < 4; ++k) cold[i][k] = 0.0f;
      if (row < p.M && e.beta != 0.0f) {
        const float* c = e.C + static_cast<int64_t>(row) * e.ldc + col;
        if (full && e.c_vec4) {
          const float4 o = *reinterpret_cast<const float4*>(c);
          cold[i][0] = o.x; cold[i][1] = o.y; cold[i][2] = o.z; cold[i][3] = o.w;
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) cold[i][k] = col + k < p.N ? c[k] : 0.0f;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = i * 4 + (lane >> 3);
      const int row = row_base + rr;
      const float4 a = stg[rr * 8 + (ch ^ (rr & 7))];
      const float acc[4] = {a.x, a.y, a.z, a.w};
      float v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        v[k] = (e.beta != 0.0f) ? fmaf(e.alpha, acc[k], e.beta * cold[i][k]) : e.alpha * acc[k];
      if (row < p.M) {
        float* d = static_cast<float*>(e.D) + static_cast<int64_t>(row) * e.ldd + col;
        if (full && e.d_vec) {
          *reinterpret_cast<float4*>(d) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (col + k < p.N) d[k] = v[k];
        }
      }
    }
    __syncwarp();  // the next chunk rewrites the staging area
    return;
  }
  float bias[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  if (e.bias != nullptr) {
    if (full && e.bias_vec4) {
      const float4 b = *reinterpret_cast<const float4*>(e.bias + col);
      bias[0] = b.x; bias[1] = b.y; bias[2] = b.z; bias[3] = b.w;
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) bias[k] = col + k < p.N ? e.bias[col + k] : 0.0f;
    }
  }
  if (e.beta == 0.0f && e.R == nullptr) {
    // No per-row inputs to load ahead: one row at a time keeps the code of
    // the general stage (activation, conversions) to one copy.
#pragma unroll 1
    for (int i = 0; i < 8; ++i) {
      const int rr = i * 4 + (lane >> 3);
      const int row = row_base + rr;
      const float4 a = stg[rr * 8 + (ch ^ (rr & 7))];
      const float acc[4] = {a.x, a.y, a.z, a.w};
      float v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[k] = epi_value(e, acc[k], 0.0f, bias[k], 0.0f);
        if (row < p.M && col + k < p.N) epi_track(e, amax_acc, v[k]);
      }
      if (row < p.M) {
        if (full && e.d_vec) {
          epi_store4(e, row, col, v);
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (col + k < p.N) epi_store1(e, row, col + k, v[k]);
        }
      }
    }
    __syncwarp();  // the next chunk rewrites the staging area
    return;
  }
  float cold[8][4], res[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = row_base + i * 4 + (lane >> 3);
    const bool in = row < p.M;
#pragma unroll
    for (int k = 0; k < 4; ++k) cold[i][k] = res[i][k] = 0.0f;
    if (in && e.beta != 0.0f) {
      const float* c = e.C + static_cast<int64_t>(row) * e.ldc + col;
      if (full && e.c_vec4) {
        const float4 o = *reinterpret_cast<const float4*>(c);
        cold[i][0] = o.x; cold[i][1] = o.y; cold[i][2] = o.z; cold[i][3] = o.w;
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) cold[i][k] = col + k < p.N ? c[k] : 0.0f;
      }
    }
    if (in && e.R != nullptr) {
      const float* rr = e.R + static_cast<int64_t>(row) * e.ldr + col;
      if (full && e.r_vec4) {
        const float4 o = *reinterpret_cast<const float4*>(rr);
        res[i][0] = o.x; res[i][1] = o.y; res[i][2] = o.z; res[i][3] = o.w;
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) res[i][k] = col + k < p.N ? rr[k] : 0.0f;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int rr = i * 4 + (lane >> 3);
    const int row = row_base + rr;
    const float4 a = stg[rr * 8 + (ch ^ (rr & 7))];
    const float acc[4] = {a.x, a.y, a.z, a.w};
    float v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[k] = epi_value(e, acc[k], cold[i][k], bias[k], res[i][k]);
      if (row < p.M && col + k < p.N) epi_track(e, amax_acc, v[k]);
    }
    if (row < p.M) {
      if (full && e.d_vec) {
        epi_store4(e, row, col, v);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (col + k < p.N) epi_store1(e, row, col + k, v[k]);
      }
    }
  }
  __syncwarp();  // the next chunk rewrites the staging area
}

__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync %0, %1;" ::"n"(kEpiBarSync), "n"(kEpiThreads) : "memory");
}

// Plain output stage (fp32 D = alpha * acc; beta == 0, nothing fused) of one
// whole unit through TMA stores.  The warp's 32 rows leave in chunks of 32
// rows x 32 columns: scaled in registers, written to one of the warp's two
// 4 KB staging buffers (rows of 128 B whose 16-byte pieces are XOR-swizzled by
// row % 8, the tensor map's 128-byte swizzle, so the 32 lanes' stores fall in
// distinct banks) and stored by one TMA copy, which the tensor map clips at
// the matrix edges.  Lane 0 issues the copies; before a buffer is rewritten it
// waits until the copy issued from it two chunks earlier has read it.  The
// accumulator columns of the next chunk are read from TMEM while this chunk
// is staged.  Far fewer instructions per element than the store_chunk path,
// whose issue latency bounds the kernel on problems with a short k loop.
static_assert(kTcStoreBoxCols == 32 && kTcStoreBoxRows == 32 && kEpiWarpStageBytes == 2 * 4096,
              "TMA output stage: two 32 x 32 fp32 buffers per epilogue warp");

// Waits for this thread's TMEM loads; r is tied to the wait so that no use of
// the loaded registers is scheduled before it.
__device__ __forceinline__ void tc_wait_ld_into(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// One chunk: buffer `buf` (byte offset in the warp's staging), columns
// col0 .. col0 + 31 of rows row_base .. row_base + 31.
__device__ __forceinline__ void stage_chunk_tma(const CUtensorMap* tmD, const uint32_t (&r)[32],
                                                float alpha, uint32_t stg, uint32_t buf, int col0,
                                                int row_base) {
  const uint32_t lane = threadIdx.x & 31;
  if (lane == 0) bulk_wait_group_read<1>();
  __syncwarp();
  const uint32_t row_addr = stg + buf + lane * 128u;
#pragma unroll
  for (uint32_t q = 0; q < 8; ++q)
    st_shared_v4(row_addr + ((q ^ (lane & 7u)) << 4), alpha * __uint_as_float(r[4 * q]),
                 alpha * __uint_as_float(r[4 * q + 1]), alpha * __uint_as_float(r[4 * q + 2]),
                 alpha * __uint_as_float(r[4 * q + 3]));
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmD, stg + buf, col0, row_base);
    bulk_commit_group();
  }
}

// seq: chunks this warp has staged so far; the buffers alternate across units
// too, so the copy two chunks back always read the buffer being rewritten.
__device__ __forceinline__ void store_unit_tma(const TcArgs& p, const CUtensorMap* tmD,
                                               uint32_t taddr, uint32_t stg, int row_base,
                                               int col_base, uint32_t& seq) {
  if (row_base >= p.M) return;
  const float alpha = p.epi.alpha;
  // chunks holding at least one column < N (uniform over the warp)
  const int chunks = min(BN / 32, (p.N - col_base + 31) / 32);
  const uint32_t buf0 = (seq & 1u) * 4096u, buf1 = 4096u - buf0;
  seq += static_cast<uint32_t>(chunks);
  uint32_t ra[32], rb[32];
  tmem_ld_32x32b_x32(taddr, ra);
  tc_wait_ld_into(ra);
#pragma unroll 1
  for (int c = 0; c < chunks; c += 2) {
    const bool next = c + 1 < chunks;
    if (next) tmem_ld_32x32b_x32(taddr + (c + 1) * 32, rb);
    stage_chunk_tma(tmD, ra, alpha, stg, buf0, col_base + c * 32, row_base);
    if (!next) break;
    tc_wait_ld_into(rb);
    if (c + 2 < chunks) tmem_ld_32x32b_x32(taddr + (c + 2) * 32, ra);
    stage_chunk_tma(tmD, rb, alpha, stg, buf1, col_base + (c + 1) * 32, row_base);
    tc_wait_ld_into(ra);
  }
}

// Before the staging area is written by other code: every TMA store issued
// from it has read it.
__device__ __forceinline__ void staging_release(const TcArgs& p) {
  if (p.d_tma) {
    if ((threadIdx.x & 31) == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }
}

// Output stage of one work unit, run by the 4 epilogue warps of a CTA (thread
// et = TMEM lane et = row et of the CTA's 128-row tile).  taddr: this warp's
// lanes of the accumulator.  cpi / rank: CTAs per item (1, or 2 on pairs) and
// this CTA's rank in it; every CTA of an item keeps its own counter (tail
// index * cpi + rank) and its own partial sums (slot * cpi + rank).
//
// A part of a split item stores its partial sums (thread-major float4s,
// coalesced per warp), then counts its arrival; the last of the item's parts
// re-reads its own accumulator and adds all parts in k order -- a fixed
// order, so the result does not depend on which part finishes last -- and
// writes D.
template <bool FUSED>
__device__ __forceinline__ void epilogue_unit(const TcArgs& p, const CUtensorMap* tmD,
                                              uint32_t& tma_seq, const Unit& w, uint32_t taddr,
                                              float4* stg, int row_base, int tn, int cpi,
                                              int rank, int num_kb, int64_t W, int et,
                                              int* last_flag, float& amax_acc) {
  if (w.tail < 0) {
    if (!FUSED && p.d_tma) {
      store_unit_tma(p, tmD, taddr, smem_u32(stg), row_base, tn * BN, tma_seq);
      return;
    }
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(taddr + c * 32, r);
      tc_wait_ld();
      store_chunk<FUSED>(p, stg, row_base, tn * BN + c * 32, r, amax_acc);
    }
    return;
  }
  if (!FUSED) staging_release(p);
  float4* const ws4 = reinterpret_cast<float4*>(p.ws);
  auto part_base = [&](int slot) {
    return ws4 + (static_cast<int64_t>(slot) * cpi + rank) * (kPartFloats / 4);
  };
  {
    float4* mine = part_base(w.slot);
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
  const int counter = w.tail * cpi + rank;
  epi_bar();
  if (et == 0) {
    const uint32_t before = atomic_add_acq_rel_gpu(p.counters + counter, 1u);
    *last_flag = (before == static_cast<uint32_t>(w.parts - 1)) ? 1 : 0;
  }
  epi_bar();
  if (*reinterpret_cast<volatile int*>(last_flag)) {
    // Parts are added in k order; the other parts' partial sums are read
    // two parts per round trip (the loads of a pair are independent), and
    // this part's own accumulator comes from TMEM.
    const float4 zero4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      float sum[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) sum[i] = 0.0f;
      uint32_t r[32];
#pragma unroll 1
      for (int q0 = 0; q0 < w.parts; q0 += 2) {
        const bool has_b = q0 + 1 < w.parts;
        const bool load_a = q0 != w.part;
        const bool load_b = has_b && q0 + 1 != w.part;
        const float4* src_a =
            part_base(part_slot(p, w.tail, q0, num_kb, W)) + c * 8 * kEpiThreads + et;
        const float4* src_b =
            has_b ? part_base(part_slot(p, w.tail, q0 + 1, num_kb, W)) + c * 8 * kEpiThreads + et
                  : src_a;
        float4 va[8], vb[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          va[q] = load_a ? __ldcg(src_a + q * kEpiThreads) : zero4;
          vb[q] = load_b ? __ldcg(src_b + q * kEpiThreads) : zero4;
        }
        if (!load_a || (has_b && !load_b)) {  // this pair holds the own part
          tmem_ld_32x32b_x32(taddr + c * 32, r);
          tc_wait_ld();
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 a4 = load_a ? va[q] : make_float4(__uint_as_float(r[4 * q]),
              __uint_as_float(r[4 * q + 1]), __uint_as_float(r[4 * q + 2]),
              __uint_as_float(r[4 * q + 3]));
          sum[4 * q] += a4.x;
          sum[4 * q + 1] += a4.y;
          sum[4 * q + 2] += a4.z;
          sum[4 * q + 3] += a4.w;
        }
        if (has_b) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 b4 = load_b ? vb[q] : make_float4(__uint_as_float(r[4 * q]),
                __uint_as_float(r[4 * q + 1]), __uint_as_float(r[4 * q + 2]),
                __uint_as_float(r[4 * q + 3]));
            sum[4 * q] += b4.x;
            sum[4 * q + 1] += b4.y;
            sum[4 * q + 2] += b4.z;
            sum[4 * q + 3] += b4.w;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(sum[i]);
      store_chunk<FUSED>(p, stg, row_base, tn * BN + c * 32, r, amax_acc);
    }
    if (et == 0) p.counters[counter] = 0u;
  }
  epi_bar();  // last_flag is rewritten by the next split unit
}

// The cluster form's reduction: CTA `rank` of a cluster of S takes the
// 32-column chunks [rank * 8 / S, (rank + 1) * 8 / S) of the tile; for each,
// every epilogue thread adds its row's 32 values from the S CTAs' partial
// sums (stored in each CTA's shared memory at `part_u32` in the workspace
// layout) in rank (= k) order, starting from zero -- the order and the
// arithmetic of the workspace fix-up -- and runs the chunk through the output
// stage.  The 8 loads from one CTA are in flight together: S round trips per
// chunk.  The plain beta == 0 output leaves through the TMA output stage.
template <bool FUSED>
__device__ __forceinline__ void cluster_chunks(const TcArgs& p, const CUtensorMap* tmD,
                                               uint32_t part_u32, int S, int rank, float4* stg,
                                               int row_base, int tn, int et, float& amax_acc) {
  const int c0 = rank * (BN / 32) / S, c1 = (rank + 1) * (BN / 32) / S;
#pragma unroll 1
  for (int c = c0; c < c1; ++c) {
    float sum[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) sum[i] = 0.0f;
#pragma unroll 1
    for (int src = 0; src < S; ++src) {
      float4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        v[q] = ld_shared_cluster_v4(mapa_shared(
            part_u32 + static_cast<uint32_t>(((c * 8 + q) * kEpiThreads + et) * 16),
            static_cast<uint32_t>(src)));
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        sum[4 * q] += v[q].x;
        sum[4 * q + 1] += v[q].y;
        sum[4 * q + 2] += v[q].z;
        sum[4 * q + 3] += v[q].w;
      }
    }
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(sum[i]);
    if (!FUSED && p.d_tma) {
      const int col0 = tn * BN + c * 32;
      if (row_base < p.M && col0 < p.N)
        stage_chunk_tma(tmD, r, p.epi.alpha, smem_u32(stg), ((c - c0) & 1) * 4096u, col0,
                        row_base);
    } else {
      store_chunk<FUSED>(p, stg, row_base, tn * BN + c * 32, r, amax_acc);
    }
  }
  // The TMA stores are complete before the CTA leaves.
  if (!FUSED && p.d_tma) {
    if ((threadIdx.x & 31) == 0) bulk_wait_group_all();
    __syncwarp();
  }
}

// CLUSTER: one unit per CTA -- a k-part of a tile, full_items = 0, split =
// p.cluster -- and the parts of a tile form a cluster that adds its partial
// sums through distributed shared memory (cluster_chunks) instead of the
// workspace.  Every thread of the CTA reaches the two cluster barriers after
// its role, also after a bounded wait ran out, so none can hang there.
template <bool FUSED, bool CLUSTER>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bf16_kernel(const __grid_constant__ TcArgs p, const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem<1024>(smem_raw);
  uint8_t* epi_stage = smem + STAGES * kStageBytes;
  TcSmemTail* tail = reinterpret_cast<TcSmemTail*>(epi_stage + kEpiStageBytes);
  volatile int* abort_flag = &tail->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int num_kb = (p.K + BK - 1) / BK;
  const int num_items = tiles_m * tiles_n;
  const int units = num_units(p, num_items);
  const int64_t W = static_cast<int64_t>(num_items - p.full_items) * num_kb;  // stream-K tail

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
  // Launched with programmatic stream serialization: everything above touches
  // no global memory and may overlap the previous kernel's last CTAs; every
  // global access below follows its completion.
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  float amax_acc = 0.0f;
  bool parts_stored = false;  // CLUSTER: this CTA's partial sums are in shared memory

  if (warp == 0) {
    // -------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit w = unit_of(p, u, num_kb, num_items);
        int tm, tn;
        tile_coords(w.item, tiles_m, tiles_n, p.group_m, tm, tn);
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
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit w = unit_of(p, u, num_kb, num_items);
        if (w.kb0 == w.kb1) continue;
        const uint32_t ab = j & 1u, ar = j >> 1;
        ++j;
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
    float4* stg = reinterpret_cast<float4*>(epi_stage + quarter * kEpiWarpStageBytes);
    uint32_t tma_seq = 0;  // chunks staged by the TMA output stage (buffer parity)
    uint32_t j = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit w = unit_of(p, u, num_kb, num_items);
      if (w.kb0 == w.kb1) continue;
      int tm, tn;
      tile_coords(w.item, tiles_m, tiles_n, p.group_m, tm, tn);
      const uint32_t ab = j & 1u, ar = j >> 1;
      ++j;
      const bool ok = mbar_wait(&tail->tmem_full[ab], ar & 1u, abort_flag, p.err);
      // Leave together if a wait ran out anywhere (see named_bar_any).
      if (named_bar_any(kEpiBarAny, kEpiThreads, !ok)) break;
      tc_fence_after_sync();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + ab * BN;
      if (CLUSTER) {
        // The MMAs are done and this CTA has no further unit, so the ring
        // is free: the part's 128 x 256 partial sums go to its first 128 KB,
        // laid out as in the workspace (thread-major float4s).
        float4* part = reinterpret_cast<float4*>(smem);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c * 32, r);
          tc_wait_ld();
#pragma unroll
          for (int q = 0; q < 8; ++q)
            part[(c * 8 + q) * kEpiThreads + et] =
                make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                            __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
        }
        parts_stored = true;
      } else {
        epilogue_unit<FUSED>(p, &tmD, tma_seq, w, taddr, stg, tm * BM + quarter * 32, tn, 1, 0, num_kb,
                             W, et, &tail->last_flag, amax_acc);
      }
      tc_fence_before_sync();
      mbar_arrive(&tail->tmem_empty[ab]);
    }
    if (FUSED && !CLUSTER) epi_flush_amax(p.epi, amax_acc);
    // The TMA stores of the output stage are complete before the CTA leaves.
    if (!FUSED && p.d_tma) {
      if (lane == 0) bulk_wait_group_all();
      __syncwarp();
    }
  }

  if (CLUSTER) {
    __syncwarp();
    cluster_sync();  // every part's partial sums are in its shared memory
    // parts_stored is the same in all epilogue threads (they leave the loop
    // together); without it some part is missing and the error word is set.
    if (warp >= 2 && parts_stored) {
      const int quarter = warp & 3;
      int tm, tn;
      tile_coords(static_cast<int>(blockIdx.x) / p.cluster, tiles_m, tiles_n, p.group_m, tm, tn);
      cluster_chunks<FUSED>(p, &tmD, smem_u32(smem), p.cluster,
                            static_cast<int>(cluster_cta_rank()),
                            reinterpret_cast<float4*>(epi_stage + quarter * kEpiWarpStageBytes),
                            tm * BM + quarter * 32, tn, quarter * 32 + lane, amax_acc);
      if (FUSED) epi_flush_amax(p.epi, amax_acc);
    }
    __syncwarp();
    cluster_sync();  // no CTA leaves while another may still read its shared memory
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
constexpr int PBK = 128;                                 // k per stage (64 or 128)
static_assert(PBK == 64 || PBK == 128, "pair kernel k-block");
constexpr int PS = PBK == 64 ? 6 : 3;                    // stages of the ring
constexpr int kPairBN = BN / 2;                         // B columns held per CTA
constexpr int kABoxBytes = BM * 64 * 2;                 // one 64-wide swizzled A box, 16 KB
constexpr int kPairStageBytesA = BM * PBK * 2;          // PBK / 64 A boxes
constexpr int kPairBoxBytesB = PBK * 64 * 2;            // one 64-column B box of PBK rows
constexpr int kPairStageBytesB = PBK * kPairBN * 2;     // two B boxes
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

constexpr size_t kPairSmemBytes =
    1024 + PS * kPairStageBytes + kEpiStageBytes + sizeof(PairSmemTail);
static_assert(kPairSmemBytes <= 227 * 1024, "pair kernel shared memory");

template <bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bf16_pair_kernel(const __grid_constant__ TcArgs p, const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmD) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem<1024>(smem_raw);
  uint8_t* epi_stage = smem + PS * kPairStageBytes;
  PairSmemTail* tail = reinterpret_cast<PairSmemTail*>(epi_stage + kEpiStageBytes);
  volatile int* abort_flag = &tail->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles_m = (p.M + BM - 1) / BM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int pairs_m = (tiles_m + 1) / 2;
  const int num_items = pairs_m * tiles_n;
  const int units = num_units(p, num_items);
  const int num_kb = (p.K + PBK - 1) / PBK;
  const int64_t W = static_cast<int64_t>(num_items - p.full_items) * num_kb;  // stream-K tail
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
  // Launched with programmatic stream serialization: everything above touches
  // no global memory and may overlap the previous kernel's last CTAs; every
  // global access below follows its completion.
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();

  if (warp == 0) {
    // -------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint32_t full0 = mapa_shared(smem_u32(&tail->full[0]), 0);
      uint32_t it = 0;
      bool ok = true;
      for (int u = first_item; u < units && ok; u += item_stride) {
        const Unit w = unit_of(p, u, num_kb, num_items);
        int pm, tn;
        tile_coords(w.item, pairs_m, tiles_n, p.group_m, pm, tn);
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
#pragma unroll
          for (int q = 0; q < PBK / 64; ++q)
            tma_load_2d_pair(sa + q * kABoxBytes, &tmA, kb * PBK + q * 64, tm * BM, full);
#pragma unroll
          for (int j = 0; j < kPairBN / 64; ++j)
            tma_load_2d_pair(sb + j * kPairBoxBytesB, &tmB,
                             tn * BN + static_cast<int>(rank) * kPairBN + j * 64, kb * PBK, full);
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
      for (int u = first_item; u < units && ok; u += item_stride) {
        const Unit w = unit_of(p, u, num_kb, num_items);
        if (w.kb0 == w.kb1) continue;
        const uint32_t ab = j & 1u, ar = j >> 1;
        ++j;
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
          for (int kk = 0; kk < PBK / 16; ++kk) {
            // A: K-major, 64-wide boxes 16 KB apart; B: MN-major, 64-column
            // boxes of PBK rows, a K step of 16 rows is 2048 B.
            const uint64_t adesc =
                smem_desc_sw128(sa + (kk / 4) * kABoxBytes + (kk % 4) * 32, 16, 1024);
            const uint64_t bdesc = smem_desc_sw128(sb + kk * 2048, kPairBoxBytesB, 1024);
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
    float4* stg = reinterpret_cast<float4*>(epi_stage + quarter * kEpiWarpStageBytes);
    float amax_acc = 0.0f;
    const uint32_t tmem_empty0 = mapa_shared(smem_u32(&tail->tmem_empty[0]), 0);
    uint32_t tma_seq = 0;  // chunks staged by the TMA output stage (buffer parity)
    uint32_t j = 0;
    for (int u = first_item; u < units; u += item_stride) {
      const Unit w = unit_of(p, u, num_kb, num_items);
      if (w.kb0 == w.kb1) continue;
      int pm, tn;
      tile_coords(w.item, pairs_m, tiles_n, p.group_m, pm, tn);
      const int tm = pm * 2 + static_cast<int>(rank);
      const uint32_t ab = j & 1u, ar = j >> 1;
      ++j;
      const bool ok = mbar_wait(&tail->tmem_full[ab], ar & 1u, abort_flag, p.err);
      if (named_bar_any(kEpiBarAny, kEpiThreads, !ok)) break;
      tc_fence_after_sync();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + ab * BN;
      // each CTA of the pair owns the counter and partials of its 128 rows
      epilogue_unit<FUSED>(p, &tmD, tma_seq, w, taddr, stg, tm * BM + quarter * 32, tn, 2,
                           static_cast<int>(rank), num_kb, W, et, &tail->last_flag, amax_acc);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tmem_empty0 + ab * static_cast<uint32_t>(sizeof(uint64_t)));
    }
    if (FUSED) epi_flush_amax(p.epi, amax_acc);
    // The TMA stores of the output stage are complete before the CTA leaves.
    if (!FUSED && p.d_tma) {
      if (lane == 0) bulk_wait_group_all();
      __syncwarp();
    }
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
  auto kernel = tc_bf16_pair_kernel<false>;
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

// Clusters of S single-CTA kernels (cluster form) that can be resident at
// once on the current device (one CTA per SM; a cluster must fit in one GPC).
// Queried once per device, size and instance.
static int single_max_clusters(int S, bool fused) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev][9][2];  // 0 = not yet known
  int dev = 0;
  if (S < 2 || S > 8 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return 0;
  }
  const int known = cache[dev][S][fused ? 1 : 0].load(std::memory_order_relaxed);
  if (known != 0) return known;
  auto kernel = fused ? tc_bf16_kernel<true, true> : tc_bf16_kernel<false, true>;
  int n = 0;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes)) == cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(S));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
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
  if (n > 0) cache[dev][S][fused ? 1 : 0].store(n, std::memory_order_relaxed);
  return n;
}

int tc_b_box_rows(bool pair) { return pair ? PBK : BK; }

// Whether an output stage needs the general (fused) kernel instance.
bool tc_fused(const Epilogue& ep) {
  return ep.bias != nullptr || ep.act != kActNone || ep.R != nullptr || ep.d_type != kOutF32 ||
         ep.d_scale != 1.0f || ep.amax != nullptr;
}

bool tc_use_cluster(TcPlan& pl, int M, int N, const Epilogue& epi) {
  const bool fused = tc_fused(epi);
  pl.cluster = 0;
  if (pl.pair || pl.sk_workers != 0 || pl.full_items != 0 || pl.split < 2 || pl.split > 8)
    return false;
  const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  if (pl.grid != tiles * pl.split || tiles > single_max_clusters(pl.split, fused)) return false;
  pl.cluster = pl.split;
  pl.ws_floats = 0;
  pl.counters = 0;
  return true;
}

// Whether automatic dispatch takes the CTA-pair kernel: on large problems
// only -- at least 128 single-CTA tiles with K > 2048, or 256 with K > 512.
// The launch-configuration sweep over M, N, K = 256 .. 8192 found the pair
// kernel fastest there (by up to 15 % at K = 1024, since the output stage
// writes through TMA) and the single-CTA kernel everywhere else (short k
// loops fill the pair kernel's 128-deep ring slowly, and few tiles leave SMs
// idle).
static bool tc_prefer_pair(int tiles, int K) {
  return (K > 2048 && tiles >= 128) || (K > 512 && tiles >= 256);
}

// Cost, in k-blocks, of cutting each single-CTA tile into S > 1 parts that
// all run at once as clusters: the longest part plus the cluster fix-up --
// the partial sums copied out of TMEM, two cluster barriers, the reduction
// and the reduced tile's output stage.  Fitted on the launch-configuration
// sweep's one-round classes: with the TMA output stage, whose whole tiles
// leave quickly, ~9.5 k-blocks plus ~2.75 per part (at K = 512 and 1024 a
// split of 2 or 4 lost 10-27 % to whole tiles; at K = 4096, 4 parts won);
// with the staged output stage, ~1 k-block per part.
constexpr double kTcClusterFixedKb = 9.5, kTcClusterPartKb = 2.75;
constexpr double kTcClusterPartKbStaged = 1.0;

TcPlan tc_plan(int M, int N, int K, int num_sms, const TileConfig* fixed, bool tma_out) {
  TcPlan pl{};
  const int tiles_m = (M + BM - 1) / BM;
  const int tiles_n = (N + BN - 1) / BN;
  const bool pinned = fixed != nullptr && fixed->kernel != GEMM_KERNEL_AUTO;
  pl.pair = pinned ? fixed->kernel == GEMM_KERNEL_CTA_PAIR
                   : (tiles_m >= 2 && tc_prefer_pair(tiles_m * tiles_n, K));
  const int kblock = pl.pair ? PBK : BK;
  const int num_kb = (K + kblock - 1) / kblock;
  pl.group_m = (fixed != nullptr && fixed->group_m > 0) ? fixed->group_m : 8;
  const int ctas_per_item = pl.pair ? 2 : 1;
  const int items = pl.pair ? ((tiles_m + 1) / 2) * tiles_n : tiles_m * tiles_n;
  const int workers = pl.pair ? pair_max_clusters(num_sms) : num_sms;
  const int tail_items = items >= workers ? items % workers : items;
  // Stream-K (pinned, or chosen by the dispatch table): the tail items'
  // k-blocks dealt out to all workers, at least one each (with fewer k-blocks
  // than workers the equal split below is used instead).
  if (fixed != nullptr && fixed->split == GEMM_SPLIT_STREAM && tail_items > 0 &&
      static_cast<int64_t>(tail_items) * num_kb >= workers) {
    pl.split = 1;
    pl.sk_workers = workers;
    pl.full_items = items - tail_items;
    pl.grid = ctas_per_item * workers;
    pl.ws_floats = 2 * static_cast<int64_t>(workers) * ctas_per_item * kPartFloats;
    pl.counters = static_cast<int64_t>(tail_items) * ctas_per_item;
    return pl;
  }
  // a pinned split is capped at one k-block per part
  pl.split = (fixed != nullptr && fixed->split > 0)
                 ? (fixed->split < num_kb ? fixed->split : num_kb)
                 : tail_split(items, num_kb, workers, kTcFixupKb * BK / kblock);
  if (!pl.pair && items < workers && (fixed == nullptr || fixed->split == 0)) {
    // Every tile in one round: the cluster split (see tc_use_cluster) costs
    // far less than the workspace's, so take the cheapest S whose clusters
    // can all be resident, or none.
    int best = 1;
    double best_cost = num_kb;
    for (int S = 2; S <= 8 && S <= num_kb; ++S) {
      if (static_cast<int64_t>(items) * S > workers || items > single_max_clusters(S, false))
        continue;
      const double cost = static_cast<double>((num_kb + S - 1) / S) +
                          (tma_out ? kTcClusterFixedKb + kTcClusterPartKb * S
                                   : kTcClusterPartKbStaged * S);
      if (cost < best_cost - 1e-9) {
        best = S;
        best_cost = cost;
      }
    }
    pl.split = best;
  }
  if (pl.split < 1) pl.split = 1;
  if (tail_items == 0) pl.split = 1;
  const int tail = pl.split > 1 ? tail_items : 0;
  pl.full_items = items - tail;
  const int units = pl.full_items + tail * pl.split;
  pl.grid = ctas_per_item * (units < workers ? units : workers);
  pl.ws_floats = static_cast<int64_t>(tail) * pl.split * ctas_per_item * kPartFloats;
  pl.counters = static_cast<int64_t>(tail) * ctas_per_item;
  return pl;
}

int tc_plan_max_parts(const TcPlan& pl, int M, int N, int K) {
  if (pl.sk_workers == 0) return pl.split;
  const int tiles_m = (M + BM - 1) / BM;
  const int tiles_n = (N + BN - 1) / BN;
  const int items = pl.pair ? ((tiles_m + 1) / 2) * tiles_n : tiles_m * tiles_n;
  const int64_t num_kb = (K + (pl.pair ? PBK : BK) - 1) / (pl.pair ? PBK : BK);
  const int64_t tail = items - pl.full_items;
  const int64_t W = tail * num_kb, G = pl.sk_workers;
  int most = 1;
  for (int64_t t = 0; t < tail; ++t) {
    const int64_t parts = sk_worker((t + 1) * num_kb - 1, W, G) - sk_worker(t * num_kb, W, G) + 1;
    if (parts > most) most = static_cast<int>(parts);
  }
  return most;
}

cudaError_t launch_tc_bf16(const TcArgs& a, const TcPlan& plan, const CUtensorMap* tmA,
                           const CUtensorMap* tmB, const CUtensorMap* tmD, cudaStream_t stream) {
  // tmD is read only when a.d_tma is set; any valid map stands in otherwise.
  if (tmD == nullptr) {
    if (a.d_tma) return cudaErrorInvalidValue;
    tmD = tmB;
  }
  if (plan.grid < 1) return cudaSuccess;
  const bool fused = tc_fused(a.epi);
  if (plan.pair) {
    auto kernel = fused ? tc_bf16_pair_kernel<true> : tc_bf16_pair_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kPairSmemBytes));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kPairSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kernel, a, *tmA, *tmB, *tmD);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  const bool cluster = a.cluster > 1;
  if (cluster) {
    // Every CTA must have its one unit and its cluster (each waits for the
    // others at the cluster barriers): see tc_use_cluster.
    const int tiles = ((a.M + BM - 1) / BM) * ((a.N + BN - 1) / BN);
    if (a.cluster > 8 || a.full_items != 0 || a.sk_workers != 0 || a.split != a.cluster ||
        plan.grid != tiles * a.cluster)
      return cudaErrorInvalidValue;
  }
  auto kernel = cluster ? (fused ? tc_bf16_kernel<true, true> : tc_bf16_kernel<false, true>)
                        : (fused ? tc_bf16_kernel<true, false> : tc_bf16_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster ? static_cast<unsigned>(a.cluster) : 1u;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = cluster ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, kernel, a, *tmA, *tmB, *tmD);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace g12
