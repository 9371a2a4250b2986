// bf16_decode.cu -- decode-shaped GEMM (small M, up to 128): C = alpha * A * B +
// beta * C with bf16 A (M x K) and B (K x N), fp32 accumulation and fp32 C.
//
// "Tiled matrix multiplication" ("Avoid when") notes that a decode GEMV with
// M <= 16 is bound by memory bandwidth: the whole cost is streaming B once
// (and so it stays for a few times that M).  With M = 16 no tile of C is big
// enough to fill the machine, so the k range
// is split across CTAs and the partial sums are reduced afterwards ("Split-K"
// in the same page's "Variants and alternatives"; "A GEMM Kernel, Step by
// Step", "What is left").  On sm_103a the tensor core's smallest M is 128, so
// the product is computed transposed, D^T = B^T A^T: the MMA's M runs over
// 128 columns of C and its N over the rows of A: the kernel has instances
// for N = 16, 32 and 64 (a launch with M rows takes the smallest that holds
// them), and no row of the MMA's M is padding.  M > 64 runs as row blocks of
// 64 rows (the grid's y dimension, see row_block), each streaming B for its
// own rows at the same time.
//
// Work split.  B is cut into n-groups of 128 columns; a unit is one n-group x
// 128 values of k (32 KB of B, fetched as two 64 x 128 TMA boxes).  With at
// least ~60 % as many n-groups as SMs (N = 12288 gives 96) every CTA streams
// whole n-groups: no k range is split and nothing is exchanged.  With fewer
// n-groups, clusters of S CTAs (S a power of two up to 8, groups x S <= SMs)
// split each n-group's k range into S equal runs (split-K); the S partial
// sums are exchanged through distributed shared memory and each CTA adds the
// S values of its 128 / S columns in rank order, which is k order
// (cluster_reduce_store).  With more n-groups than SMs, units are numbered
// n-group-major and every CTA takes one contiguous, equal-sized run of them,
// cut into segments at n-group boundaries.
// A segment that spans the whole k range of its n-group writes C directly;
// otherwise the CTA holding the group's first k-piece combines: it waits a
// short, bounded time for the other contributors' partial sums (published in
// the workspace, announced on the group's arrival counter) and preloads them
// while its own MMAs drain; the others publish and never wait.  If the bound
// runs out the combiner publishes too and whichever CTA arrives last adds the
// partials.  Partials are always added in k order, so results are
// deterministic, and the combiner resets the counter for the next launch.
//
// Roles: warp 0 TMA producer (B boxes and two BMr x 64 K-major boxes of A per
// stage), warps 1 and 6 issue the MMAs (128 x BMr x 16, alternate stages,
// one accumulator each, double-buffered; warp 1 owns TMEM), warps 2..5 read
// the accumulators, combine and write C.  The launch uses programmatic
// dependent launch: the next kernel in the stream may set up while this one
// drains, and every global access follows grid_dependency_wait().
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace g12 {
namespace {

constexpr int BN = kDecBN;                 // MMA M: 128 columns of C per MMA tile
constexpr int NSUB = 1;                    // MMA tiles per n-group
constexpr int NW = NSUB * BN;              // columns of C per n-group
constexpr int kBoxesPerTile = BN / 64;     // 64-column TMA boxes per MMA tile
// Accumulator rows held by each epilogue warp (one 32-lane TMEM quarter each).
constexpr int kRowsPerQuarter = 32;
constexpr int BK = 128;                    // k per stage (one unit)
static_assert(BK == 64 || BK == 128, "k per stage must be 64 or 128");
constexpr int kABoxes = BK / 64;           // BMr x 64 boxes of A per stage
constexpr int kBoxBytesB = BK * 64 * 2;                   // one 64-column box of B
constexpr int kStageBytesB = NSUB * kBoxesPerTile * kBoxBytesB;
// Rows of C the output stage handles at a time (one 32x32b.x16 TMEM load).
constexpr int kChunk = 16;
// Shared memory the stage ring of one CTA may use.
constexpr int kRingSmemKb = 220;
// How long the combining CTA of a column group polls for the other
// contributors' partial sums before it falls back to publishing its own.
constexpr uint64_t kHandoffWaitNs = 20000;
// Units of B each CTA asks L2 to fetch before it waits for the previous
// kernel in the stream (measured on back-to-back launches at N = 12288:
// 0 units 17.92 us, 2 17.75, 4 17.68, 6 17.65, 8 17.77 -- more delays the
// CTA's own first TMA loads).
constexpr int kEarlyUnits = 4;
// Threads issuing tcgen05.mma, each in its own warp and taking every
// kIssuers-th stage into its own accumulator: with N = 16 the issue cost of
// an MMA, not the tensor core, bounds how fast one thread can consume B.
constexpr int kIssuers = 2;
static_assert(kIssuers == 1 || kIssuers == 2, "one or two MMA issuers");
constexpr int kThreads = 192 + (kIssuers - 1) * 32;
constexpr int kEpiThreads = 128;
constexpr int kSecondIssuerWarp = 6;
// Shape of one instance of the kernel: BMR rows of A and C (the MMA's N:
// 16, 32 or 64; a launch with M rows uses the smallest BMR >= M).
template <int BMR>
struct DecCfg {
  static_assert(BMR == 16 || BMR == 32 || BMR == 64, "rows of a decode launch");
  static constexpr int kChunks = BMR / kChunk;
  static constexpr int kStageBytesA = BMR * BK * 2;                  // 4, 8 or 16 KB
  static constexpr int kStageBytes = kStageBytesB + kStageBytesA;    // multiple of 1024
  static constexpr int kStageBudget = (kRingSmemKb * 1024) / kStageBytes;
  // Stages are a multiple of the issuer count, so that every stage is always
  // consumed by the same issuer.  An issuer then waits for the rounds of its
  // stages strictly in order; if two issuers alternated on one stage, one
  // could wait for round r+1 before round r completed, which a parity wait
  // cannot tell apart.
  static constexpr int STAGES = ((kStageBudget > 20 ? 20 : kStageBudget) / kIssuers) * kIssuers;
  static_assert(STAGES >= kIssuers && STAGES % kIssuers == 0, "stages per issuer");
  static constexpr uint32_t kIssuerCols = NSUB * BMR;           // TMEM columns per issuer
  static constexpr uint32_t kAccCols = kIssuers * kIssuerCols;  // TMEM columns per segment
  static constexpr uint32_t kTmemCols = 2 * kAccCols < 32 ? 32 : 2 * kAccCols;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(BN, BMR, /*A MN-major*/ 1, /*B MN-major*/ 0);
  static constexpr int kPartialFloats = BMR * NW;
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert((kTmemCols & (kTmemCols - 1)) == 0, "TMEM allocation must be a power of 2");
  static_assert(kPartialFloats * 4 <= kStageBytes, "a cluster's partial sums fit in stage 0");

  struct __align__(8) Tail {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain[2];
    uint32_t tmem_base;
    int abort_flag;
    int last_flag;
    int others_ready;  // set once every other contributor of the segment's group has published
  };
  static constexpr size_t kSmemBytes = 1024 + STAGES * kStageBytes + sizeof(Tail);
};

struct Split {
  int64_t units;       // n_groups * kb_total
  int kb_total;        // k-blocks per n-group
  int grid;            // CTAs
  int segs_max;        // segment slots per CTA in the workspace
};

__host__ __device__ inline Split make_split(int N, int K, int grid) {
  Split s;
  const int n_groups = (N + NW - 1) / NW;
  s.kb_total = (K + BK - 1) / BK;
  s.units = static_cast<int64_t>(n_groups) * s.kb_total;
  s.grid = grid;
  const int64_t per_cta = (s.units + grid - 1) / grid;
  s.segs_max = static_cast<int>((per_cta + s.kb_total - 1) / s.kb_total) + 1;
  return s;
}

__host__ __device__ inline int64_t run_start(const Split& s, int64_t c) {
  return (c * s.units) / s.grid;
}

// The CTA whose run contains unit u: the largest c with run_start(c) <= u.
__device__ __forceinline__ int64_t run_owner(const Split& s, int64_t u) {
  return ((u + 1) * s.grid + s.units - 1) / s.units - 1;
}

__device__ __forceinline__ void named_bar_epi() {
  asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");
}

// Old values of rows m0 .. m0 + kChunk - 1 of column n of C (rows < M; the
// first chunk is loaded ahead of time so that its final write costs no read
// round trip).
__device__ __forceinline__ void load_c_column(const DecodeArgs& p, int n, int m0,
                                              float (&old)[kChunk]) {
  const Epilogue& e = p.epi;
  const float* c = e.C + n;
#pragma unroll
  for (int i = 0; i < kChunk; ++i) {
    const int m = m0 + i;
    old[i] = (e.beta != 0.0f && n < p.N && m < p.M) ? c[static_cast<int64_t>(m) * e.ldc] : 0.0f;
  }
}

// Residual values of the same rows of column n, loaded like old C values.
__device__ __forceinline__ void load_r_column(const DecodeArgs& p, int n, int m0,
                                              float (&res)[kChunk]) {
  const Epilogue& e = p.epi;
#pragma unroll
  for (int i = 0; i < kChunk; ++i) {
    const int m = m0 + i;
    res[i] = (e.R != nullptr && n < p.N && m < p.M) ? e.R[static_cast<int64_t>(m) * e.ldr + n]
                                                     : 0.0f;
  }
}

// Column n of this thread through the output stage (see epilogue.cuh).
// FUSED = false is the plain GEMM output (fp32 D = C, no bias, no
// activation, no residual, d_scale 1, no amax), compiled without the general
// stage.
template <bool FUSED>
__device__ __forceinline__ void store_c_column(const DecodeArgs& p, int n, int m0,
                                               const float (&v)[kChunk],
                                               const float (&old)[kChunk],
                                               const float (&res)[kChunk], float& amax_acc) {
  if (n >= p.N) return;
  const Epilogue& e = p.epi;
  if (!FUSED) {
    // plain GEMM: D is C itself (fp32, ldd == ldc)
    float* d = static_cast<float*>(e.D) + n;
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      const int m = m0 + i;
      if (m < p.M)
        d[static_cast<int64_t>(m) * e.ldc] =
            (e.beta != 0.0f) ? fmaf(e.alpha, v[i], e.beta * old[i]) : e.alpha * v[i];
    }
    return;
  }
  const float bias = epi_bias(e, n);  // one column: one bias value, loaded before any store
#pragma unroll
  for (int i = 0; i < kChunk; ++i) {
    const int m = m0 + i;
    if (m < p.M) {
      const float val = epi_value(e, v[i], old[i], bias, res[i]);
      epi_track(e, amax_acc, val);
      epi_store1(e, m, n, val);
    }
  }
}

// Cluster split (p.cluster = S > 1): the S CTAs of a cluster hold the partial
// sums of one column group over S consecutive k ranges (rank order = k
// order), each as a BMR x NW fp32 array at shared address `part` (same offset
// in every CTA).  CTA `rank` writes columns [rank NW / S, (rank + 1) NW / S)
// of the group: epilogue thread ept takes one of them and BMR / S of its rows,
// reads the S partial sums of each element from the cluster's shared memory,
// adds them in rank order (a fixed order: results do not depend on timing)
// and runs the output stage.  Called by the 128 epilogue threads between two
// cluster barriers.
template <bool FUSED, int BMR, int S>
__device__ __forceinline__ void cluster_reduce_store_s(const DecodeArgs& p, uint32_t part,
                                                       int ept) {
  constexpr int slice = NW / S;                    // columns written by this CTA
  constexpr int rows = BMR * slice / kEpiThreads;  // rows per thread: BMR / S
  static_assert(rows >= 1 && rows * S == BMR, "rows per thread");
  const int rank = static_cast<int>(cluster_cta_rank());
  const int ng = static_cast<int>(blockIdx.x) / S;
  const int col = rank * slice + ept % slice;
  const int m0 = (ept / slice) * rows;
  const int n = ng * NW + col;
  const Epilogue& e = p.epi;
  float amax_acc = 0.0f;
  if (n < p.N) {
    // Every load is issued before any sum: the S x rows partial sums of this
    // thread's elements from the cluster's shared memory, and the old C and
    // residual values (one round trip in all, not one per element).
    float val[S][rows], old[rows], res[rows];
    const uint32_t a0 = part + static_cast<uint32_t>((m0 * NW + col) * 4);
#pragma unroll
    for (int q = 0; q < S; ++q) {
      const uint32_t aq = mapa_shared(a0, static_cast<uint32_t>(q));
#pragma unroll
      for (int i = 0; i < rows; ++i) val[q][i] = ld_shared_cluster_f32(aq + i * NW * 4);
    }
#pragma unroll
    for (int i = 0; i < rows; ++i) {
      const int m = m0 + i;
      old[i] = (e.beta != 0.0f && m < p.M) ? e.C[static_cast<int64_t>(m) * e.ldc + n] : 0.0f;
      res[i] = (FUSED && m < p.M) ? epi_residual(e, m, n) : 0.0f;
    }
    const float bias = FUSED ? epi_bias(e, n) : 0.0f;
#pragma unroll
    for (int i = 0; i < rows; ++i) {
      const int m = m0 + i;
      float v = val[0][i];
#pragma unroll
      for (int q = 1; q < S; ++q) v += val[q][i];  // rank order = k order
      if (m < p.M) {
        if (!FUSED) {
          // plain GEMM: D is C itself (fp32, ldd == ldc)
          static_cast<float*>(e.D)[static_cast<int64_t>(m) * e.ldc + n] =
              (e.beta != 0.0f) ? fmaf(e.alpha, v, e.beta * old[i]) : e.alpha * v;
        } else {
          const float out = epi_value(e, v, old[i], bias, res[i]);
          epi_track(e, amax_acc, out);
          epi_store1(e, m, n, out);
        }
      }
    }
  }
  if (FUSED) epi_flush_amax(e, amax_acc);
}

template <bool FUSED, int BMR>
__device__ __forceinline__ void cluster_reduce_store(const DecodeArgs& p, uint32_t part, int ept) {
  if (p.cluster == 2)
    cluster_reduce_store_s<FUSED, BMR, 2>(p, part, ept);
  else if (p.cluster == 4)
    cluster_reduce_store_s<FUSED, BMR, 4>(p, part, ept);
  else
    cluster_reduce_store_s<FUSED, BMR, 8>(p, part, ept);
}

// The arguments row block rb of a launch sees: rows [rb * BMR, rb * BMR + BMR)
// of the product, C, D and the residual (M counts only those rows), and its
// own arrival counters (n_groups per block) and workspace (ws_floats per
// block).  Row block 0 sees the launch's own arguments.
template <int BMR>
__device__ __forceinline__ DecodeArgs row_block(const DecodeArgs& a, int rb, int n_groups,
                                                int64_t ws_floats) {
  DecodeArgs p = a;
  const int64_t m0 = static_cast<int64_t>(rb) * BMR;
  const int64_t rows = static_cast<int64_t>(a.M) - m0;
  p.M = static_cast<int>(rows < BMR ? rows : BMR);
  const Epilogue& e = a.epi;
  const int d_bytes = e.d_type == kOutF32 ? 4 : (e.d_type == kOutBf16 ? 2 : 1);
  if (e.C != nullptr) p.epi.C = e.C + m0 * e.ldc;
  p.epi.D = static_cast<uint8_t*>(e.D) + m0 * e.ldd * d_bytes;
  if (e.R != nullptr) p.epi.R = e.R + m0 * e.ldr;
  if (a.counters != nullptr) p.counters = a.counters + static_cast<int64_t>(rb) * n_groups;
  if (a.workspace != nullptr) p.workspace = a.workspace + rb * ws_floats;
  return p;
}

template <bool FUSED, int BMR>
__global__ void __launch_bounds__(kThreads, 1)
    tc_decode_kernel(const __grid_constant__ DecodeArgs pa, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB) {
  using Cfg = DecCfg<BMR>;
  constexpr int BMr = BMR;
  constexpr int STAGES = Cfg::STAGES;
  constexpr int kStageBytes = Cfg::kStageBytes;
  constexpr uint32_t kIssuerCols = Cfg::kIssuerCols;
  constexpr uint32_t kAccCols = Cfg::kAccCols;
  constexpr uint32_t kTmemCols = Cfg::kTmemCols;
  constexpr uint32_t kIdesc = Cfg::kIdesc;
  constexpr int kPartialFloats = Cfg::kPartialFloats;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = align_smem<1024>(smem_raw);
  auto* tail = reinterpret_cast<typename Cfg::Tail*>(smem + STAGES * kStageBytes);
  volatile int* abort_flag = &tail->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Split sp = make_split(pa.N, pa.K, gridDim.x);
  // This CTA's row block (blockIdx.y; one unless M exceeds the instance's rows).
  const int row0 = static_cast<int>(blockIdx.y) * BMr;
  const DecodeArgs p = row_block<BMR>(pa, static_cast<int>(blockIdx.y), (pa.N + NW - 1) / NW,
                                      static_cast<int64_t>(gridDim.x) * sp.segs_max *
                                          kPartialFloats);
  const int64_t u_begin = run_start(sp, blockIdx.x);
  const int64_t u_end = run_start(sp, static_cast<int64_t>(blockIdx.x) + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&tail->full[s], 1);
      mbar_init(&tail->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tail->tmem_full[b], kIssuers);
      mbar_init(&tail->tmem_empty[b], kEpiThreads);
    }
    for (int q = 0; q < 2; ++q) mbar_init(&tail->drain[q], 1);
    tail->abort_flag = 0;
    tail->last_flag = 0;
    tail->others_ready = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&tail->tmem_base, kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  // Under programmatic dependent launch this prologue may run while the
  // previous kernel in the stream is still finishing.  Before waiting for it,
  // ask L2 for the first tiles of B this CTA will stream: an L2 prefetch is
  // only a hint and L2 is the coherence point, so it cannot return stale data
  // even if the previous kernel writes B.  Every other global access comes
  // after grid_dependency_wait().
  if (warp == 0 && lane == 0) {
    for (int64_t v = u_begin; v < u_end && v < u_begin + kEarlyUnits; ++v) {
      const int png = static_cast<int>(v / sp.kb_total);
      const int pkb = static_cast<int>(v - static_cast<int64_t>(png) * sp.kb_total);
#pragma unroll
      for (int b = 0; b < NSUB * kBoxesPerTile; ++b)
        tma_prefetch_l2_2d(&tmB, png * NW + b * 64, pkb * BK);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tail->tmem_base;
  grid_dependency_wait();

  if (warp == 0) {
    // -------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int64_t u = u_begin; u < u_end; ++u, ++it) {
        const int ng = static_cast<int>(u / sp.kb_total);
        const int kb = static_cast<int>(u - static_cast<int64_t>(ng) * sp.kb_total);
        const int s = it % STAGES;
        const uint32_t round = it / STAGES;
        if (!mbar_wait(&tail->empty[s], (round & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        uint8_t* sb = smem + s * kStageBytes;
        uint8_t* sa = sb + kStageBytesB;
        mbar_arrive_expect_tx(&tail->full[s], kStageBytes);
#pragma unroll
        for (int b = 0; b < NSUB * kBoxesPerTile; ++b)
          tma_load_2d(sb + b * kBoxBytesB, &tmB, ng * NW + b * 64, kb * BK, &tail->full[s]);
#pragma unroll
        for (int a = 0; a < kABoxes; ++a)
          tma_load_2d(sa + a * (BMr * 64 * 2), &tmA, kb * BK + a * 64, row0, &tail->full[s]);
      }
      // This CTA has issued all its loads: the next kernel in the stream may
      // start launching (it waits for this grid's completion before use).
      grid_launch_dependents();
      if (!ok) {
        const uint32_t first = it > STAGES ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j)
          mbar_drain_wait(&tail->full[j % STAGES], (j / STAGES) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1 || (kIssuers == 2 && warp == kSecondIssuerWarp)) {
    // -------------------------------------------------------- MMA issuers
    const uint32_t q = (warp == 1) ? 0u : 1u;  // this issuer's stage parity
    if (lane == 0) {
      uint32_t it = 0, seg = 0;
      bool ok = true, issued = false;
      int64_t u = u_begin;
      while (u < u_end && ok) {
        const int ng = static_cast<int>(u / sp.kb_total);
        const int64_t seg_end_u = min(u_end, static_cast<int64_t>(ng + 1) * sp.kb_total);
        const uint32_t ab = seg & 1u, ar = seg >> 1;
        if (!mbar_wait(&tail->tmem_empty[ab], (ar & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + ab * kAccCols + q * kIssuerCols;
        bool first = true;
        for (; u < seg_end_u; ++u, ++it) {
          if (it % kIssuers != q) continue;
          const int s = it % STAGES;
          const uint32_t round = it / STAGES;
          if (!mbar_wait(&tail->full[s], round & 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t sb = smem_u32(smem + s * kStageBytes);
          const uint32_t sa = sb + kStageBytesB;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // MMA B operand = A^T tile: K-major, 8-row groups 1024 B apart,
            // k step of 16 elements = 32 B.
            const uint64_t bdesc =
                smem_desc_sw128(sa + (kk / 4) * (BMr * 64 * 2) + (kk % 4) * 32, 16, 1024);
#pragma unroll
            for (int j = 0; j < NSUB; ++j) {
              // MMA A operand = B^T tile j: MN-major, its two 64-column boxes
              // 8 KB apart (LBO), 8-row k groups 1024 B apart (SBO), k step
              // of 16 rows = 2048 B.
              const uint64_t adesc = smem_desc_sw128(
                  sb + j * kBoxesPerTile * kBoxBytesB + kk * 2048, kBoxBytesB, 1024);
              tc_mma_f16(d_tmem + j * BMr, adesc, bdesc, kIdesc,
                         (first && kk == 0) ? 0u : 1u);
            }
          }
          first = false;
          issued = true;
          tc_commit(&tail->empty[s]);
        }
        if (!ok) break;
        tc_commit(&tail->tmem_full[ab]);
        ++seg;
      }
      if (!ok && issued) {
        tc_commit(&tail->drain[q]);
        mbar_drain_wait(&tail->drain[q], 0);
      }
    }
    __syncwarp();
  } else if (warp >= 2 && warp <= 5) {
    // -------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    // row of each MMA tile held by this thread = column of C within the tile
    const int n_local = quarter * kRowsPerQuarter + lane;
    const bool row_valid = lane < kRowsPerQuarter && n_local < BN;
    const int ept = threadIdx.x - 64;         // 0..127
    float amax_acc = 0.0f;
    uint32_t seg = 0;
    int64_t u = u_begin;
    while (u < u_end) {
      const int ng = static_cast<int>(u / sp.kb_total);
      const int64_t grp_u0 = static_cast<int64_t>(ng) * sp.kb_total;
      const int64_t grp_u1 = grp_u0 + sp.kb_total;
      const int64_t seg_end_u = min(u_end, grp_u1);
      const bool whole = (u == grp_u0) && (seg_end_u == grp_u1);
      const int64_t c_first = run_owner(sp, grp_u0);
      const int64_t c_last = run_owner(sp, grp_u1 - 1);
      const uint32_t nsegs = static_cast<uint32_t>(c_last - c_first + 1);
      // While the MMAs of this segment run: fetch the old C values this
      // thread may have to combine with, and watch whether every other
      // contributor of the n-group has already published its partial sums --
      // if so, preload them, so that once this segment's accumulator is ready
      // the group's result is a few adds away.
      const bool clustered = p.cluster > 1;
      // Old C and residual values of the first 16-row chunk (the only chunk
      // when BMr == 16), loaded while the MMAs of this segment run; further
      // chunks are loaded when stored.  (A cluster split loads them in
      // cluster_reduce_store.)
      float old[NSUB][kChunk], res[NSUB][kChunk];
#pragma unroll
      for (int j = 0; j < NSUB; ++j) {
        const int nc = (row_valid && !clustered) ? ng * NW + j * BN + n_local : p.N;
        load_c_column(p, nc, 0, old[j]);
        if (FUSED) load_r_column(p, nc, 0, res[j]);
      }
      // While the MMAs of this segment run, watch whether every other
      // contributor of the n-group has already published its partial sums --
      // if so, preload them (one 16-row chunk: BMr == 16 only), so that once
      // this segment's accumulator is ready the group's result is a few adds
      // away.
      constexpr int kPre = 2;  // partial sums of other CTAs held in registers
      float pre[kPre][NSUB][kChunk];
      bool preloaded = false;
      const bool can_preload = Cfg::kChunks == 1 && row_valid && !whole && !clustered &&
                               (nsegs - 1 <= static_cast<uint32_t>(kPre));
      auto preload = [&]() {
        // the kk-th contributor other than this CTA, in CTA order
#pragma unroll
        for (int kk = 0; kk < kPre; ++kk) {
          int64_t cc = c_first + kk;
          if (cc >= blockIdx.x) ++cc;
          if (cc > c_last) break;
          const int sl = static_cast<int>(ng - run_start(sp, cc) / sp.kb_total);
          const float* src = p.workspace + (cc * sp.segs_max + sl) * kPartialFloats;
#pragma unroll
          for (int j = 0; j < NSUB; ++j)
#pragma unroll
            for (int m = 0; m < kChunk; ++m)
              pre[kk][j][m] = __ldcg(src + m * NW + j * BN + n_local);
        }
      };

      const uint32_t ab = seg & 1u, ar = seg >> 1;
      bool ok = true;
      if (!mbar_try_wait(&tail->tmem_full[ab], ar & 1u)) {
        const uint64_t t0 = globaltimer_ns();
        uint32_t spins = 0;
        while (!mbar_try_wait(&tail->tmem_full[ab], ar & 1u)) {
          if ((++spins & 15u) != 0) continue;
          if (*abort_flag) { ok = false; break; }
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(p.err, kErrWaitTimeout);
            ok = false;
            break;
          }
          if (!whole && !clustered && ept == 0 && !tail->others_ready &&
              ld_acquire_gpu(p.counters + ng) == nsegs - 1)
            st_release_cta_shared(&tail->others_ready, 1);
          if (can_preload && !preloaded && ld_acquire_cta_shared(&tail->others_ready)) {
            preload();
            preloaded = true;
          }
        }
      }
      // Leave together if a wait ran out anywhere (see named_bar_any).
      if (named_bar_any(1, kEpiThreads, !ok)) break;
      tc_fence_after_sync();
      // This thread's column of the segment's sums, BMr rows, read from TMEM
      // 16 rows at a time.  Issuer qq wrote an accumulator for this segment
      // iff one of the segment's units has stage index it = u - u_begin with
      // it % kIssuers == qq; the written ones are added in issuer order.
      uint32_t r[NSUB][BMr];
      {
        const int64_t it0 = u - u_begin;
        const int64_t len = seg_end_u - u;
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c) {
          uint32_t acc[kIssuers][NSUB][kChunk];
#pragma unroll
          for (int qq = 0; qq < kIssuers; ++qq)
#pragma unroll
            for (int j = 0; j < NSUB; ++j)
              tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                     ab * kAccCols + qq * kIssuerCols + j * BMr + c * kChunk,
                                 acc[qq][j]);
          tc_wait_ld();
#pragma unroll
          for (int j = 0; j < NSUB; ++j)
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
              float v = 0.0f;
              bool any = false;
#pragma unroll
              for (int qq = 0; qq < kIssuers; ++qq) {
                const bool wrote = len >= kIssuers || it0 % kIssuers == qq;
                if (wrote) {
                  v = any ? v + __uint_as_float(acc[qq][j][i]) : __uint_as_float(acc[qq][j][i]);
                  any = true;
                }
              }
              r[j][c * kChunk + i] = __float_as_uint(v);
            }
        }
        tc_fence_before_sync();
        mbar_arrive(&tail->tmem_empty[ab]);
      }
      // Output stage of rows c*16 .. c*16 + 15 of column n: old C and
      // residual values of chunk 0 were loaded ahead.
      auto store_chunk = [&](int j, int c, const float (&v)[kChunk]) {
        const int n = row_valid ? ng * NW + j * BN + n_local : p.N;
        if (c == 0) {
          store_c_column<FUSED>(p, n, 0, v, old[j], res[j], amax_acc);
        } else {
          float oc[kChunk], rc[kChunk];
          load_c_column(p, n, c * kChunk, oc);
          if (FUSED) load_r_column(p, n, c * kChunk, rc);
          else
#pragma unroll
            for (int i = 0; i < kChunk; ++i) rc[i] = 0.0f;
          store_c_column<FUSED>(p, n, c * kChunk, v, oc, rc, amax_acc);
        }
      };

      if (clustered) {
        // This CTA's k range is its run's only segment: every MMA has read
        // its stage and every copy has landed, so stage 0 holds the partial
        // sums for the exchange after the loop.
        float* part = reinterpret_cast<float*>(smem);
        if (row_valid) {
#pragma unroll
          for (int j = 0; j < NSUB; ++j)
#pragma unroll
            for (int m = 0; m < BMr; ++m) part[m * NW + j * BN + n_local] = __uint_as_float(r[j][m]);
        }
      } else if (whole) {
#pragma unroll
        for (int j = 0; j < NSUB; ++j)
#pragma unroll
          for (int c = 0; c < Cfg::kChunks; ++c) {
            float v[kChunk];
#pragma unroll
            for (int i = 0; i < kChunk; ++i) v[i] = __uint_as_float(r[j][c * kChunk + i]);
            store_chunk(j, c, v);
          }
      } else {
        // last_flag: 2 = every other contributor had already arrived (this
        // CTA adds its own sum straight from registers and publishes nothing),
        // 1 = this CTA's arrival was the last one, 0 = another CTA finishes.
        if (ept == 0) {
          bool ready = tail->others_ready != 0;
          if (!ready) ready = ld_acquire_gpu(p.counters + ng) == nsegs - 1;
          // The CTA holding the group's first k-piece finishes it last in its
          // run, so it is the designated combiner: rather than publish its
          // own partial it waits a short, bounded time for the others (which
          // never wait on anyone), then falls back to the arrival protocol.
          if (!ready && blockIdx.x == c_first) {
            const uint64_t t0 = globaltimer_ns();
            while (!ready && globaltimer_ns() - t0 < kHandoffWaitNs)
              ready = ld_acquire_gpu(p.counters + ng) == nsegs - 1;
          }
          tail->last_flag = ready ? 2 : 0;
        }
        named_bar_epi();
        const int mode = tail->last_flag;
        if (mode != 2) {
          const int seg_local = static_cast<int>(ng - u_begin / sp.kb_total);
          float* slot = p.workspace + (static_cast<int64_t>(blockIdx.x) * sp.segs_max + seg_local) *
                                          kPartialFloats;
          if (row_valid) {
#pragma unroll
            for (int j = 0; j < NSUB; ++j)
#pragma unroll
              for (int m = 0; m < BMr; ++m)
                __stcg(slot + m * NW + j * BN + n_local, __uint_as_float(r[j][m]));
          }
          named_bar_epi();
          if (ept == 0) {
            __threadfence();  // publish the whole CTA's partial before arriving
            const uint32_t before = atomicAdd(p.counters + ng, 1u);
            tail->last_flag = (before == nsegs - 1) ? 1 : 0;
          }
          named_bar_epi();
        }
        const int fin = tail->last_flag;
        if (fin) {
          if (fin == 1) __threadfence();  // acquire the other partials after the atomic
          const bool use_pre = (fin == 2) && preloaded;
#pragma unroll
          for (int j = 0; j < NSUB; ++j)
#pragma unroll
            for (int c = 0; c < Cfg::kChunks; ++c) {
              // add the partial sums in k order (CTA order), whoever arrived last
              float sum[kChunk];
#pragma unroll
              for (int i = 0; i < kChunk; ++i) sum[i] = 0.0f;
              int k = 0;
              for (int64_t cc = c_first; cc <= c_last; ++cc) {
                if (cc == blockIdx.x) {
#pragma unroll
                  for (int i = 0; i < kChunk; ++i) sum[i] += __uint_as_float(r[j][c * kChunk + i]);
                } else if (use_pre) {
#pragma unroll
                  for (int kk = 0; kk < kPre; ++kk)
                    if (kk == k)
#pragma unroll
                      for (int i = 0; i < kChunk; ++i) sum[i] += pre[kk][j][i];
                  ++k;
                } else {
                  const int sl = static_cast<int>(ng - run_start(sp, cc) / sp.kb_total);
                  const float* src = p.workspace + (cc * sp.segs_max + sl) * kPartialFloats;
#pragma unroll
                  for (int i = 0; i < kChunk; ++i)
                    sum[i] += row_valid ? __ldcg(src + (c * kChunk + i) * NW + j * BN + n_local)
                                        : 0.0f;
                }
              }
              store_chunk(j, c, sum);
            }
          if (ept == 0) p.counters[ng] = 0u;
        }
        if (ept == 0) tail->others_ready = 0;
        named_bar_epi();  // last_flag / others_ready are rewritten by the next segment
      }
      u = seg_end_u;
      ++seg;
    }
    if (FUSED) epi_flush_amax(p.epi, amax_acc);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (p.cluster > 1) {
    // Every CTA of the cluster reaches these barriers, also after a wait ran
    // out (each wait above is bounded), so none can hang here.
    cluster_sync();  // the partial sums of every CTA of the cluster are written
    if (warp >= 2 && warp <= 5)
      cluster_reduce_store<FUSED, BMR>(p, smem_u32(smem), static_cast<int>(threadIdx.x) - 64);
    cluster_sync();  // no CTA leaves while another may still read its shared memory
  }
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// Clusters of S decode CTAs that can be resident at once on the current
// device (cudaOccupancyMaxActiveClusters; one CTA per SM, and a cluster must
// fit in one GPC: on a 152-SM GB300, 76 of 2, 36 of 4, 15 of 8).  Queried
// once per device, kernel instance and size.
template <int BMR>
int max_clusters_of(int S) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev][4];  // S = 1, 2, 4, 8; 0 = not yet known
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) {
    cudaGetLastError();
    return 0;
  }
  const int slot = S >= 8 ? 3 : S >= 4 ? 2 : S >= 2 ? 1 : 0;
  const int known = cache[dev][slot].load(std::memory_order_relaxed);
  if (known != 0) return known;
  auto kernel = tc_decode_kernel<false, BMR>;
  int n = 0;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(DecCfg<BMR>::kSmemBytes)) == cudaSuccess) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(S));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = DecCfg<BMR>::kSmemBytes;
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
  if (n > 0) cache[dev][slot].store(n, std::memory_order_relaxed);
  return n;
}

int decode_max_clusters(int S, int rows) {
  return rows <= 16 ? max_clusters_of<16>(S) : rows <= 32 ? max_clusters_of<32>(S)
                                                          : max_clusters_of<64>(S);
}

template <int BMR>
cudaError_t launch_rows(const DecodeArgs& a, const CUtensorMap* tmA, const CUtensorMap* tmB,
                        int num_ctas, bool fused, cudaStream_t stream) {
  constexpr size_t kSmemBytes = DecCfg<BMR>::kSmemBytes;
  auto kernel = fused ? tc_decode_kernel<true, BMR> : tc_decode_kernel<false, BMR>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  // Programmatic stream serialization: this launch may begin while the
  // previous kernel in the stream drains (see grid_dependency_wait).
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(num_ctas, decode_row_blocks(a.M));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.cluster > 1) {
    if (num_ctas % a.cluster != 0) return cudaErrorInvalidValue;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(a.cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  e = cudaLaunchKernelEx(&cfg, kernel, a, *tmA, *tmB);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int decode_b_box_rows() { return BK; }

int decode_rows(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : 64; }

int decode_row_blocks(int M) { return M <= kDecBlockRows ? 1 : (M + kDecBlockRows - 1) / kDecBlockRows; }

int64_t decode_groups(int N) { return (N + NW - 1) / NW; }

int decode_cluster(int M, int N, int K, int num_sms) {
  const int64_t groups = (N + NW - 1) / NW;
  const int64_t kb_total = (K + BK - 1) / BK;
  const int blocks = decode_row_blocks(M);
  const int64_t slots = num_sms / blocks;  // SMs per row block
  if (groups * 5 >= slots * 3) return 1;  // whole groups, or runs of them
  // The largest power of two S <= 8 (portable cluster size) with at least
  // one k-block per CTA and all groups' clusters (of every row block)
  // resident at once (more would run in two waves: 16 clusters of 8 took
  // twice as long as 8).
  const int rows = decode_rows(M);
  int S = 1;
  while (S < 8 && groups * S * 2 <= slots && S * 2 <= kb_total &&
         groups * blocks <= decode_max_clusters(S * 2, rows))
    S *= 2;
  return S;
}

int decode_grid(int M, int N, int K, int num_sms) {
  const int64_t groups = (N + NW - 1) / NW;
  const int64_t units = groups * ((K + BK - 1) / BK);
  const int64_t slots = num_sms / decode_row_blocks(M);  // SMs per row block
  // Enough column groups to keep most SMs streaming (>= ~60 % of them): one
  // CTA per group, so no group's k range is split and no partial sums are
  // exchanged.  Fewer groups: clusters of S CTAs per group split its k range
  // evenly (run_start then never crosses a group) and add their partial sums
  // through distributed shared memory; where no S >= 2 fits, whole groups
  // again.  More groups than SMs: each CTA takes a run of whole groups (only
  // the groups at run boundaries are split, through the workspace).
  if (groups <= slots) {
    const int S = decode_cluster(M, N, K, num_sms);
    return static_cast<int>(groups * S);
  }
  return static_cast<int>(units < slots ? units : slots);
}

int64_t decode_workspace_floats(int M, int N, int K, int num_ctas) {
  const Split s = make_split(N, K, num_ctas);
  return static_cast<int64_t>(num_ctas) * s.segs_max * decode_rows(M) * NW * decode_row_blocks(M);
}

int64_t decode_counter_count(int M, int N) { return decode_groups(N) * decode_row_blocks(M); }

cudaError_t launch_tc_decode(const DecodeArgs& a, const CUtensorMap* tmA, const CUtensorMap* tmB,
                             int num_ctas, cudaStream_t stream) {
  const Epilogue& ep = a.epi;
  const bool fused = ep.bias != nullptr || ep.act != kActNone || ep.R != nullptr ||
                     ep.d_type != kOutF32 || ep.d_scale != 1.0f || ep.amax != nullptr ||
                     ep.D != static_cast<const void*>(ep.C) || ep.ldd != ep.ldc;
  if (a.M < 1 || a.M > kDecMaxM) return cudaErrorInvalidValue;
  const int rows = decode_rows(a.M);
  if (rows == 16) return launch_rows<16>(a, tmA, tmB, num_ctas, fused, stream);
  if (rows == 32) return launch_rows<32>(a, tmA, tmB, num_ctas, fused, stream);
  return launch_rows<64>(a, tmA, tmB, num_ctas, fused, stream);
}

}  // namespace g12
