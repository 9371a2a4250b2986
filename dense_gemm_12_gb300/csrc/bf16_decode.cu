// bf16_decode.cu -- decode-shaped GEMM (M <= 16): C = alpha * A * B + beta * C
// with bf16 A (M x K) and B (K x N), fp32 accumulation and fp32 C.
//
// "Tiled matrix multiplication" ("Avoid when") notes that a decode GEMV with
// M <= 16 is bound by memory bandwidth: the whole cost is streaming B once.
// With M = 16 no tile of C is big enough to fill the machine, so the k range
// is split across CTAs and the partial sums are reduced afterwards ("Split-K"
// in the same page's "Variants and alternatives"; "A GEMM Kernel, Step by
// Step", "What is left").  On sm_103a the tensor core's smallest M is 128, so
// the product is computed transposed, D^T = B^T A^T: the MMA's M runs over
// 128 columns of C and its N (16) over the rows of A, and no row of the MMA
// is padding.
//
// Work split.  The (n-tile, k-block) units -- 128 columns x 64 k each -- are
// numbered n-tile-major and every CTA takes one contiguous, equal-sized run of
// them, so each SM streams the same number of bytes of B (no last wave).  A
// run is cut into segments at n-tile boundaries.  A segment that spans the
// whole k range of its n-tile writes C directly; otherwise it stores its
// 128 x 16 fp32 partial in the workspace and bumps the n-tile's arrival
// counter, and the CTA that arrives last adds the partials in k order (a
// fixed order, so results are deterministic), applies alpha/beta, writes C and
// resets the counter to zero for the next launch.
//
// Roles: warp 0 TMA producer (two 64-column MN-major boxes of B and a 16 x 64
// K-major box of A per stage), warp 1 TMEM owner and MMA issuer (128 x 16 x 16
// MMAs, two accumulators), warps 2..5 epilogue / fix-up.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace g12 {
namespace {

constexpr int BN = kDecBN;   // MMA M: columns of C per n-tile
constexpr int BMr = kDecBM;  // MMA N: rows of A / C
constexpr int BK = kDecBK;
constexpr int STAGES = 8;
constexpr int kStageBytesB = BK * BN * 2;   // 16 KB: two 64-column boxes
constexpr int kBoxBytesB = BK * 64 * 2;     // 8 KB
constexpr int kStageBytesA = BMr * BK * 2;  // 2 KB
constexpr int kStageBytes = kStageBytesB + kStageBytesA;  // 18 KB (multiple of 1024)
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr uint32_t kTmemCols = 32;
constexpr uint32_t kIdesc = idesc_bf16_f32(BN, BMr, /*A MN-major*/ 1, /*B MN-major*/ 0);
constexpr int kPartialFloats = BMr * BN;    // 2048

struct __align__(8) DecSmemTail {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int last_flag;
};

constexpr size_t kSmemBytes = 1024 + STAGES * kStageBytes + sizeof(DecSmemTail);

struct Split {
  int64_t units;       // n_tiles * kb_total
  int kb_total;        // k-blocks per n-tile
  int grid;            // CTAs
  int segs_max;        // segment slots per CTA in the workspace
};

__host__ __device__ inline Split make_split(int N, int K, int grid) {
  Split s;
  const int n_tiles = (N + BN - 1) / BN;
  s.kb_total = (K + BK - 1) / BK;
  s.units = static_cast<int64_t>(n_tiles) * s.kb_total;
  s.grid = grid;
  const int64_t per_cta = (s.units + grid - 1) / grid;
  s.segs_max = static_cast<int>((per_cta + s.kb_total - 1) / s.kb_total) + 1;
  return s;
}

__device__ __forceinline__ int64_t run_start(const Split& s, int64_t c) {
  return (c * s.units) / s.grid;
}

// The CTA whose run contains unit u: the largest c with run_start(c) <= u.
__device__ __forceinline__ int64_t run_owner(const Split& s, int64_t u) {
  return ((u + 1) * s.grid + s.units - 1) / s.units - 1;
}

__device__ __forceinline__ void named_bar_epi() {
  asm volatile("bar.sync 1, %0;" ::"r"(kEpiThreads) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    tc_decode_kernel(const DecodeArgs p, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  DecSmemTail* tail = reinterpret_cast<DecSmemTail*>(smem + STAGES * kStageBytes);
  volatile int* abort_flag = &tail->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Split sp = make_split(p.N, p.K, gridDim.x);
  const int64_t u_begin = run_start(sp, blockIdx.x);
  const int64_t u_end = run_start(sp, static_cast<int64_t>(blockIdx.x) + 1);

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
      for (int64_t u = u_begin; u < u_end; ++u, ++it) {
        const int nt = static_cast<int>(u / sp.kb_total);
        const int kb = static_cast<int>(u - static_cast<int64_t>(nt) * sp.kb_total);
        const int s = it % STAGES;
        const uint32_t round = it / STAGES;
        if (!mbar_wait(&tail->empty[s], (round & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        uint8_t* sb = smem + s * kStageBytes;
        uint8_t* sa = sb + kStageBytesB;
        mbar_arrive_expect_tx(&tail->full[s], kStageBytes);
        tma_load_2d(sb, &tmB, nt * BN, kb * BK, &tail->full[s]);
        tma_load_2d(sb + kBoxBytesB, &tmB, nt * BN + 64, kb * BK, &tail->full[s]);
        tma_load_2d(sa, &tmA, kb * BK, 0, &tail->full[s]);
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
      uint32_t it = 0, seg = 0;
      bool ok = true, issued = false;
      int64_t u = u_begin;
      while (u < u_end && ok) {
        const int nt = static_cast<int>(u / sp.kb_total);
        const int64_t seg_end_u = min(u_end, static_cast<int64_t>(nt + 1) * sp.kb_total);
        const uint32_t ab = seg & 1u, ar = seg >> 1;
        if (!mbar_wait(&tail->tmem_empty[ab], (ar & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + ab * BMr;
        bool first = true;
        for (; u < seg_end_u; ++u, ++it) {
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
            // MMA A operand = B^T tile: MN-major, two 64-column boxes 8 KB
            // apart (LBO), 8-row k groups 1024 B apart (SBO), k step 2048 B.
            const uint64_t adesc = smem_desc_sw128(sb + kk * 2048, kBoxBytesB, 1024);
            // MMA B operand = A^T tile: K-major, 8-row groups 1024 B apart,
            // k step of 16 elements = 32 B.
            const uint64_t bdesc = smem_desc_sw128(sa + kk * 32, 16, 1024);
            tc_mma_f16(d_tmem, adesc, bdesc, kIdesc, (first && kk == 0) ? 0u : 1u);
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
        tc_commit(&tail->drain);
        mbar_drain_wait(&tail->drain, 0);
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int n_local = quarter * 32 + lane;
    const int ept = threadIdx.x - 64;  // 0..127
    uint32_t seg = 0;
    int64_t u = u_begin;
    while (u < u_end) {
      const int nt = static_cast<int>(u / sp.kb_total);
      const int64_t tile_u0 = static_cast<int64_t>(nt) * sp.kb_total;
      const int64_t tile_u1 = tile_u0 + sp.kb_total;
      const int64_t seg_end_u = min(u_end, tile_u1);
      const bool whole = (u == tile_u0) && (seg_end_u == tile_u1);
      const uint32_t ab = seg & 1u, ar = seg >> 1;
      if (!mbar_wait(&tail->tmem_full[ab], ar & 1u, abort_flag, p.err)) break;
      tc_fence_after_sync();
      uint32_t r[16];
      tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + ab * BMr, r);
      tc_wait_ld();
      tc_fence_before_sync();
      mbar_arrive(&tail->tmem_empty[ab]);

      const int n = nt * BN + n_local;
      if (whole) {
        if (n < p.N) {
#pragma unroll
          for (int m = 0; m < BMr; ++m) {
            if (m < p.M) {
              float* c = p.C + static_cast<int64_t>(m) * p.ldc + n;
              const float v = __uint_as_float(r[m]);
              *c = (p.beta != 0.0f) ? fmaf(p.alpha, v, p.beta * *c) : p.alpha * v;
            }
          }
        }
      } else {
        const int64_t first_u = u_begin;
        const int seg_local = static_cast<int>(nt - first_u / sp.kb_total);
        float* slot = p.workspace +
                      (static_cast<int64_t>(blockIdx.x) * sp.segs_max + seg_local) * kPartialFloats;
#pragma unroll
        for (int m = 0; m < BMr; ++m) __stcg(slot + m * BN + n_local, __uint_as_float(r[m]));
        __threadfence();
        named_bar_epi();
        const int64_t c_first = run_owner(sp, tile_u0);
        const int64_t c_last = run_owner(sp, tile_u1 - 1);
        if (ept == 0) {
          const uint32_t nsegs = static_cast<uint32_t>(c_last - c_first + 1);
          const uint32_t before = atomicAdd(p.counters + nt, 1u);
          tail->last_flag = (before == nsegs - 1) ? 1 : 0;
        }
        named_bar_epi();
        if (tail->last_flag) {
          __threadfence();
          float sum[BMr];
#pragma unroll
          for (int m = 0; m < BMr; ++m) sum[m] = 0.0f;
          for (int64_t cc = c_first; cc <= c_last; ++cc) {
            const int sl = static_cast<int>(nt - run_start(sp, cc) / sp.kb_total);
            const float* src = p.workspace + (cc * sp.segs_max + sl) * kPartialFloats;
#pragma unroll
            for (int m = 0; m < BMr; ++m) sum[m] += __ldcg(src + m * BN + n_local);
          }
          if (n < p.N) {
#pragma unroll
            for (int m = 0; m < BMr; ++m) {
              if (m < p.M) {
                float* c = p.C + static_cast<int64_t>(m) * p.ldc + n;
                *c = (p.beta != 0.0f) ? fmaf(p.alpha, sum[m], p.beta * *c) : p.alpha * sum[m];
              }
            }
          }
          if (ept == 0) p.counters[nt] = 0u;
        }
      }
      u = seg_end_u;
      ++seg;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace

int decode_grid(int N, int K, int num_sms) {
  const int64_t units = static_cast<int64_t>((N + BN - 1) / BN) * ((K + BK - 1) / BK);
  return static_cast<int>(units < num_sms ? units : num_sms);
}

int64_t decode_workspace_floats(int N, int K, int num_ctas) {
  const Split s = make_split(N, K, num_ctas);
  return static_cast<int64_t>(num_ctas) * s.segs_max * kPartialFloats;
}

int64_t decode_counter_count(int N) { return (N + BN - 1) / BN; }

cudaError_t launch_tc_decode(const DecodeArgs& a, const CUtensorMap* tmA, const CUtensorMap* tmB,
                             int num_ctas, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(tc_decode_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  tc_decode_kernel<<<num_ctas, kThreads, kSmemBytes, stream>>>(a, *tmA, *tmB);
  return cudaGetLastError();
}

}  // namespace g12
