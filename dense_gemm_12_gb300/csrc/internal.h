// internal.h -- host-side interface between the C ABI (api.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "epilogue.cuh"

namespace g12 {

// How one operand of the CUDA-core kernel reaches shared memory.
enum LoadMode : int {
  kLoadTma = 0,         // tiled TMA copy (fp32, 16-B aligned base and pitch)
  kLoadCpAsyncF32 = 1,  // 4-byte cp.async by producer warps (any fp32 layout)
  kLoadConvertBf16 = 2, // bf16 loads widened to fp32 by producer warps
};

struct SimtArgs {
  int M, N, K;
  float alpha, beta;
  const void* A;   // fp32 or bf16 elements
  int64_t lda;
  const void* B;
  int64_t ldb;
  float* C;
  int64_t ldc;
  int c_vec4;      // 1 if C rows may be written as aligned float4
  uint32_t* err;   // device error word
  // Work plan (see simt_plan): items [0, full_items) are whole tiles in
  // raster order.  The later ("tail") tiles are either cut into `split`
  // equal k-ranges each (sk_workers == 0), or, with sk_workers = G > 0, their
  // k-blocks taken together are dealt out evenly to G workers (stream-K, see
  // sk_range).  Partial sums meet in `ws` (one tile of floats per part) and
  // are added, in k order, by the last part to arrive on the tile's counter
  // in `counters` (zero between launches).
  int full_items;
  int split;
  int sk_workers;
  float* ws;
  uint32_t* counters;
  int group_m;     // raster group height in tile rows
  // > 1: every tile runs in this one round, cut into `cluster` (= split)
  // parts that form a thread-block cluster and add their partial sums
  // through distributed shared memory: no workspace, no counters.
  int cluster;
};

// A launch configuration of the tile kernels: gemm_config_t of the C ABI
// with every field resolved (no "auto" values).
struct TileConfig {
  int kernel;    // GEMM_KERNEL_SINGLE_CTA, GEMM_KERNEL_CTA_PAIR or GEMM_KERNEL_WIDE
  int split;     // k-ranges per item of the last round, 1..8, or GEMM_SPLIT_STREAM
  int group_m;   // raster group height, 1..64
};

// Work plan of the CUDA-core kernel for an M x N x K problem on up to
// num_sms persistent CTAs: the tile width, how many tiles run whole, how the
// rest are cut along k, and the grid.  `fixed` pins the kernel (tile width),
// the split (or stream-K) and the group height; nullptr or zero fields let
// the cost model choose.  allow_wide = false keeps 128-wide tiles.
struct SimtPlan {
  bool wide;           // 128 x 256 tiles (else 128 x 128)
  int full_items;
  int split;
  int sk_workers;      // > 0: stream-K tail over this many workers
  int grid;
  int group_m;
  int64_t ws_floats;   // workspace the split tiles need
  int64_t counters;    // counters the split tiles need
  int cluster;         // > 1: the parts of each tile form a cluster (see SimtArgs)
};
SimtPlan simt_plan(int M, int N, int K, int num_sms, const TileConfig* fixed, bool allow_wide);
// Largest cluster of k-parts (the portable cluster size).
constexpr int kSimtMaxCluster = 8;
// Turns a plan whose tiles all run in one round, each cut into 2..8 equal
// k-parts, into its cluster form (pl.cluster = pl.split, no workspace) when
// every tile's cluster can be resident at once on the current device.  For
// 128-wide tiles with both operands on TMA only; returns whether it did.
bool simt_use_cluster(SimtPlan& pl, int M, int N);
// Clusters of S (2..8) CTAs of the cluster form that can be resident at once
// on the current device (one CTA per SM; a cluster must fit in one GPC), 0
// if unknown.  Queried once per device and size.
int simt_max_clusters(int S);
// Largest number of parts any tail tile of the plan is cut into (1 = none).
int simt_plan_max_parts(const SimtPlan& pl, int M, int N, int K);

// CUDA-core (FFMA) GEMM: 128 x 128 block tiles (warp tiles 32 x 64, 8 x 8
// register micro-tiles) or 128 x 256 (warp tiles 32 x 128, 8 x 16), as
// planned.  tmA / tmB are used only for operands in kLoadTma mode; tmB's box
// is simt_bn(plan.wide) columns wide.
cudaError_t launch_simt(const SimtArgs& a, const SimtPlan& plan, LoadMode mode_a,
                        LoadMode mode_b, const CUtensorMap* tmA, const CUtensorMap* tmB,
                        cudaStream_t stream);

// Tile geometry of the CUDA-core kernel (also used by the launch planner).
constexpr int kSimtBM = 128, kSimtBK = 32;
constexpr int simt_bn(bool wide) { return wide ? 256 : 128; }

// Stream-K tail: the tail's W = tail_tiles x num_kb k-blocks, taken tile after
// tile, are dealt to G workers in contiguous ranges [lo(j), lo(j + 1)) with
// lo(j) = floor(j W / G).  With G >= tail_tiles a range is at most one tile
// long, so it touches one or two tiles: its first segment (s = 0) lies in
// tile lo(j) / num_kb, its second (s = 1), if any, in the next tile.  The
// partial sums of worker j's segment s go to workspace slot 2 j + s.
__host__ __device__ inline int64_t sk_lo(int64_t j, int64_t W, int64_t G) { return j * W / G; }
// The worker whose range holds k-block x of the tail: the largest j with lo(j) <= x.
__host__ __device__ inline int64_t sk_worker(int64_t x, int64_t W, int64_t G) {
  return ((x + 1) * G - 1) / W;
}

// Number of k-parts S (1 = none) into which the items of the last round are
// cut when `items` equal work items of num_kb k-blocks run on `workers`
// persistent workers.  With R = ceil(tail * S / workers) rounds of parts the
// tail takes, in item-times,
//     R / S  +  R * S * fixup_kb / num_kb
// instead of 1: each round of parts also pays the split's own work (storing
// partial sums, and for the last part of a tile reading the other S - 1 and
// writing the tile), measured at about fixup_kb k-block times per part.
// Every part keeps at least 4 k-blocks.
int tail_split(int items, int num_kb, int workers, double fixup_kb);

struct TcArgs {
  int M, N, K;
  Epilogue epi;
  uint32_t* err;
  // Work plan (see tc_plan): work items are tiles (128 x 256) or, on CTA
  // pairs, pair tiles (256 x 256) in raster order.  Items [0, full_items) run
  // whole; the later ("tail") items are either cut into `split` equal
  // k-ranges each (sk_workers == 0), or, with sk_workers = G > 0, their
  // k-blocks taken together are dealt out evenly to G workers (stream-K, see
  // sk_lo).  Partial sums meet in `ws` (128 x 256 floats per part and CTA)
  // and are added, in k order, by the last part to arrive on its item's
  // counter in `counters` (one per tail item and CTA, zero between launches).
  int full_items;
  int split;
  int sk_workers;
  float* ws;
  uint32_t* counters;
  int group_m;     // raster group height in tile rows (pair-tile rows on pairs)
  // > 1 (single-CTA kernel only): every tile runs in this one round, cut into
  // `cluster` (= split) parts that form a thread-block cluster and add their
  // partial sums through distributed shared memory: no workspace, no counters.
  int cluster;
  // 1: the plain output stage (fp32 D = alpha * acc, beta == 0) writes whole
  // units through TMA stores described by the kernel's D tensor map (fp32,
  // dims {N, M}, row pitch ldd, box 32 x 32, 128-byte swizzle).
  int d_tma;
};

// Launch plan of the bf16 tensor-core GEMM for one shape.
struct TcPlan {
  bool pair;          // CTA-pair kernel or single-CTA kernel
  int full_items;
  int split;
  int sk_workers;     // > 0: stream-K tail over this many workers (split is then 1)
  int grid;           // CTAs to launch (pairs: twice the clusters)
  int group_m;
  int64_t ws_floats;  // workspace the split items need
  int64_t counters;   // counters the split items need
  int cluster;        // > 1: the parts of each tile form a cluster (see TcArgs)
};
// `fixed` pins kernel, split (GEMM_SPLIT_STREAM: a stream-K tail) and group
// height; nullptr: the pair kernel for M > 128, the cost model's split,
// groups of 8.
// tma_out: the output stage writes whole tiles through TMA stores (plain fp32
// output with beta == 0 and a D that TMA can describe), which makes whole
// tiles cheaper against split ones; the planning queries assume it.
TcPlan tc_plan(int M, int N, int K, int num_sms, const TileConfig* fixed, bool tma_out = true);
// Largest number of parts any tail item of the plan is cut into (1 = none).
int tc_plan_max_parts(const TcPlan& pl, int M, int N, int K);
// Turns a single-CTA plan whose tiles all run in one round, each cut into
// 2..8 equal k-parts, into its cluster form (pl.cluster = pl.split, no
// workspace) when every tile's cluster can be resident at once on the
// current device; returns whether it did.
bool tc_use_cluster(TcPlan& pl, int M, int N, const Epilogue& epi);
// k-rows of B per TMA box of the single-CTA (pair = false) or pair kernel.
int tc_b_box_rows(bool pair);

// bf16 tensor-core GEMM (tcgen05, accumulator in TMEM): 128 x 256 tiles on
// one CTA, or 256 x 256 tiles on CTA pairs, as planned by tc_plan.
cudaError_t launch_tc_bf16(const TcArgs& a, const TcPlan& plan, const CUtensorMap* tmA,
                           const CUtensorMap* tmB, const CUtensorMap* tmD, cudaStream_t stream);
// The output stage `ep` does more than fp32 D = alpha * acc + beta * C (bias,
// activation, residual, scaling, another output type or amax).
bool tc_fused(const Epilogue& ep);
// Box of the D tensor map for the TMA output stage (see TcArgs::d_tma).
constexpr int kTcStoreBoxCols = 32, kTcStoreBoxRows = 32;
constexpr int kTcBM = 128, kTcBN = 256, kTcBK = 64;

struct DecodeArgs {
  int M, N, K;
  Epilogue epi;
  float* workspace;     // partial sums, see decode_workspace_floats
  uint32_t* counters;   // one arrival counter per 128-column n-tile and row
                        // block, zeroed
  uint32_t* err;
  int cluster;          // > 1: clusters of this many CTAs split each column
                        // group's k range (decode_cluster); 0 or 1: none
};

// bf16 decode GEMM (M <= kDecMaxM): tcgen05 with the operands swapped
// (D^T = B^T A^T, MMA M = 128 over N, MMA N = 16, 32 or 64 over M), split
// over K.  M > 64 runs in row blocks of 64 (the launch's y dimension), each
// streaming B for its own rows at the same time as the others.  num_ctas:
// CTAs per row block (decode_grid).
cudaError_t launch_tc_decode(const DecodeArgs& a, const CUtensorMap* tmA,
                             const CUtensorMap* tmB, int num_ctas, cudaStream_t stream);
constexpr int kDecBN = 128, kDecBM = 16;
// Rows of the largest kernel instance (the MMA's N) and so of a row block.
constexpr int kDecBlockRows = 64;
// Largest M the decode kernel takes (eight row blocks); larger M runs on the
// tile kernels.
constexpr int kDecMaxM = 512;
// Whether automatic dispatch runs a bf16 M x N x K GEMM on the decode kernel.
// Every M <= 32.  32 < M <= 128 up to N = 16384 (two row blocks above 64
// rows); measured against the tile kernels (back-to-back launches, us):
// M = 17, 32, 48, 64 at 4096 x 4096: 10.3, 10.2, 11.9, 11.9 against
// 27.0-28.7; M = 64 at 8192 x 8192 27.8 vs 49.8, at 12288 x 4096 24.6 vs
// 43.3; M = 72-128 at N = 1024, 4096, 8192, 12288, 16384 (K = 4096): 8.7,
// 13.8, 20.9, 35.0, 41.9 against 27.9, 27.4, 36.1, 43.6, 45.6 on the
// single-CTA tile kernel (K = 8192 at N = 16384: 65.6 vs 65.8); but M = 64
// at N = 28672 (more column groups than SMs) 52.8 vs 51.1 on the tile kernel.
// 128 < M <= 512 (3 to 8 row blocks, each reading all of B, from L2 after
// the first): while the 128-column groups times the row blocks stay within
// about one round of a 152-SM GPU -- at most 128, or 160 for K >= 4096,
// where the tile kernels' fixed costs weigh less.  Measured over M = 160-512,
// N = 1024-16384, K = 1024-8192 (us, decode vs tile kernels): 256 x 4096 x
// 4096 19.1 vs 29.9, 512 x 1024 x 4096 14.3 vs 30.7, 512 x 2048 x 8192 30.2
// vs 40.2, 320 x 4096 x 4096 (160 units) 27.7 vs 32.2; beyond the bound the
// tile kernels win (256 x 8192 x 4096 38.2 vs 34.0, 512 x 4096 x 4096 35.4
// vs 34.3, 320 x 4096 x 1024 18.9 vs 18.5).
inline bool decode_path(int64_t M, int64_t N, int64_t K) {
  if (M > kDecMaxM) return false;
  if (M <= 32) return true;
  if (M <= 128) return N <= 16384;
  const int64_t units = ((N + kDecBN - 1) / kDecBN) * ((M + kDecBlockRows - 1) / kDecBlockRows);
  return units <= (K >= 4096 ? 160 : 128);
}
// Rows of the kernel instance a launch with M rows uses (16, 32 or 64).
int decode_rows(int M);
// Row blocks of a decode launch with M rows (ceil(M / 64), 1 to 8).
int decode_row_blocks(int M);
// 128-column groups of C (one arrival counter each, per row block).
int64_t decode_groups(int N);
// k-rows of B per TMA box of the decode kernel (the A box is always 64 wide).
int decode_b_box_rows();
// Workspace floats and counters a decode launch of this shape needs (all row
// blocks together).
int64_t decode_workspace_floats(int M, int N, int K, int num_ctas);
int64_t decode_counter_count(int M, int N);
// CTAs per row block.
int decode_grid(int M, int N, int K, int num_sms);
// CTAs per cluster of the decode launch (1: no clusters): when the column
// groups are few, the CTAs of a cluster split one group's k range and add
// their partial sums through distributed shared memory (no workspace).
int decode_cluster(int M, int N, int K, int num_sms);

// Pieces of the C ABI shared with entry points in other translation units.
}  // namespace g12
#include "../../include/gemm12.h"
namespace g12 {
gemm_status_t abi_check_args(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                             int64_t ldc);
bool abi_tma_ok(const void* base, int64_t ld, int elem_bytes);
bool abi_encode_bf16_2d(CUtensorMap* map, const void* base, int64_t inner, int64_t outer,
                        int64_t ld, uint32_t bx, uint32_t by);
// Current device's SM count and error-word address (GEMM_OK), or the status
// the entry points return when there is no usable sm_103a device.
gemm_status_t abi_device(int* num_sms, uint32_t** err_word);

// The output stage of the plain GEMM: D = C (fp32, in place), no bias, no
// activation.
Epilogue plain_epilogue(float alpha, float beta, float* C, int64_t ldc);
// D <- act(beta * C + bias) for an empty product.
cudaError_t launch_epilogue_only(int M, int N, const Epilogue& e, cudaStream_t stream);

// C <- beta * C (beta == 0 writes zeros without reading C).
// Copies a rows x cols row-major matrix of elem_bytes-wide elements (2 or 4)
// from src (pitch lds elements) into dst (pitch ldd elements; dst 16-byte
// aligned, ldd * elem_bytes a multiple of 16), zero-filling each row's pad.
cudaError_t launch_stage_rows(int elem_bytes, const void* src, int64_t lds, void* dst, int64_t ldd,
                              int64_t rows, int64_t cols, int num_sms, cudaStream_t stream);
cudaError_t launch_scale_c(int M, int N, float beta, float* C, int64_t ldc,
                           cudaStream_t stream);

}  // namespace g12
