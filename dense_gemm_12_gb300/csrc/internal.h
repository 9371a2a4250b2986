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
  // raster order; every later tile is cut into `split` k-ranges whose partial
  // sums meet in `ws` (split x 64 KB per tile) and are added by the last of
  // them to arrive on the tile's counter in `counters` (zero between launches).
  int full_items;
  int split;
  float* ws;
  uint32_t* counters;
  int group_m;     // raster group height in tile rows
};

// A launch configuration of the tile kernels: gemm_config_t of the C ABI
// with every field resolved (no "auto" values).
struct TileConfig {
  int kernel;    // GEMM_KERNEL_SINGLE_CTA or GEMM_KERNEL_CTA_PAIR
  int split;     // k-ranges per item of the last round, 1..8
  int group_m;   // raster group height, 1..64
};

// Work plan of the CUDA-core kernel for tiles output tiles, num_kb k-blocks
// and up to num_sms persistent CTAs: how many tiles run whole, how the rest
// are split along k, and the grid.  `fixed` pins the split (and carries the
// group height); nullptr lets the cost model choose.
struct SimtPlan {
  int full_items;
  int split;
  int grid;
  int group_m;
  int64_t ws_floats;   // workspace the split tiles need
  int64_t counters;    // counters the split tiles need
};
SimtPlan simt_plan(int tiles, int num_kb, int num_sms, const TileConfig* fixed);

// CUDA-core (FFMA) GEMM: 128 x 128 block tiles, warp tiles 32 x 64, 8 x 8
// register micro-tiles.  tmA / tmB are used only for operands in kLoadTma mode.
cudaError_t launch_simt(const SimtArgs& a, LoadMode mode_a, LoadMode mode_b,
                        const CUtensorMap* tmA, const CUtensorMap* tmB, int num_sms,
                        cudaStream_t stream);

// Tile geometry of the CUDA-core kernel (also used by the launch planner).
constexpr int kSimtBM = 128, kSimtBN = 128, kSimtBK = 32;

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
  // whole; every later one is cut into `split` k-ranges whose partial sums
  // meet in `ws` (128 x 256 floats per part and CTA) and are added, in part
  // order, by the last part to arrive on its counter in `counters` (one per
  // item and CTA, zero between launches).
  int full_items;
  int split;
  float* ws;
  uint32_t* counters;
  int group_m;     // raster group height in tile rows (pair-tile rows on pairs)
};

// Launch plan of the bf16 tensor-core GEMM for one shape.
struct TcPlan {
  bool pair;          // CTA-pair kernel or single-CTA kernel
  int full_items;
  int split;
  int grid;           // CTAs to launch (pairs: twice the clusters)
  int group_m;
  int64_t ws_floats;  // workspace the split items need
  int64_t counters;   // counters the split items need
};
// `fixed` pins kernel, split and group height; nullptr: the pair kernel for
// M > 128, the cost model's split, groups of 8.
TcPlan tc_plan(int M, int N, int K, int num_sms, const TileConfig* fixed);
// k-rows of B per TMA box of the single-CTA (pair = false) or pair kernel.
int tc_b_box_rows(bool pair);

// bf16 tensor-core GEMM (tcgen05, accumulator in TMEM): 128 x 256 tiles on
// one CTA, or 256 x 256 tiles on CTA pairs, as planned by tc_plan.
cudaError_t launch_tc_bf16(const TcArgs& a, const TcPlan& plan, const CUtensorMap* tmA,
                           const CUtensorMap* tmB, cudaStream_t stream);
constexpr int kTcBM = 128, kTcBN = 256, kTcBK = 64;

struct DecodeArgs {
  int M, N, K;
  Epilogue epi;
  float* workspace;     // partial sums, see decode_workspace_floats
  uint32_t* counters;   // one arrival counter per 128-column n-tile, zeroed
  uint32_t* err;
};

// bf16 decode GEMM (M <= 16): tcgen05 with the operands swapped
// (D^T = B^T A^T, MMA M = 128 over N, MMA N = 16 over M), split over K.
cudaError_t launch_tc_decode(const DecodeArgs& a, const CUtensorMap* tmA,
                             const CUtensorMap* tmB, int num_ctas, cudaStream_t stream);
constexpr int kDecBN = 128, kDecBM = 16;
// k-rows of B per TMA box of the decode kernel (the A box is always 64 wide).
int decode_b_box_rows();
// Workspace floats and counters a decode launch of this shape needs.
int64_t decode_workspace_floats(int N, int K, int num_ctas);
int64_t decode_counter_count(int N);
int decode_grid(int N, int K, int num_sms);

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
cudaError_t launch_scale_c(int M, int N, float beta, float* C, int64_t ldc,
                           cudaStream_t stream);

}  // namespace g12
