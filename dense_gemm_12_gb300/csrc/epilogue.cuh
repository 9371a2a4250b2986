// epilogue.cuh -- the fused output stage of the bf16 kernels:
//
//     D[i][j] = act(alpha * acc[i][j] + beta * C[i][j] + bias[j])
//
// written as fp32 or bf16 ("Tiled matrix multiplication", "Implementation
// notes": fuse bias, activation, scaling and quantisation while the tile is
// still in registers, which saves a full read and write of C).  The plain GEMM
// is the special case act = none, no bias, D = C in fp32.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace g12 {

enum : int { kActNone = 0, kActRelu = 1, kActGelu = 2 };

struct Epilogue {
  float alpha, beta;
  const float* C;      // read when beta != 0 (ldc)
  int64_t ldc;
  void* D;             // output (ldd); may be C itself when fp32 with ldd == ldc
  int64_t ldd;
  const float* bias;   // length N, or nullptr
  int act;             // kActNone / kActRelu / kActGelu
  int d_bf16;          // 1: D holds bf16 (rounded to nearest even), 0: fp32
  int c_vec4;          // C rows may be read as aligned float4
  int d_vec;           // D rows may be written with aligned 16-byte stores
};

__device__ __forceinline__ float epi_activate(int act, float x) {
  if (act == kActRelu) return x > 0.0f ? x : 0.0f;
  if (act == kActGelu) return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
  return x;
}

// Bias of column col (0 without a bias).  Callers load every bias value they
// need before their first store to D: a load placed after a store to a
// possibly aliasing address cannot be issued early and costs a full memory
// round trip.
__device__ __forceinline__ float epi_bias(const Epilogue& e, int col) {
  return e.bias != nullptr ? e.bias[col] : 0.0f;
}

// The value of one element before it is stored.
__device__ __forceinline__ float epi_value(const Epilogue& e, float acc, float c_old, float bias) {
  const float v = (e.beta != 0.0f) ? fmaf(e.alpha, acc, e.beta * c_old) : e.alpha * acc;
  return epi_activate(e.act, e.bias != nullptr ? v + bias : v);
}

// Store one element of D.
__device__ __forceinline__ void epi_store1(const Epilogue& e, int64_t row, int col, float v) {
  if (e.d_bf16)
    static_cast<__nv_bfloat16*>(e.D)[row * e.ldd + col] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(e.D)[row * e.ldd + col] = v;
}

// Store 8 consecutive elements of D starting at an aligned column.
__device__ __forceinline__ void epi_store8(const Epilogue& e, int64_t row, int col,
                                           const float (&v)[8]) {
  if (e.d_bf16) {
    __nv_bfloat162 h[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) h[q] = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(e.D) + row * e.ldd + col) =
        *reinterpret_cast<const uint4*>(h);
  } else {
    float* d = static_cast<float*>(e.D) + row * e.ldd + col;
    *reinterpret_cast<float4*>(d) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(d + 4) = make_float4(v[4], v[5], v[6], v[7]);
  }
}

}  // namespace g12
