// epilogue.cuh -- the fused output stage of the bf16 kernels:
//
//     v[i][j] = act(alpha * acc[i][j] + beta * C[i][j] + bias[j]) + R[i][j]
//     D[i][j] = convert(d_scale * v[i][j])       amax = max |v[i][j]|
//
// written as fp32, bf16, fp8 e4m3 or int8 ("Tiled matrix multiplication",
// "Implementation notes": fuse bias, activation, residual, scaling and
// fp8/int8 quantisation while the tile is still in registers, which saves a
// full read and write of C).  The plain GEMM is the special case act = none,
// no bias, no residual, d_scale = 1, D = C in fp32.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

namespace g12 {

enum : int { kActNone = 0, kActRelu = 1, kActGelu = 2 };
enum : int { kOutF32 = 0, kOutBf16 = 1, kOutE4M3 = 2, kOutS8 = 3 };

struct Epilogue {
  float alpha, beta;
  const float* C;      // read when beta != 0 (ldc)
  int64_t ldc;
  void* D;             // output (ldd); may be C itself when fp32 with ldd == ldc
  int64_t ldd;
  const float* bias;   // length N, or nullptr
  const float* R;      // residual added after the activation (ldr), or nullptr
  int64_t ldr;
  float d_scale;       // multiplies v before the conversion to D's type
  float* amax;         // raised to max |v| over this launch's outputs, or nullptr
  int act;             // kActNone / kActRelu / kActGelu
  int d_type;          // kOutF32 / kOutBf16 / kOutE4M3 / kOutS8
  int c_vec4;          // C rows may be read as aligned float4
  int r_vec4;          // residual rows may be read as aligned float4
  int bias_vec4;       // bias may be read as aligned float4
  int d_vec;           // D rows may be written 8 (and 4) elements at a time (aligned)
};

__device__ __forceinline__ float epi_gelu(float x) {
  return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
}

__device__ __forceinline__ float epi_activate(int act, float x) {
  if (act == kActRelu) return x > 0.0f ? x : 0.0f;
  if (act == kActGelu) return epi_gelu(x);
  return x;
}

// Bias of column col (0 without a bias).  Callers load every bias and
// residual value they need before their first store to D: a load placed after
// a store to a possibly aliasing address cannot be issued early and costs a
// full memory round trip.
__device__ __forceinline__ float epi_bias(const Epilogue& e, int col) {
  return e.bias != nullptr ? e.bias[col] : 0.0f;
}

__device__ __forceinline__ float epi_residual(const Epilogue& e, int64_t row, int col) {
  return e.R != nullptr ? e.R[row * e.ldr + col] : 0.0f;
}

// v of one element (before d_scale).
__device__ __forceinline__ float epi_value(const Epilogue& e, float acc, float c_old, float bias,
                                           float res) {
  const float v = (e.beta != 0.0f) ? fmaf(e.alpha, acc, e.beta * c_old) : e.alpha * acc;
  const float a = epi_activate(e.act, e.bias != nullptr ? v + bias : v);
  return e.R != nullptr ? a + res : a;
}

// Running maximum of |v| for the amax output (NaN never raises it).
__device__ __forceinline__ void epi_track(const Epilogue& e, float& amax_acc, float v) {
  if (e.amax != nullptr) amax_acc = fmaxf(amax_acc, fabsf(v));
}

// Fold every lane's running maximum into *amax: one atomic per warp.  All 32
// lanes of the warp call it together.  Non-negative floats order like their
// bit patterns, so an unsigned maximum is the float maximum.
__device__ __forceinline__ void epi_flush_amax(const Epilogue& e, float amax_acc) {
  if (e.amax == nullptr) return;
  const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(amax_acc));
  if ((threadIdx.x & 31) == 0 && m != 0u) atomicMax(reinterpret_cast<unsigned*>(e.amax), m);
}

// Conversions of d_scale * v.  e4m3: CUDA's round-to-nearest-even conversion
// with saturation to the largest finite value (+-448); int8: round half to
// even, saturate to [-128, 127], NaN -> 0.
__device__ __forceinline__ uint8_t epi_to_e4m3(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint8_t epi_to_s8(float x) {
  if (x != x) return 0;
  const float r = fminf(fmaxf(rintf(x), -128.0f), 127.0f);
  return static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(r)));
}

__device__ __forceinline__ uint8_t epi_to_byte(const Epilogue& e, float v) {
  const float x = e.d_scale * v;
  return e.d_type == kOutE4M3 ? epi_to_e4m3(x) : epi_to_s8(x);
}

// Store one element of D.
__device__ __forceinline__ void epi_store1(const Epilogue& e, int64_t row, int col, float v) {
  const int64_t at = row * e.ldd + col;
  if (e.d_type == kOutF32)
    static_cast<float*>(e.D)[at] = e.d_scale * v;
  else if (e.d_type == kOutBf16)
    static_cast<__nv_bfloat16*>(e.D)[at] = __float2bfloat16_rn(e.d_scale * v);
  else
    static_cast<uint8_t*>(e.D)[at] = epi_to_byte(e, v);
}

// Store 4 consecutive elements of D starting at a column that is a multiple
// of 4 (requires d_vec): one 16-, 8- or 4-byte store.
__device__ __forceinline__ void epi_store4(const Epilogue& e, int64_t row, int col,
                                           const float (&v)[4]) {
  const int64_t at = row * e.ldd + col;
  const float s = e.d_scale;
  if (e.d_type == kOutF32) {
    *reinterpret_cast<float4*>(static_cast<float*>(e.D) + at) =
        make_float4(s * v[0], s * v[1], s * v[2], s * v[3]);
  } else if (e.d_type == kOutBf16) {
    __nv_bfloat162 h[2] = {__floats2bfloat162_rn(s * v[0], s * v[1]),
                           __floats2bfloat162_rn(s * v[2], s * v[3])};
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(e.D) + at) =
        *reinterpret_cast<const uint2*>(h);
  } else {
    uint32_t w = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) w |= static_cast<uint32_t>(epi_to_byte(e, v[q])) << (8 * q);
    *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(e.D) + at) = w;
  }
}

// Store 8 consecutive elements of D starting at a column that is a multiple
// of 8 (requires d_vec).
__device__ __forceinline__ void epi_store8(const Epilogue& e, int64_t row, int col,
                                           const float (&v)[8]) {
  const int64_t at = row * e.ldd + col;
  if (e.d_type == kOutF32) {
    float* d = static_cast<float*>(e.D) + at;
    const float s = e.d_scale;
    *reinterpret_cast<float4*>(d) = make_float4(s * v[0], s * v[1], s * v[2], s * v[3]);
    *reinterpret_cast<float4*>(d + 4) = make_float4(s * v[4], s * v[5], s * v[6], s * v[7]);
  } else if (e.d_type == kOutBf16) {
    __nv_bfloat162 h[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      h[q] = __floats2bfloat162_rn(e.d_scale * v[2 * q], e.d_scale * v[2 * q + 1]);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(e.D) + at) =
        *reinterpret_cast<const uint4*>(h);
  } else {
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int q = 0; q < 8; ++q) w[q >> 2] |= static_cast<uint32_t>(epi_to_byte(e, v[q])) << (8 * (q & 3));
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(e.D) + at) = make_uint2(w[0], w[1]);
  }
}

}  // namespace g12
