// decode_noalloc.cu -- gemm_bf16gemm_decode_static: the decode-shaped bf16
// GEMM (M <= 16) for callers that cannot allocate device memory.
//
// gemm_bf16gemm allocates the decode kernel's scratch memory (split-K partial
// sums and per-column-group arrival counters) with cudaMalloc on its first
// decode-shaped call.  This entry point runs the same kernel with that scratch
// in a fixed-size array owned by the library instead: the array below is
// created when the library is loaded onto a device and lives until the
// process exits, so a call never allocates or frees anything.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace g12 {
namespace {

// Scratch capacity: 4 MiB per device.  The first kStaticCounters words are
// the arrival counters (one per 128-column group), the rest holds partial
// sums: CTAs x segment slots x 16 rows x 128 columns.  The partial sums bind
// first: with more column groups than SMs each CTA needs 3 slots up to twice
// as many groups as SMs (152 x 3 x 2048 floats on a 152-SM GB300) and 4
// beyond, which no longer fits -- so N <= 256 x SMs (38,912 on 152 SMs).
constexpr size_t kStaticScratchBytes = size_t{4} << 20;
constexpr int64_t kStaticCounters = 4096;
constexpr int64_t kStaticPartialFloats =
    static_cast<int64_t>(kStaticScratchBytes / 4) - kStaticCounters;

static __device__ __align__(256) uint32_t g_decode_scratch[kStaticScratchBytes / 4];

constexpr int kMaxDevices = 64;

// Device address of g_decode_scratch, looked up once per device with that
// device current.  In host code the symbol is only a host-side handle; the
// kernel must be given this address.
struct ScratchAddress {
  std::once_flag once;
  cudaError_t error = cudaSuccess;
  uint32_t* ptr = nullptr;
};
ScratchAddress g_scratch_addr[kMaxDevices];

uint32_t* scratch_on_current_device(gemm_status_t* status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *status = GEMM_ERR_UNSUPPORTED;
    return nullptr;
  }
  ScratchAddress& sa = g_scratch_addr[dev];
  std::call_once(sa.once, [&sa] {
    void* p = nullptr;
    sa.error = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (sa.error == cudaSuccess)
      sa.ptr = static_cast<uint32_t*>(p);
    else
      cudaGetLastError();
  });
  if (sa.error != cudaSuccess || sa.ptr == nullptr) {
    *status = GEMM_ERR_LAUNCH;
    return nullptr;
  }
  *status = GEMM_OK;
  return sa.ptr;
}

}  // namespace
}  // namespace g12

using namespace g12;

extern "C" gemm_status_t gemm_bf16gemm_decode_static(int64_t M, int64_t N, int64_t K,
                                                     float alpha, const void* A, int64_t lda,
                                                     const void* B, int64_t ldb, float beta,
                                                     float* C, int64_t ldc, void* stream) {
  gemm_status_t s = abi_check_args(M, N, K, lda, ldb, ldc);
  if (s != GEMM_OK) return s;
  if (M == 0 || N == 0) return GEMM_OK;
  if (C == nullptr || (reinterpret_cast<uintptr_t>(C) & 3u)) return GEMM_ERR_INVALID_VALUE;
  int num_sms = 0;
  uint32_t* err_word = nullptr;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (K == 0 || alpha == 0.0f) {
    s = abi_device(&num_sms, &err_word);
    if (s != GEMM_OK) return s;
    const cudaError_t e = launch_scale_c(static_cast<int>(M), static_cast<int>(N), beta, C, ldc, cs);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
  }
  if (A == nullptr || B == nullptr) return GEMM_ERR_INVALID_VALUE;
  if ((reinterpret_cast<uintptr_t>(A) & 1u) || (reinterpret_cast<uintptr_t>(B) & 1u))
    return GEMM_ERR_MISALIGNED;
  // Only the decode shape, with operands the TMA engine can describe.
  if (M > kDecBM || !abi_tma_ok(A, lda, 2) || !abi_tma_ok(B, ldb, 2)) return GEMM_ERR_UNSUPPORTED;
  s = abi_device(&num_sms, &err_word);
  if (s != GEMM_OK) return s;

  const int n = static_cast<int>(N), k = static_cast<int>(K);
  const int m = static_cast<int>(M);
  const int grid = decode_grid(m, n, k, num_sms);
  const int64_t counters = decode_counter_count(m, n);
  const int64_t partials = decode_workspace_floats(m, n, k, grid);
  if (counters > kStaticCounters || partials > kStaticPartialFloats) return GEMM_ERR_UNSUPPORTED;

  uint32_t* scratch = scratch_on_current_device(&s);
  if (scratch == nullptr) return s;

  CUtensorMap tmA, tmB;
  if (!abi_encode_bf16_2d(&tmA, A, K, M, lda, 64, kDecBM) ||
      !abi_encode_bf16_2d(&tmB, B, N, K, ldb, 64, static_cast<uint32_t>(decode_b_box_rows())))
    return GEMM_ERR_LAUNCH;

  DecodeArgs a{};
  a.M = static_cast<int>(M);
  a.N = n;
  a.K = k;
  a.epi = plain_epilogue(alpha, beta, C, ldc);
  a.err = err_word;
  a.cluster = decode_cluster(m, n, k, num_sms);
  // One CTA per column group, or clusters that add their partial sums in
  // shared memory: the kernel touches no scratch, so none is passed and
  // nothing is cleared (a memset between two launches would also keep this
  // launch from overlapping the previous kernel's last CTAs).  Only when the
  // column groups outnumber the SMs do runs of groups meet in the array.
  if (grid == decode_groups(n) || a.cluster > 1) {
    a.counters = nullptr;
    a.workspace = nullptr;
  } else {
    // The counters must start at zero.  The kernel leaves them at zero after
    // a completed launch, but a launch that gave up part-way may not have.
    if (cudaMemsetAsync(scratch, 0, counters * sizeof(uint32_t), cs) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_LAUNCH;
    }
    a.counters = scratch;
    a.workspace = reinterpret_cast<float*>(scratch + kStaticCounters);
  }
  const cudaError_t e = launch_tc_decode(a, &tmA, &tmB, grid, cs);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  return GEMM_OK;
}
