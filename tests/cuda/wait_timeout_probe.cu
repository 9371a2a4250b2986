// Test-only probe: the bounded mbarrier wait every kernel of the library uses
// (mbar_wait in ptx.cuh), run on a barrier that nothing ever completes.  The
// wait must end after the library's time limit, report the timeout in the
// error word and return, leaving the CUDA context usable.
#include <cuda_runtime.h>

#include <chrono>
#include <cstdint>

#include "../../dense_gemm_12_gb300/csrc/ptx.cuh"

__device__ uint32_t g_probe_err;

__global__ void wait_for_nothing(int* result) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    g12::mbar_init(&bar, 1);  // expects one arrival; none is ever made
    abort_flag = 0;
    g12::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool completed = g12::mbar_wait(&bar, 0, &abort_flag, &g_probe_err);
    result[0] = completed ? 1 : 0;
    result[1] = abort_flag;
  }
}

// Runs the probe once; returns 0 on success of every CUDA call.
extern "C" int probe_wait_timeout(int* completed, int* aborted, unsigned* err_word,
                                  double* seconds) {
  int* d = nullptr;
  unsigned zero = 0;
  if (cudaMalloc(&d, 2 * sizeof(int)) != cudaSuccess) return 1;
  if (cudaMemcpyToSymbol(g_probe_err, &zero, sizeof zero) != cudaSuccess) return 2;
  const auto t0 = std::chrono::steady_clock::now();
  wait_for_nothing<<<1, 32>>>(d);
  if (cudaGetLastError() != cudaSuccess) return 3;
  if (cudaDeviceSynchronize() != cudaSuccess) return 4;
  *seconds = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
  int h[2];
  if (cudaMemcpy(h, d, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return 5;
  if (cudaMemcpyFromSymbol(err_word, g_probe_err, sizeof(unsigned)) != cudaSuccess) return 6;
  cudaFree(d);
  *completed = h[0];
  *aborted = h[1];
  return 0;
}
