// api.cu -- the C ABI declared in include/gemm12.h: argument checks, kernel
// path selection, TMA tensor-map encoding, the decode workspace, the device
// error word, and the C <- beta*C kernel for the degenerate cases.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>

#include "../../include/gemm12.h"
#include "internal.h"

namespace g12 {

// Error word shared by every kernel of this library on a device; its device
// address is looked up once per device and passed to the kernels.
__device__ uint32_t g_error_word = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;

struct Scratch {
  float* ws = nullptr;
  int64_t ws_floats = 0;
  uint32_t* counters = nullptr;
  int64_t counter_count = 0;
  // Aligned copies of operands the TMA engine cannot describe (stage_operands).
  uint8_t* stage = nullptr;
  int64_t stage_bytes = 0;
};

struct DeviceState {
  std::once_flag once;
  cudaError_t init_error = cudaSuccess;
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
  uint32_t* err_word = nullptr;
  // Split-K scratch (partial sums + arrival counters) and operand staging
  // copies, one set per stream: calls on one stream are ordered by it, calls
  // on different streams never share a buffer.  Grown on demand, freed by
  // gemm_shutdown.
  std::mutex ws_mutex;
  std::map<void*, Scratch> scratch;
};

DeviceState g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

// Current device's state, initialised on first use.  Returns nullptr if
// there is no usable device.
DeviceState* device_state(gemm_status_t* status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *status = GEMM_ERR_UNSUPPORTED;
    return nullptr;
  }
  DeviceState& st = g_dev[dev];
  std::call_once(st.once, [&st, dev] {
    cudaError_t e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&st.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&st.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err_word), g_error_word);
    st.init_error = e;
    if (e != cudaSuccess) cudaGetLastError();
  });
  if (st.init_error != cudaSuccess) {
    *status = GEMM_ERR_UNSUPPORTED;
    return nullptr;
  }
  // The kernels are built for sm_103a only.
  if (!(st.cc_major == 10 && st.cc_minor == 3)) {
    *status = GEMM_ERR_UNSUPPORTED;
    return nullptr;
  }
  *status = GEMM_OK;
  return &st;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// TMA can describe a row-major matrix when its base is 16-byte aligned and
// its row pitch is a multiple of 16 bytes.
bool tma_ok(const void* base, int64_t ld, int elem_bytes) {
  return aligned16(base) && ((ld * elem_bytes) % 16 == 0);
}

// 2-D tensor map: dims {inner, outer}, row pitch ld elements, box {bx, by}.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, int elem_bytes, const void* base,
               int64_t inner, int64_t outer, int64_t ld, uint32_t bx, uint32_t by,
               CUtensorMapSwizzle swizzle) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * elem_bytes};
  cuuint32_t box[2] = {bx, by};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

gemm_status_t check_common(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                           int64_t ldc) {
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_INVALID_VALUE;
  if (lda > kMaxDim || ldb > kMaxDim || ldc > kMaxDim) return GEMM_ERR_INVALID_VALUE;
  if (lda < (K > 1 ? K : 1)) return GEMM_ERR_INVALID_VALUE;
  if (ldb < (N > 1 ? N : 1)) return GEMM_ERR_INVALID_VALUE;
  if (ldc < (N > 1 ? N : 1)) return GEMM_ERR_INVALID_VALUE;
  return GEMM_OK;
}

gemm_path_t select_path(bool bf16, int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                        int64_t lda, const void* B, int64_t ldb) {
  if (M == 0 || N == 0) return GEMM_PATH_NONE;
  if (K == 0 || alpha == 0.0f) return GEMM_PATH_SCALE_C;
  if (!bf16) {
    const bool a_tma = tma_ok(A, lda, 4);
    const bool b_tma = tma_ok(B, ldb, 4);
    return (a_tma && b_tma) ? GEMM_PATH_SIMT_TMA : GEMM_PATH_SIMT_GENERIC;
  }
  const bool tma = tma_ok(A, lda, 2) && tma_ok(B, ldb, 2);
  if (!tma) return GEMM_PATH_SIMT_BF16;
  if (decode_path(M, N, K)) return GEMM_PATH_TC_DECODE;
  return M <= kTcBM ? GEMM_PATH_TC_BF16 : GEMM_PATH_TC_BF16_PAIR;
}

gemm_status_t from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return GEMM_OK;
  cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? GEMM_ERR_NO_MEMORY : GEMM_ERR_LAUNCH;
}

gemm_status_t run_scale(int64_t M, int64_t N, float beta, float* C, int64_t ldc,
                        cudaStream_t stream) {
  return from_cuda(launch_scale_c(static_cast<int>(M), static_cast<int>(N), beta, C, ldc, stream));
}

int c_vec4_ok(const float* C, int64_t ldc) { return (aligned16(C) && (ldc % 4 == 0)) ? 1 : 0; }

// Whether `stream` is capturing into a CUDA graph.  A failed query counts as
// capturing, so that nothing is allocated.
bool capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return true;
  }
  return cs != cudaStreamCaptureStatusNone;
}

// Replaces *buf (of *have bytes) by a stream-ordered allocation of `bytes`
// on `stream`: the old buffer is released after the work already queued on
// the stream (its only user), the new one is ready for the work queued after
// this call.  Nothing waits on the host.
gemm_status_t regrow(void** buf, int64_t* have, int64_t bytes, cudaStream_t stream) {
  if (*buf != nullptr && cudaFreeAsync(*buf, stream) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  *buf = nullptr;
  *have = 0;
  if (cudaMallocAsync(buf, static_cast<size_t>(bytes), stream) != cudaSuccess) {
    cudaGetLastError();
    *buf = nullptr;
    return GEMM_ERR_NO_MEMORY;
  }
  *have = bytes;
  return GEMM_OK;
}

// The scratch area of `stream` on this device, grown to at least the given
// sizes (new counters start at zero).  Growth is stream-ordered on `stream`
// and never blocks the host.  Inside a stream capture nothing is allocated:
// a scratch area too small returns GEMM_ERR_NO_MEMORY, and the caller plans
// the launch without one.  Caller holds st.ws_mutex.
gemm_status_t ensure_scratch(DeviceState& st, cudaStream_t stream, int64_t floats,
                             int64_t counters, Scratch** out) {
  Scratch& sc = st.scratch[static_cast<void*>(stream)];
  *out = &sc;
  if (sc.ws_floats >= floats && sc.counter_count >= counters) return GEMM_OK;
  if (capturing(stream)) return GEMM_ERR_NO_MEMORY;
  if (sc.ws_floats < floats) {
    int64_t bytes = 0;
    const gemm_status_t s = regrow(reinterpret_cast<void**>(&sc.ws), &bytes,
                                   floats * static_cast<int64_t>(sizeof(float)), stream);
    sc.ws_floats = bytes / static_cast<int64_t>(sizeof(float));
    if (s != GEMM_OK) return s;
  }
  if (sc.counter_count < counters) {
    int64_t bytes = 0;
    const gemm_status_t s = regrow(reinterpret_cast<void**>(&sc.counters), &bytes,
                                   counters * static_cast<int64_t>(sizeof(uint32_t)), stream);
    sc.counter_count = bytes / static_cast<int64_t>(sizeof(uint32_t));
    if (s != GEMM_OK) return s;
    if (cudaMemsetAsync(sc.counters, 0, static_cast<size_t>(bytes), stream) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_LAUNCH;
    }
  }
  return GEMM_OK;
}

// The operand staging area of `stream` on this device, grown to at least
// `bytes` (stream-ordered, as ensure_scratch; nothing is allocated inside a
// stream capture).  Caller holds st.ws_mutex.
gemm_status_t ensure_stage(DeviceState& st, cudaStream_t stream, int64_t bytes, uint8_t** out) {
  Scratch& sc = st.scratch[static_cast<void*>(stream)];
  if (sc.stage_bytes < bytes) {
    if (capturing(stream)) return GEMM_ERR_NO_MEMORY;
    const gemm_status_t s = regrow(reinterpret_cast<void**>(&sc.stage), &sc.stage_bytes, bytes,
                                   stream);
    if (s != GEMM_OK) return s;
  }
  *out = sc.stage;
  return GEMM_OK;
}

// Whether a call first copies the operands the TMA engine cannot describe
// into an aligned staging buffer and then runs the TMA-fed kernels, instead
// of the generic-load kernels on the operands as given.  fp32: the TMA-fed
// kernel is ~20 % faster (3000x5000x1999: wide tiles and a stream-K tail
// instead of 128x128 tiles with 4-byte copies), so the copy -- one read and
// one write of the operand -- must be small next to the GEMM: at least 2^31
// FLOPs, and N >= 256 when A is copied (M >= 256 for B), which keeps the
// copy under ~2 % of the GEMM.  bf16: the tensor cores are ~25x faster than
// the CUDA-core fallback, so any tile-kernel shape of at least 2^24 FLOPs is
// copied (and then run on the tile kernels or the decode kernel, whichever
// automatic dispatch picks for the shape); M <= 16 keeps the fallback.
bool stage_wanted(bool bf16, int64_t M, int64_t N, int64_t K, bool a_ok, bool b_ok) {
  if (a_ok && b_ok) return false;
  const double flops = 2.0 * static_cast<double>(M) * static_cast<double>(N) *
                       static_cast<double>(K);
  if (!bf16) {
    if (flops < 2147483648.0) return false;
    if (!a_ok && N < 256) return false;
    if (!b_ok && M < 256) return false;
    return true;
  }
  return M > kDecBM && flops >= 16777216.0;
}

// Copies each operand the TMA engine cannot describe into this stream's
// staging area (rows padded to a 16-byte pitch, 256-byte aligned) and points
// A / B and lda / ldb at the copy.  The copy kernels are queued on `cs`
// ahead of the GEMM; the caller holds st.ws_mutex until the GEMM is queued.
// GEMM_ERR_NO_MEMORY: the staging area could not be grown, nothing changed.
gemm_status_t stage_operands(DeviceState& st, cudaStream_t cs, int elem_bytes, int64_t M,
                             int64_t N, int64_t K, const void*& A, int64_t& lda, const void*& B,
                             int64_t& ldb) {
  const int64_t per = 16 / elem_bytes;
  const bool sa = !tma_ok(A, lda, elem_bytes), sb = !tma_ok(B, ldb, elem_bytes);
  const int64_t lda2 = (K + per - 1) / per * per, ldb2 = (N + per - 1) / per * per;
  const int64_t bytes_a = sa ? (M * lda2 * elem_bytes + 255) / 256 * 256 : 0;
  const int64_t bytes_b = sb ? K * ldb2 * elem_bytes : 0;
  uint8_t* base = nullptr;
  const gemm_status_t s = ensure_stage(st, cs, bytes_a + bytes_b, &base);
  if (s != GEMM_OK) return s;
  if (sa) {
    const cudaError_t e = launch_stage_rows(elem_bytes, A, lda, base, lda2, M, K, st.num_sms, cs);
    if (e != cudaSuccess) return from_cuda(e);
    A = base;
    lda = lda2;
  }
  if (sb) {
    const cudaError_t e =
        launch_stage_rows(elem_bytes, B, ldb, base + bytes_a, ldb2, K, N, st.num_sms, cs);
    if (e != cudaSuccess) return from_cuda(e);
    B = base + bytes_a;
    ldb = ldb2;
  }
  return GEMM_OK;
}

// Work plan of the CUDA-core kernel for `a` (whole tiles, and the last wave's
// tiles split along k when that balances the SMs better).  A split plan needs
// this stream's scratch area; `lock` (on st->ws_mutex) is then held until the
// caller has launched.
}  // namespace

int tail_split(int items, int num_kb, int workers, double fixup_kb) {
  if (items <= 0 || workers <= 0 || num_kb <= 0) return 1;
  const int tail = items >= workers ? items % workers : items;
  if (tail == 0) return 1;
  int best_s = 1;
  double best = 1.0;
  for (int s = 2; s <= 8 && s * 4 <= num_kb; ++s) {
    const double rounds =
        static_cast<double>((static_cast<int64_t>(tail) * s + workers - 1) / workers);
    const double t = rounds / s + rounds * s * fixup_kb / num_kb;
    if (t < best - 1e-9) {
      best = t;
      best_s = s;
    }
  }
  return best_s;
}

// ------------------------------------------------ launch configuration
// Entries of the offline sweep's table (dispatch_table.inc).
struct TunedEntry {
  int is_bf16, log2_m, log2_n, log2_k;
  int kernel, split, group_m;
};
#include "dispatch_table.inc"

namespace {

int ceil_log2(int64_t x) {
  int b = 0;
  while ((int64_t{1} << b) < x) ++b;
  return b;
}

bool config_fields_valid(const gemm_config_t* c, bool bf16) {
  if (c == nullptr) return true;
  const bool kernel_ok = c->kernel == GEMM_KERNEL_AUTO || c->kernel == GEMM_KERNEL_SINGLE_CTA ||
                         (bf16 && c->kernel == GEMM_KERNEL_CTA_PAIR) ||
                         (!bf16 && c->kernel == GEMM_KERNEL_WIDE);
  const bool split_ok = (c->split >= 0 && c->split <= 8) || c->split == GEMM_SPLIT_STREAM;
  return kernel_ok && split_ok && c->group_m >= 0 && c->group_m <= 64;
}

// The tile-kernel configuration of one call: the sweep's table entry for the
// shape's class (on the GPU it was measured on), then every non-zero field of
// `user` on top.  Fields left 0 are decided by the planners (cost model).
TileConfig resolve_config(bool bf16, int64_t M, int64_t N, int64_t K, int num_sms,
                          const gemm_config_t* user, bool* from_table, bool use_table = true) {
  TileConfig c{GEMM_KERNEL_AUTO, 0, 0};
  bool table = false;
  if (use_table && num_sms == kTunedSms) {
    const int lm = ceil_log2(M), ln = ceil_log2(N), lk = ceil_log2(K);
    for (const TunedEntry& e : kTuned) {
      if (e.is_bf16 < 0) break;
      if (e.is_bf16 == (bf16 ? 1 : 0) && e.log2_m == lm && e.log2_n == ln && e.log2_k == lk) {
        c = TileConfig{e.kernel, e.split, e.group_m};
        table = true;
        break;
      }
    }
  }
  if (user != nullptr) {
    if (user->kernel != GEMM_KERNEL_AUTO) c.kernel = user->kernel;
    if (user->split != 0) c.split = user->split;
    if (user->group_m != 0) c.group_m = user->group_m;
  }
  if (from_table != nullptr) *from_table = table;
  return c;
}

}  // namespace

namespace {

// The plan `pl` with every tile run whole (no split, no stream-K tail): what
// a launch runs when it cannot have its scratch area.
SimtPlan simt_plan_whole(const SimtPlan& pl, int M, int N, int num_sms) {
  SimtPlan w = pl;
  const int tiles = ((M + kSimtBM - 1) / kSimtBM) * ((N + simt_bn(pl.wide) - 1) / simt_bn(pl.wide));
  w.full_items = tiles;
  w.split = 1;
  w.sk_workers = 0;
  w.grid = tiles < num_sms ? tiles : num_sms;
  w.ws_floats = 0;
  w.counters = 0;
  w.cluster = 0;
  return w;
}

// Fills the work plan fields of `a` from `pl`, with this stream's scratch
// area when the plan splits tiles.  Without scratch (inside a stream capture
// on a stream whose area is too small, or out of memory) `pl` becomes the
// plan of whole tiles: same kernel, same result bound.
gemm_status_t plan_simt(DeviceState* st, cudaStream_t cs, SimtArgs& a, SimtPlan& pl,
                        std::unique_lock<std::mutex>& lock) {
  a.ws = nullptr;
  a.counters = nullptr;
  if ((pl.split != 1 || pl.sk_workers != 0) && pl.cluster <= 1) {
    if (!lock.owns_lock()) lock.lock();
    Scratch* sc = nullptr;
    const gemm_status_t s = ensure_scratch(*st, cs, pl.ws_floats, pl.counters, &sc);
    if (s == GEMM_OK) {
      a.ws = sc->ws;
      a.counters = sc->counters;
    } else if (s == GEMM_ERR_NO_MEMORY) {
      pl = simt_plan_whole(pl, a.M, a.N, st->num_sms);
    } else {
      return s;
    }
  }
  a.full_items = pl.full_items;
  a.split = pl.split;
  a.sk_workers = pl.sk_workers;
  a.group_m = pl.group_m;
  a.cluster = pl.cluster;
  return GEMM_OK;
}

}  // namespace

// ------------------------------------------------------------ C <- beta*C
namespace {
__global__ void scale_c_kernel(int M, int N, float beta, float* C, int64_t ldc) {
  const int64_t total = static_cast<int64_t>(M) * N;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = e / N, j = e - i * N;
    float* c = C + i * ldc + j;
    *c = (beta == 0.0f) ? 0.0f : beta * *c;
  }
}
}  // namespace

cudaError_t launch_scale_c(int M, int N, float beta, float* C, int64_t ldc, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(M) * N;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  scale_c_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(M, N, beta, C, ldc);
  return cudaGetLastError();
}

// ------------------------------------------------ operand staging copy
namespace {
// Copies a rows x cols matrix of T (2- or 4-byte bit patterns, copied
// unchanged) from src (row pitch lds elements, any T-aligned address) to dst
// (row pitch ldd elements, ldd * sizeof(T) a multiple of 16, dst 16-byte
// aligned).  Item t of the grid-stride loop is the 16-byte piece t % pieces
// of row t / pieces: consecutive threads read consecutive elements of a row
// and write whole 16-byte pieces; columns past `cols` in a row's last piece
// are written as zero bits.
template <typename T>
__global__ void stage_rows_kernel(const T* __restrict__ src, int64_t lds, T* __restrict__ dst,
                                  int64_t ldd, int64_t rows, int64_t cols) {
  constexpr int kPer = 16 / static_cast<int>(sizeof(T));
  const int64_t pieces = (cols + kPer - 1) / kPer;
  const int64_t total = rows * pieces;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = t / pieces;
    const int64_t c0 = (t - r * pieces) * kPer;
    const T* s = src + r * lds + c0;
    union {
      T e[kPer];
      uint4 v;
    } u;
#pragma unroll
    for (int i = 0; i < kPer; ++i) u.e[i] = (c0 + i < cols) ? s[i] : T(0);
    *reinterpret_cast<uint4*>(dst + r * ldd + c0) = u.v;
  }
}
}  // namespace

cudaError_t launch_stage_rows(int elem_bytes, const void* src, int64_t lds, void* dst, int64_t ldd,
                              int64_t rows, int64_t cols, int num_sms, cudaStream_t stream) {
  const int64_t per = 16 / elem_bytes;
  const int64_t total = rows * ((cols + per - 1) / per);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (elem_bytes == 4)
    stage_rows_kernel<uint32_t><<<static_cast<int>(blocks), 256, 0, stream>>>(
        static_cast<const uint32_t*>(src), lds, static_cast<uint32_t*>(dst), ldd, rows, cols);
  else
    stage_rows_kernel<uint16_t><<<static_cast<int>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(src), lds, static_cast<uint16_t*>(dst), ldd, rows, cols);
  return cudaGetLastError();
}

Epilogue plain_epilogue(float alpha, float beta, float* C, int64_t ldc) {
  Epilogue e{};
  e.alpha = alpha;
  e.beta = beta;
  e.C = C;
  e.ldc = ldc;
  e.D = C;
  e.ldd = ldc;
  e.bias = nullptr;
  e.R = nullptr;
  e.ldr = 0;
  e.d_scale = 1.0f;
  e.amax = nullptr;
  e.act = kActNone;
  e.d_type = kOutF32;
  const int v = (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && ldc % 4 == 0 ? 1 : 0;
  e.c_vec4 = v;
  e.r_vec4 = 0;
  e.bias_vec4 = 0;
  e.d_vec = v;
  return e;
}

namespace {
// D <- act(beta * C + bias): the fused output stage when the product is empty
// (K == 0 or alpha == 0).
// The output stage of an empty product (K == 0 or alpha == 0): the
// accumulator is 0, so v = act(beta * C + bias) + R.
__global__ void epilogue_only_kernel(int M, int N, Epilogue e) {
  const int64_t total = static_cast<int64_t>(M) * N;
  float amax_acc = 0.0f;
  for (int64_t x = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; x < total;
       x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = x / N;
    const int j = static_cast<int>(x - i * N);
    // alpha never enters: alpha * 0 would be NaN for an infinite alpha
    float v = (e.beta != 0.0f) ? e.beta * e.C[i * e.ldc + j] : 0.0f;
    if (e.bias != nullptr) v += e.bias[j];
    v = epi_activate(e.act, v);
    if (e.R != nullptr) v += epi_residual(e, i, j);
    epi_track(e, amax_acc, v);
    epi_store1(e, i, j, v);
  }
  epi_flush_amax(e, amax_acc);
}
}  // namespace

cudaError_t launch_epilogue_only(int M, int N, const Epilogue& e, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(M) * N;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  epilogue_only_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(M, N, e);
  return cudaGetLastError();
}

// Shared pieces of the C ABI for entry points defined in other translation
// units (thin wrappers; the entry points above do not use them).
gemm_status_t abi_check_args(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                             int64_t ldc) {
  return check_common(M, N, K, lda, ldb, ldc);
}

bool abi_tma_ok(const void* base, int64_t ld, int elem_bytes) {
  return tma_ok(base, ld, elem_bytes);
}

bool abi_encode_bf16_2d(CUtensorMap* map, const void* base, int64_t inner, int64_t outer,
                        int64_t ld, uint32_t bx, uint32_t by) {
  return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer, ld, bx, by,
                   CU_TENSOR_MAP_SWIZZLE_128B);
}

gemm_status_t abi_device(int* num_sms, uint32_t** err_word) {
  gemm_status_t s;
  DeviceState* st = device_state(&s);
  if (st == nullptr) return s;
  *num_sms = st->num_sms;
  *err_word = st->err_word;
  return GEMM_OK;
}

}  // namespace g12

using namespace g12;

extern "C" {

int gemm_version(void) { return 100; }

const char* gemm_status_string(gemm_status_t s) {
  switch (s) {
    case GEMM_OK: return "GEMM_OK: success";
    case GEMM_ERR_INVALID_VALUE: return "GEMM_ERR_INVALID_VALUE: bad size, leading dimension or pointer";
    case GEMM_ERR_MISALIGNED: return "GEMM_ERR_MISALIGNED: bf16 pointer not 2-byte aligned";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED: no sm_103a device or unsupported size";
    case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH: kernel launch or CUDA runtime error";
    case GEMM_ERR_DEVICE_TIMEOUT: return "GEMM_ERR_DEVICE_TIMEOUT: a bounded device wait ran out";
    case GEMM_ERR_NO_MEMORY: return "GEMM_ERR_NO_MEMORY: workspace allocation failed";
  }
  return "unknown gemm status";
}

gemm_path_t gemm_select_path(int is_bf16, int64_t M, int64_t N, int64_t K, float alpha,
                             const void* A, int64_t lda, const void* B, int64_t ldb) {
  if (check_common(M, N, K, lda, ldb, N > 1 ? N : 1) != GEMM_OK) return GEMM_PATH_NONE;
  const bool bf16 = is_bf16 != 0;
  gemm_path_t p = select_path(bf16, M, N, K, alpha, A, lda, B, ldb);
  if (p == GEMM_PATH_TC_BF16 || p == GEMM_PATH_TC_BF16_PAIR) {
    // the tile kernel automatic dispatch runs (the sweep's table may pick
    // single CTAs for M > 128); without a usable device, the M rule
    gemm_status_t s;
    DeviceState* st = device_state(&s);
    if (st != nullptr) {
      const TileConfig tc = resolve_config(true, M, N, K, st->num_sms, nullptr, nullptr);
      const TcPlan pl = tc_plan(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                                st->num_sms, &tc);
      p = pl.pair ? GEMM_PATH_TC_BF16_PAIR : GEMM_PATH_TC_BF16;
    }
  }
  const int eb = bf16 ? 2 : 4;
  if ((p == GEMM_PATH_SIMT_GENERIC || p == GEMM_PATH_SIMT_BF16) &&
      stage_wanted(bf16, M, N, K, tma_ok(A, lda, eb), tma_ok(B, ldb, eb)))
    return bf16 ? GEMM_PATH_TC_STAGED : GEMM_PATH_SIMT_STAGED;
  return p;
}

int gemm_split_parts(int is_bf16, int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return 0;
  gemm_status_t s;
  DeviceState* st = device_state(&s);
  if (st == nullptr) return 0;
  if (M == 0 || N == 0 || K == 0) return 1;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  const TileConfig tc = resolve_config(is_bf16 != 0, M, N, K, st->num_sms, nullptr, nullptr);
  if (is_bf16) {
    if (decode_path(M, N, K)) return 1;
    return tc_plan_max_parts(tc_plan(m, n, k, st->num_sms, &tc), m, n, k);
  }
  return simt_plan_max_parts(simt_plan(m, n, k, st->num_sms, &tc, true), m, n, k);
}

int gemm_split_cluster(int is_bf16, int64_t M, int64_t N, int64_t K, const gemm_config_t* cfg) {
  const bool bf16 = is_bf16 != 0;
  if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX ||
      !config_fields_valid(cfg, bf16))
    return 0;
  gemm_status_t s;
  DeviceState* st = device_state(&s);
  if (st == nullptr) return 0;
  if (M == 0 || N == 0 || K == 0) return 1;
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  const TileConfig tc = resolve_config(bf16, M, N, K, st->num_sms, cfg, nullptr);
  if (bf16) {
    // the decode kernel (automatic dispatch only) plans its own clusters
    if (decode_path(M, N, K) && (cfg == nullptr || cfg->kernel == GEMM_KERNEL_AUTO)) return 1;
    TcPlan pl = tc_plan(m, n, k, st->num_sms, &tc);
    Epilogue plain{};
    plain.alpha = 1.0f;
    plain.d_scale = 1.0f;
    return tc_use_cluster(pl, m, n, plain) ? pl.cluster : 1;
  }
  SimtPlan pl = simt_plan(m, n, k, st->num_sms, &tc, true);
  return simt_use_cluster(pl, m, n) ? pl.cluster : 1;
}

gemm_status_t gemm_quantization(int64_t M, int64_t N, int64_t BM, int64_t BN, int64_t num_sms,
                                int64_t ctas_per_sm, gemm_quantization_t* out) {
  if (out == nullptr || M < 0 || N < 0 || BM <= 0 || BN <= 0 || num_sms <= 0 || ctas_per_sm <= 0)
    return GEMM_ERR_INVALID_VALUE;
  gemm_quantization_t q{};
  q.tiles_m = (M + BM - 1) / BM;
  q.tiles_n = (N + BN - 1) / BN;
  q.tiles = q.tiles_m * q.tiles_n;
  q.covered_m = q.tiles_m * BM;
  q.covered_n = q.tiles_n * BN;
  q.per_wave = num_sms * ctas_per_sm;
  q.waves = (q.tiles + q.per_wave - 1) / q.per_wave;
  if (q.tiles == 0) {
    q.useful_fraction = 1.0;
    q.wave_efficiency = 1.0;
  } else {
    q.useful_fraction = (static_cast<double>(M) * static_cast<double>(N)) /
                        (static_cast<double>(q.covered_m) * static_cast<double>(q.covered_n));
    q.wave_efficiency =
        static_cast<double>(q.tiles) / (static_cast<double>(q.waves) * q.per_wave);
  }
  *out = q;
  return GEMM_OK;
}

static gemm_status_t sgemm_impl(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                                int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                                int64_t ldc, const gemm_config_t* cfg, void* stream) {
  if (!config_fields_valid(cfg, false)) return GEMM_ERR_INVALID_VALUE;
  gemm_status_t s = check_common(M, N, K, lda, ldb, ldc);
  if (s != GEMM_OK) return s;
  const gemm_path_t path = select_path(false, M, N, K, alpha, A, lda, B, ldb);
  if (path == GEMM_PATH_NONE) return GEMM_OK;
  if (C == nullptr) return GEMM_ERR_INVALID_VALUE;
  if (path != GEMM_PATH_SCALE_C && (A == nullptr || B == nullptr)) return GEMM_ERR_INVALID_VALUE;
  if ((reinterpret_cast<uintptr_t>(C) & 3u) ||
      (path != GEMM_PATH_SCALE_C && ((reinterpret_cast<uintptr_t>(A) & 3u) ||
                                     (reinterpret_cast<uintptr_t>(B) & 3u))))
    return GEMM_ERR_INVALID_VALUE;
  DeviceState* st = device_state(&s);
  if (st == nullptr) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (path == GEMM_PATH_SCALE_C) return run_scale(M, N, beta, C, ldc, cs);

  // Held from staging (if any) until the kernel is queued: the staging copy
  // and the split-K scratch of this stream must not be regrown meanwhile.
  std::unique_lock<std::mutex> lock(st->ws_mutex, std::defer_lock);
  if (path == GEMM_PATH_SIMT_GENERIC &&
      stage_wanted(false, M, N, K, tma_ok(A, lda, 4), tma_ok(B, ldb, 4))) {
    lock.lock();
    const void* sa = A;
    const void* sb = B;
    s = stage_operands(*st, cs, 4, M, N, K, sa, lda, sb, ldb);
    if (s == GEMM_OK) {
      A = static_cast<const float*>(sa);
      B = static_cast<const float*>(sb);
    } else if (s != GEMM_ERR_NO_MEMORY) {
      return s;
    }
    // No memory for the copies: the generic-load kernel reads the operands
    // as given.
  }

  SimtArgs a{};
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.alpha = alpha;
  a.beta = beta;
  a.A = A;
  a.lda = lda;
  a.B = B;
  a.ldb = ldb;
  a.C = C;
  a.ldc = ldc;
  a.c_vec4 = c_vec4_ok(C, ldc);
  a.err = st->err_word;
  const TileConfig tc = resolve_config(false, M, N, K, st->num_sms, cfg, nullptr);
  CUtensorMap tmA, tmB;
  LoadMode ma = kLoadCpAsyncF32, mb = kLoadCpAsyncF32;
  if (tma_ok(A, lda, 4) &&
      encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, A, K, M, lda, kSimtBK, kSimtBM,
                CU_TENSOR_MAP_SWIZZLE_128B))
    ma = kLoadTma;
  // The wide tile runs only with both operands on TMA; its B box is 256 wide.
  SimtPlan pl = simt_plan(a.M, a.N, a.K, st->num_sms, &tc, ma == kLoadTma && tma_ok(B, ldb, 4));
  if (tma_ok(B, ldb, 4)) {
    if (encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, B, N, K, ldb, simt_bn(pl.wide),
                  kSimtBK, CU_TENSOR_MAP_SWIZZLE_NONE)) {
      mb = kLoadTma;
    } else if (pl.wide) {
      pl = simt_plan(a.M, a.N, a.K, st->num_sms, &tc, false);
      if (encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, B, N, K, ldb, simt_bn(false),
                    kSimtBK, CU_TENSOR_MAP_SWIZZLE_NONE))
        mb = kLoadTma;
    }
  }
  // Tiles that all fit in one round add their k-parts through distributed
  // shared memory.
  if (ma == kLoadTma && mb == kLoadTma) simt_use_cluster(pl, a.M, a.N);
  s = plan_simt(st, cs, a, pl, lock);
  if (s != GEMM_OK) return s;
  return from_cuda(launch_simt(a, pl, ma, mb, ma == kLoadTma ? &tmA : nullptr,
                               mb == kLoadTma ? &tmB : nullptr, cs));
}

gemm_status_t gemm_sgemm(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                         int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                         int64_t ldc, void* stream) {
  return sgemm_impl(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, nullptr, stream);
}

gemm_status_t gemm_sgemm_config(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                                int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                                int64_t ldc, const gemm_config_t* cfg, void* stream) {
  return sgemm_impl(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, cfg, stream);
}

// Runs the tensor-core path (tile kernel or decode kernel) of a bf16 GEMM
// whose operands TMA can describe, with output stage `epi`.
// `lock` (on st->ws_mutex) is taken here when the launch needs this stream's
// scratch, unless the caller already holds it (operands staged).
static gemm_status_t run_bf16_tensor_core(DeviceState* st, gemm_path_t path, int64_t M, int64_t N,
                                          int64_t K, const void* A, int64_t lda, const void* B,
                                          int64_t ldb, const Epilogue& epi, cudaStream_t cs,
                                          const gemm_config_t* cfg,
                                          std::unique_lock<std::mutex>& lock) {
  CUtensorMap tmA, tmB;
  if (path == GEMM_PATH_TC_BF16 || path == GEMM_PATH_TC_BF16_PAIR) {
    TcArgs a{};
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.epi = epi;
    a.err = st->err_word;
    const TileConfig tc = resolve_config(true, M, N, K, st->num_sms, cfg, nullptr);
    // The plain output stage with beta == 0 writes whole tiles by TMA when
    // D's base and row pitch allow a tensor map.
    const bool tma_out = !tc_fused(epi) && epi.beta == 0.0f && tma_ok(epi.D, epi.ldd, 4);
    TcPlan pl = tc_plan(a.M, a.N, a.K, st->num_sms, &tc, tma_out);
    // Tiles that all fit in one round add their k-parts through distributed
    // shared memory (single-CTA kernel).
    tc_use_cluster(pl, a.M, a.N, epi);
    const uint32_t b_rows = static_cast<uint32_t>(tc_b_box_rows(pl.pair));
    if (!encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, K, M, lda, 64, kTcBM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, N, K, ldb, 64, b_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B))
      return GEMM_ERR_LAUNCH;
    TcPlan run = pl;
    a.ws = nullptr;
    a.counters = nullptr;
    if ((pl.split > 1 || pl.sk_workers > 0) && pl.cluster <= 1) {
      // Split items: the stream's scratch stays locked until the launch is
      // queued, so no other thread can regrow it underneath.  Without scratch
      // (inside a stream capture, or out of memory) every item runs whole.
      if (!lock.owns_lock()) lock.lock();
      Scratch* sc = nullptr;
      const gemm_status_t s = ensure_scratch(*st, cs, pl.ws_floats, pl.counters, &sc);
      if (s == GEMM_OK) {
        a.ws = sc->ws;
        a.counters = sc->counters;
      } else if (s == GEMM_ERR_NO_MEMORY) {
        const TileConfig whole{pl.pair ? GEMM_KERNEL_CTA_PAIR : GEMM_KERNEL_SINGLE_CTA, 1,
                               pl.group_m};
        run = tc_plan(a.M, a.N, a.K, st->num_sms, &whole, tma_out);
      } else {
        return s;
      }
    }
    a.full_items = run.full_items;
    a.split = run.split;
    a.sk_workers = run.sk_workers;
    a.group_m = run.group_m;
    a.cluster = run.cluster;
    CUtensorMap tmD;
    a.d_tma = 0;
    if (tma_out && encode_2d(&tmD, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, epi.D, N, M, epi.ldd,
                             kTcStoreBoxCols, kTcStoreBoxRows, CU_TENSOR_MAP_SWIZZLE_128B))
      a.d_tma = 1;
    return from_cuda(launch_tc_bf16(a, run, &tmA, &tmB, a.d_tma ? &tmD : nullptr, cs));
  }
  // GEMM_PATH_TC_DECODE
  if (!encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, K, M, lda, 64,
                 static_cast<uint32_t>(decode_rows(static_cast<int>(M))),
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, N, K, ldb, 64,
                 static_cast<uint32_t>(decode_b_box_rows()), CU_TENSOR_MAP_SWIZZLE_128B))
    return GEMM_ERR_LAUNCH;
  const int grid =
      decode_grid(static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), st->num_sms);
  DecodeArgs a{};
  a.M = static_cast<int>(M);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.epi = epi;
  a.err = st->err_word;
  a.cluster = decode_cluster(a.M, a.N, a.K, st->num_sms);
  // One CTA per column group, or clusters that exchange their partial sums
  // in shared memory: no scratch is touched.
  if (grid == decode_groups(a.N) || a.cluster > 1) {
    a.workspace = nullptr;
    a.counters = nullptr;
    return from_cuda(launch_tc_decode(a, &tmA, &tmB, grid, cs));
  }
  if (!lock.owns_lock()) lock.lock();
  Scratch* sc = nullptr;
  gemm_status_t s = ensure_scratch(*st, cs, decode_workspace_floats(a.M, a.N, a.K, grid),
                                   decode_counter_count(a.M, a.N), &sc);
  if (s == GEMM_ERR_NO_MEMORY) {
    // No scratch for the runs of column groups (inside a stream capture, or
    // out of memory): the single-CTA tile kernel with whole tiles needs none.
    const gemm_config_t whole{GEMM_KERNEL_SINGLE_CTA, 1, 0};
    return run_bf16_tensor_core(st, GEMM_PATH_TC_BF16, M, N, K, A, lda, B, ldb, epi, cs, &whole,
                                lock);
  }
  if (s != GEMM_OK) return s;
  a.workspace = sc->ws;
  a.counters = sc->counters;
  return from_cuda(launch_tc_decode(a, &tmA, &tmB, grid, cs));
}

static gemm_status_t bf16gemm_impl(int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                                   int64_t lda, const void* B, int64_t ldb, float beta, float* C,
                                   int64_t ldc, const gemm_config_t* cfg, void* stream) {
  if (!config_fields_valid(cfg, true)) return GEMM_ERR_INVALID_VALUE;
  gemm_status_t s = check_common(M, N, K, lda, ldb, ldc);
  if (s != GEMM_OK) return s;
  gemm_path_t path = select_path(true, M, N, K, alpha, A, lda, B, ldb);
  // a pinned kernel runs the tile kernels, also for decode shapes
  if (path == GEMM_PATH_TC_DECODE && cfg != nullptr && cfg->kernel != GEMM_KERNEL_AUTO)
    path = cfg->kernel == GEMM_KERNEL_CTA_PAIR ? GEMM_PATH_TC_BF16_PAIR : GEMM_PATH_TC_BF16;
  if (path == GEMM_PATH_NONE) return GEMM_OK;
  if (C == nullptr) return GEMM_ERR_INVALID_VALUE;
  if (reinterpret_cast<uintptr_t>(C) & 3u) return GEMM_ERR_INVALID_VALUE;
  if (path != GEMM_PATH_SCALE_C) {
    if (A == nullptr || B == nullptr) return GEMM_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(A) & 1u) || (reinterpret_cast<uintptr_t>(B) & 1u))
      return GEMM_ERR_MISALIGNED;
  }
  DeviceState* st = device_state(&s);
  if (st == nullptr) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (path == GEMM_PATH_SCALE_C) return run_scale(M, N, beta, C, ldc, cs);

  std::unique_lock<std::mutex> lock(st->ws_mutex, std::defer_lock);
  if (path == GEMM_PATH_SIMT_BF16 &&
      stage_wanted(true, M, N, K, tma_ok(A, lda, 2), tma_ok(B, ldb, 2))) {
    lock.lock();
    s = stage_operands(*st, cs, 2, M, N, K, A, lda, B, ldb);
    if (s == GEMM_OK)
      path = select_path(true, M, N, K, alpha, A, lda, B, ldb);  // on the aligned copies
    else if (s != GEMM_ERR_NO_MEMORY)
      return s;
    // No memory for the copies: the CUDA-core kernel reads the operands as
    // given.
  }

  if (path == GEMM_PATH_SIMT_BF16) {
    SimtArgs a{};
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.alpha = alpha;
    a.beta = beta;
    a.A = A;
    a.lda = lda;
    a.B = B;
    a.ldb = ldb;
    a.C = C;
    a.ldc = ldc;
    a.c_vec4 = c_vec4_ok(C, ldc);
    a.err = st->err_word;
    // the CUDA-core kernel's table entries are the fp32 ones
    gemm_config_t simt_cfg{GEMM_KERNEL_AUTO, cfg ? cfg->split : 0, cfg ? cfg->group_m : 0};
    const TileConfig tc = resolve_config(false, M, N, K, st->num_sms, &simt_cfg, nullptr);
    SimtPlan pl = simt_plan(a.M, a.N, a.K, st->num_sms, &tc, false);
    s = plan_simt(st, cs, a, pl, lock);
    if (s != GEMM_OK) return s;
    return from_cuda(launch_simt(a, pl, kLoadConvertBf16, kLoadConvertBf16, nullptr, nullptr,
                                 cs));
  }
  return run_bf16_tensor_core(st, path, M, N, K, A, lda, B, ldb,
                              plain_epilogue(alpha, beta, C, ldc), cs, cfg, lock);
}

gemm_status_t gemm_bf16gemm(int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                            int64_t lda, const void* B, int64_t ldb, float beta, float* C,
                            int64_t ldc, void* stream) {
  return bf16gemm_impl(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, nullptr, stream);
}

gemm_status_t gemm_bf16gemm_config(int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                                   int64_t lda, const void* B, int64_t ldb, float beta, float* C,
                                   int64_t ldc, const gemm_config_t* cfg, void* stream) {
  return bf16gemm_impl(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, cfg, stream);
}

static gemm_status_t get_config(int is_bf16, int64_t M, int64_t N, int64_t K, gemm_config_t* out,
                                int* from_table, bool use_table) {
  if (out == nullptr || M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return GEMM_ERR_INVALID_VALUE;
  gemm_status_t s;
  DeviceState* st = device_state(&s);
  if (st == nullptr) return s;
  *out = gemm_config_t{GEMM_KERNEL_AUTO, 0, 0};
  if (from_table != nullptr) *from_table = 0;
  if (is_bf16 && decode_path(M, N, K)) return GEMM_OK;  // the decode kernel plans itself
  bool table = false;
  const TileConfig tc =
      resolve_config(is_bf16 != 0, M, N, K, st->num_sms, nullptr, &table, use_table);
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  if (is_bf16) {
    const TcPlan pl = tc_plan(m, n, k, st->num_sms, &tc);
    *out = gemm_config_t{pl.pair ? GEMM_KERNEL_CTA_PAIR : GEMM_KERNEL_SINGLE_CTA,
                         pl.sk_workers > 0 ? GEMM_SPLIT_STREAM : pl.split, pl.group_m};
  } else {
    const SimtPlan pl = simt_plan(m, n, k, st->num_sms, &tc, true);
    *out = gemm_config_t{pl.wide ? GEMM_KERNEL_WIDE : GEMM_KERNEL_SINGLE_CTA,
                         pl.sk_workers > 0 ? GEMM_SPLIT_STREAM : pl.split, pl.group_m};
  }
  if (from_table != nullptr) *from_table = table ? 1 : 0;
  return GEMM_OK;
}

gemm_status_t gemm_get_config(int is_bf16, int64_t M, int64_t N, int64_t K, gemm_config_t* out,
                              int* from_table) {
  return get_config(is_bf16, M, N, K, out, from_table, true);
}

gemm_status_t gemm_get_model_config(int is_bf16, int64_t M, int64_t N, int64_t K,
                                    gemm_config_t* out) {
  return get_config(is_bf16, M, N, K, out, nullptr, false);
}

gemm_status_t gemm_bf16gemm_fused(int64_t M, int64_t N, int64_t K, float alpha, const void* A,
                                  int64_t lda, const void* B, int64_t ldb,
                                  const gemm_output_t* out, void* stream) {
  if (out == nullptr) return GEMM_ERR_INVALID_VALUE;
  const gemm_output_t& o = *out;
  if (o.act != GEMM_ACT_NONE && o.act != GEMM_ACT_RELU && o.act != GEMM_ACT_GELU)
    return GEMM_ERR_INVALID_VALUE;
  if (o.d_type != GEMM_OUT_F32 && o.d_type != GEMM_OUT_BF16 && o.d_type != GEMM_OUT_F8E4M3 &&
      o.d_type != GEMM_OUT_S8)
    return GEMM_ERR_INVALID_VALUE;
  const int64_t min_ld = N > 1 ? N : 1;
  gemm_status_t s = check_common(M, N, K, lda, ldb, o.beta != 0.0f ? o.ldc : min_ld);
  if (s != GEMM_OK) return s;
  if (o.ldd < min_ld || o.ldd > kMaxDim) return GEMM_ERR_INVALID_VALUE;
  if (o.residual != nullptr && (o.ldr < min_ld || o.ldr > kMaxDim)) return GEMM_ERR_INVALID_VALUE;
  const gemm_path_t path = select_path(true, M, N, K, alpha, A, lda, B, ldb);
  if (path == GEMM_PATH_NONE) return GEMM_OK;
  const int d_bytes = o.d_type == GEMM_OUT_F32 ? 4 : (o.d_type == GEMM_OUT_BF16 ? 2 : 1);
  auto misaligned = [](const void* p, uintptr_t mask) {
    return (reinterpret_cast<uintptr_t>(p) & mask) != 0;
  };
  if (o.D == nullptr || misaligned(o.D, static_cast<uintptr_t>(d_bytes - 1)))
    return GEMM_ERR_INVALID_VALUE;
  if (o.beta != 0.0f && (o.C == nullptr || misaligned(o.C, 3u))) return GEMM_ERR_INVALID_VALUE;
  if (o.bias != nullptr && misaligned(o.bias, 3u)) return GEMM_ERR_INVALID_VALUE;
  if (o.residual != nullptr && misaligned(o.residual, 3u)) return GEMM_ERR_INVALID_VALUE;
  if (o.amax != nullptr && misaligned(o.amax, 3u)) return GEMM_ERR_INVALID_VALUE;
  if (path != GEMM_PATH_SCALE_C) {
    if (A == nullptr || B == nullptr) return GEMM_ERR_INVALID_VALUE;
    if (misaligned(A, 1u) || misaligned(B, 1u)) return GEMM_ERR_MISALIGNED;
  }
  DeviceState* st = device_state(&s);
  if (st == nullptr) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  Epilogue epi{};
  epi.alpha = alpha;
  epi.beta = o.beta;
  epi.C = o.C;
  epi.ldc = o.ldc;
  epi.D = o.D;
  epi.ldd = o.ldd;
  epi.bias = o.bias;
  epi.R = o.residual;
  epi.ldr = o.ldr;
  epi.d_scale = o.d_scale;
  epi.amax = o.amax;
  epi.act = o.act;
  epi.d_type = o.d_type;  // gemm_out_t and the kernels' kOut* agree
  epi.c_vec4 = (o.beta != 0.0f) ? c_vec4_ok(o.C, o.ldc) : 0;
  epi.r_vec4 = (o.residual != nullptr) ? c_vec4_ok(o.residual, o.ldr) : 0;
  epi.bias_vec4 = (o.bias != nullptr && aligned16(o.bias)) ? 1 : 0;
  // 8-element stores: 16 bytes for fp32 (two float4) and bf16, 8 for bytes
  const uintptr_t vec_mask = d_bytes == 1 ? 7u : 15u;
  epi.d_vec = !misaligned(o.D, vec_mask) && (o.ldd % (d_bytes == 4 ? 4 : 8) == 0) ? 1 : 0;
  if (path == GEMM_PATH_SCALE_C)
    return from_cuda(launch_epilogue_only(static_cast<int>(M), static_cast<int>(N), epi, cs));
  std::unique_lock<std::mutex> lock(st->ws_mutex, std::defer_lock);
  gemm_path_t run_path = path;
  if (path == GEMM_PATH_SIMT_BF16) {
    // The output stage lives only in the tensor-core kernels: operands the
    // TMA engine cannot describe are always staged here, whatever the size.
    lock.lock();
    s = stage_operands(*st, cs, 2, M, N, K, A, lda, B, ldb);
    if (s != GEMM_OK) return s;
    run_path = select_path(true, M, N, K, alpha, A, lda, B, ldb);  // on the aligned copies
  }
  return run_bf16_tensor_core(st, run_path, M, N, K, A, lda, B, ldb, epi, cs, nullptr, lock);
}

gemm_status_t gemm_bf16gemm_epilogue(int64_t M, int64_t N, int64_t K, float alpha,
                                     const void* A, int64_t lda, const void* B, int64_t ldb,
                                     float beta, const float* C, int64_t ldc, const float* bias,
                                     int act, void* D, int64_t ldd, int d_type, void* stream) {
  if (d_type != GEMM_OUT_F32 && d_type != GEMM_OUT_BF16) return GEMM_ERR_INVALID_VALUE;
  gemm_output_t o{};
  o.beta = beta;
  o.C = C;
  o.ldc = ldc;
  o.bias = bias;
  o.act = act;
  o.residual = nullptr;
  o.ldr = 0;
  o.d_scale = 1.0f;
  o.amax = nullptr;
  o.D = D;
  o.ldd = ldd;
  o.d_type = d_type;
  return gemm_bf16gemm_fused(M, N, K, alpha, A, lda, B, ldb, &o, stream);
}

gemm_status_t gemm_check_device_error(void* stream) {
  gemm_status_t s;
  DeviceState* st = device_state(&s);
  if (st == nullptr) return s;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  uint32_t word = 0;
  if (cudaMemcpy(&word, st->err_word, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  if (word == 0) return GEMM_OK;
  const uint32_t zero = 0;
  cudaMemcpy(st->err_word, &zero, sizeof zero, cudaMemcpyHostToDevice);
  // A split launch that gave up may have left arrival counters non-zero, on
  // whichever stream it ran (the word does not say): let every stream's
  // work finish, then reset them all -- clearing counters under a split
  // kernel still running on another stream would break that kernel.
  {
    std::lock_guard<std::mutex> lock(st->ws_mutex);
    cudaDeviceSynchronize();
    for (auto& kv : st->scratch)
      if (kv.second.counters)
        cudaMemset(kv.second.counters, 0, kv.second.counter_count * sizeof(uint32_t));
    cudaDeviceSynchronize();
  }
  cudaGetLastError();
  return GEMM_ERR_DEVICE_TIMEOUT;
}

gemm_status_t gemm_shutdown(void) {
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_OK;
  }
  int cur = 0;
  cudaGetDevice(&cur);
  gemm_status_t result = GEMM_OK;
  for (int d = 0; d < n && d < kMaxDevices; ++d) {
    DeviceState& st = g_dev[d];
    std::lock_guard<std::mutex> lock(st.ws_mutex);
    if (st.scratch.empty()) continue;
    if (cudaSetDevice(d) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
      cudaGetLastError();
      result = GEMM_ERR_LAUNCH;
      continue;
    }
    // Stream-ordered allocations, released on the legacy stream once the
    // device is idle (the streams they were made on may no longer exist).
    for (auto& kv : st.scratch) {
      if (kv.second.ws) cudaFreeAsync(kv.second.ws, 0);
      if (kv.second.counters) cudaFreeAsync(kv.second.counters, 0);
      if (kv.second.stage) cudaFreeAsync(kv.second.stage, 0);
    }
    st.scratch.clear();
    if (cudaDeviceSynchronize() != cudaSuccess) {
      cudaGetLastError();
      result = GEMM_ERR_LAUNCH;
    }
  }
  cudaSetDevice(cur);
  return result;
}

gemm_status_t gemm_release_stream(void* stream) {
  gemm_status_t s;
  DeviceState* st = device_state(&s);
  if (st == nullptr) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(st->ws_mutex);
  auto it = st->scratch.find(stream);
  if (it == st->scratch.end()) return GEMM_OK;
  if (capturing(cs)) return GEMM_ERR_INVALID_VALUE;
  Scratch& sc = it->second;
  gemm_status_t result = GEMM_OK;
  for (void* p : {static_cast<void*>(sc.ws), static_cast<void*>(sc.counters),
                  static_cast<void*>(sc.stage)})
    if (p != nullptr && cudaFreeAsync(p, cs) != cudaSuccess) {
      cudaGetLastError();
      result = GEMM_ERR_LAUNCH;
    }
  st->scratch.erase(it);
  return result;
}

}  // extern "C"
