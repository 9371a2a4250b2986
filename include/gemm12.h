/*
 * gemm12.h -- C ABI of the GB300 (sm_103a) dense GEMM library.
 *
 * Operation (both entry points):
 *
 *     C  <-  alpha * (A x B) + beta * C
 *
 * with A an M x K matrix, B a K x N matrix and C an M x N matrix, as defined
 * in "GEMM Worklog I: Naive to Tiled" (opening equation) and used as the
 * single SGEMM call of "A GEMM Kernel, Step by Step" ("The ladder we are
 * climbing").  The pages' own host function takes (M, N, K, A, B, C, stream)
 * with dense row-major operands ("Tiled matrix multiplication", section
 * "Code"); this interface adds the scalars and leading dimensions.
 *
 * Conventions shared by every entry point below:
 *
 *  Layout     All matrices are ROW-MAJOR.  Element (i, k) of A is at
 *             A[i * lda + k], element (k, j) of B at B[k * ldb + j] and
 *             element (i, j) of C at C[i * ldc + j].  Requirements:
 *             M, N, K >= 0; lda >= max(1, K); ldb >= max(1, N);
 *             ldc >= max(1, N).  Each of M, N, K, lda, ldb, ldc must be below
 *             2^31.  A violation returns GEMM_ERR_INVALID_VALUE and launches
 *             nothing.
 *  Pointers   A, B and C are DEVICE pointers (global memory of the current
 *             device), owned by the caller; the library never frees them.
 *             NULL is accepted only for an operand that is not read:
 *             A and B when M, N or K is 0 or alpha == 0; C when M or N is 0.
 *  Scalars    beta == 0: C is write-only (its old contents, NaN included, do
 *             not reach the result).  alpha == 0 or K == 0: A and B are not
 *             read and C <- beta * C (C <- 0 when beta == 0 too).  M == 0 or
 *             N == 0: nothing is launched.
 *  Alignment  None is required beyond the element size.  Operands whose
 *             address or leading dimension the tensor-memory-accelerator
 *             (TMA) copy engine cannot describe (base not 16-byte aligned,
 *             row pitch not a multiple of 16 bytes) are, for large enough
 *             problems, first copied into an aligned per-stream staging
 *             buffer (one read and one write of the operand) so that the
 *             TMA-fed kernels run; smaller problems take generic-load
 *             kernels on the operands as given (see gemm_select_path).
 *             Either way this changes speed, not the result's error bound.
 *             A bf16 pointer that is not 2-byte aligned returns
 *             GEMM_ERR_MISALIGNED.
 *  Aliasing   C must not overlap A or B (not checked).
 *  Streams    `stream` is a cudaStream_t (NULL = the legacy default stream).
 *             Calls are asynchronous: they enqueue kernels and return.  Launch
 *             failures are reported as GEMM_ERR_LAUNCH; errors raised later
 *             by the device are reported by the CUDA runtime at the next
 *             synchronising call, and a kernel's bounded waits that ran out
 *             are reported by gemm_check_device_error().
 *  Threads    Entry points may be called from several host threads on
 *             different streams.
 *  Memory     Calls whose work is split along k through global memory --
 *             the decode kernel of gemm_bf16gemm (small M) when N exceeds
 *             128 x the SM count (narrower decode shapes exchange partial
 *             sums in shared memory and need none), and gemm_sgemm /
 *             gemm_bf16gemm when the last wave of output tiles is split to
 *             balance the SMs -- need scratch memory (partial sums and
 *             arrival counters).  The
 *             library allocates it per device and per stream the first time a
 *             call on that stream needs it (or more of it), keeps and reuses
 *             it, and frees it in gemm_release_stream(stream) or
 *             gemm_shutdown(); calls on different streams never share
 *             scratch, calls on one stream are ordered by it.  The staging
 *             copies of operands the TMA engine cannot describe (see
 *             Alignment) live in a second per-stream buffer, kept, grown and
 *             freed the same way (at most the size of the copied operands,
 *             rows padded to 16 bytes).  Allocation is stream-ordered
 *             (cudaMallocAsync / cudaFreeAsync on `stream`, from the
 *             device's default memory pool): growing never blocks the host,
 *             the old buffer is released after the work already queued on
 *             the stream.
 *             Without the scratch it needs -- out of memory, or inside a
 *             stream capture (CUDA graph), where the library allocates
 *             nothing -- a call still runs: split tiles run whole instead
 *             (same kernel), a decode launch that needs scratch runs on the
 *             single-CTA tile kernel, and an operand that cannot be staged
 *             is read by the generic-load kernels.  The result stays within
 *             the same error bound but may differ in the last bits from a
 *             call that had its scratch; to capture exactly the eager plan,
 *             make one call of the shape on the stream before capturing it.
 *             gemm_bf16gemm_fused, whose output stage exists only in the
 *             tensor-core kernels, returns GEMM_ERR_NO_MEMORY instead when
 *             an operand needs staging and no staging buffer can be had.
 *             The first call of the library on a device (it looks up the
 *             device's properties) must come before any capture.  See also
 *             gemm_bf16gemm_decode_static, which allocates nothing.
 */
#ifndef GEMM12_H
#define GEMM12_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_VALUE = 1,   /* bad size, leading dimension or NULL   */
    GEMM_ERR_MISALIGNED = 2,      /* bf16 pointer not 2-byte aligned        */
    GEMM_ERR_UNSUPPORTED = 3,     /* no sm_103a device, or size too large   */
    GEMM_ERR_LAUNCH = 4,          /* kernel launch or CUDA runtime error    */
    GEMM_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device wait ran out          */
    GEMM_ERR_NO_MEMORY = 6        /* workspace allocation failed            */
} gemm_status_t;

/*
 * gemm_sgemm -- fp32 SGEMM, C <- alpha*(A x B) + beta*C.
 *
 * A: M x K fp32 (lda), B: K x N fp32 (ldb), C: M x N fp32 (ldc), all device
 * pointers, row-major.  Products are accumulated in fp32 with fused
 * multiply-adds on the CUDA cores (the register-tiled outer-product scheme of
 * "Tiled matrix multiplication", "How it works", and of "A GEMM Kernel, Step
 * by Step", "Rungs four and five" and "The last rung").  The error against the
 * exact result is within 2e-6 * sqrt(K) of |alpha|*(|A||B|)_ij +
 * |beta|*|C_ij| per element; on integer-valued inputs whose partial sums stay
 * below 2^24 in magnitude the result is exact.
 */
gemm_status_t gemm_sgemm(int64_t M, int64_t N, int64_t K, float alpha,
                         const float *A, int64_t lda,
                         const float *B, int64_t ldb,
                         float beta, float *C, int64_t ldc, void *stream);

/*
 * gemm_bf16gemm -- bf16 inputs, fp32 accumulation, fp32 output:
 * C <- alpha*(A x B) + beta*C.
 *
 * A: M x K bf16 (__nv_bfloat16 / uint16 bit patterns, lda), B: K x N bf16
 * (ldb), C: M x N fp32 (ldc), device pointers, row-major.  The tensor-core
 * path ("Tiled matrix multiplication", "How it works": tensor cores fed from
 * shared memory by asynchronous copies) runs on the 5th-generation tensor
 * cores with the accumulator in tensor memory.  Small M takes the
 * bandwidth-bound decode kernel (the "decode GEMV (M <= 16)" case of "Tiled
 * matrix multiplication", "Avoid when", widened here to every M <= 32, to
 * 32 < M <= 128 up to N = 16384, and to 128 < M <= 512 while ceil(N / 128)
 * x ceil(M / 64) <= 128 (160 for K >= 4096) -- above 64 rows as row blocks
 * of 64 -- where it measured faster than the tile kernels; gemm_select_path
 * reports GEMM_PATH_TC_DECODE), which splits K across CTAs
 * ("Split-K" in the same page's "Variants and alternatives") and reduces the
 * partial sums in a fixed order, so results are deterministic.  Error bound:
 * 8e-3 of |alpha|*(|A||B|)_ij + |beta|*|C_ij| against the exact product of the
 * bf16 values.  With beta == 0, a 16-byte aligned C and ldc a multiple of 4,
 * the tile kernels write C through TMA stores (faster when the output
 * dominates, e.g. K <= 1024); the results are the same either way.
 */
gemm_status_t gemm_bf16gemm(int64_t M, int64_t N, int64_t K, float alpha,
                            const void *A, int64_t lda,
                            const void *B, int64_t ldb,
                            float beta, float *C, int64_t ldc, void *stream);

/* Activations and output types of gemm_bf16gemm_fused / _epilogue. */
typedef enum {
    GEMM_ACT_NONE = 0,   /* identity                                           */
    GEMM_ACT_RELU = 1,   /* max(x, 0)                                          */
    GEMM_ACT_GELU = 2    /* x * Phi(x) = 0.5 x (1 + erf(x / sqrt(2)))           */
} gemm_act_t;

typedef enum {
    GEMM_OUT_F32 = 0,    /* D holds fp32                                       */
    GEMM_OUT_BF16 = 1,   /* D holds bf16, rounded to nearest even              */
    GEMM_OUT_F8E4M3 = 2, /* D holds fp8 E4M3 (1 sign, 4 exponent bits with bias
                            7, 3 mantissa bits; no infinities; largest finite
                            value 448; S.1111.111 is NaN), rounded to nearest
                            even, saturated to +-448; NaN stays NaN          */
    GEMM_OUT_S8 = 3      /* D holds int8: rounded half to even, saturated to
                            [-128, 127]; NaN becomes 0                        */
} gemm_out_t;

/*
 * Output stage of gemm_bf16gemm_fused.  With P = A x B (fp32 accumulation):
 *
 *     v[i][j] = act(alpha * P[i][j] + beta * C[i][j] + bias[j]) + R[i][j]
 *     D[i][j] = convert_{d_type}(d_scale * v[i][j])
 *     *amax   = max(*amax, max over i, j of |v[i][j]|)
 *
 * "Tiled matrix multiplication" ("Implementation notes", fusing the
 * epilogue): bias, activation, residual, scaling and fp8/int8 quantisation
 * are applied while the tile is still in registers.  All matrices row-major;
 * every pointer is a device pointer owned by the caller.
 */
typedef struct {
    float beta;            /* weight of C; C is not read when beta == 0      */
    const float *C;        /* M x N fp32 (ldc >= max(1, N)), 4-byte aligned;
                              may be NULL when beta == 0                     */
    int64_t ldc;
    const float *bias;     /* N fp32 values (4-byte aligned) or NULL         */
    int act;               /* a gemm_act_t                                   */
    const float *residual; /* R: M x N fp32 (ldr >= max(1, N)), 4-byte
                              aligned, added after the activation; or NULL   */
    int64_t ldr;
    float d_scale;         /* multiplies v before the conversion (1 = none)  */
    float *amax;           /* one fp32 (4-byte aligned) raised to the largest
                              |v| over the output (NaN values never raise
                              it; the caller sets the start value, e.g. 0),
                              or NULL                                       */
    void *D;               /* M x N output of type d_type, aligned to its
                              element size                                   */
    int64_t ldd;           /* >= max(1, N)                                   */
    int d_type;            /* a gemm_out_t                                   */
} gemm_output_t;

/*
 * gemm_bf16gemm_fused -- bf16 GEMM (A, B, lda, ldb as in gemm_bf16gemm) with
 * the output stage `out` (see gemm_output_t).  The same tensor-core kernels
 * as gemm_bf16gemm run (including the decode kernel for small M).
 * Aliasing: D may be C itself only when d_type is GEMM_OUT_F32 and
 * ldd == ldc, and may be the residual itself only when d_type is
 * GEMM_OUT_F32 and ldd == ldr (each output element is read before it is
 * written, by the thread that writes it); otherwise D must not overlap A, B,
 * C, bias, residual or amax.  Errors: out == NULL, an unknown act or d_type,
 * a NULL or misaligned D, C (beta != 0), bias, residual or amax, or a leading
 * dimension below max(1, N) return GEMM_ERR_INVALID_VALUE.  Operands the TMA
 * engine cannot describe (base not 16-byte aligned, pitch not a multiple of
 * 16 bytes) are always copied into the stream's staging buffer first (see
 * Memory), whatever the size, since the output stage exists only in the
 * tensor-core kernels.  K == 0 or alpha == 0:
 * v = act(beta * C + bias) + R (alpha is not used).  Accuracy: v carries the
 * bf16 GEMM's bound on the pre-activation value times the activation's
 * largest slope (1 for none and ReLU, 1.13 for GELU); D adds the rounding of
 * its conversion.
 */
gemm_status_t gemm_bf16gemm_fused(int64_t M, int64_t N, int64_t K, float alpha,
                                  const void *A, int64_t lda,
                                  const void *B, int64_t ldb,
                                  const gemm_output_t *out, void *stream);

/*
 * gemm_bf16gemm_epilogue -- gemm_bf16gemm_fused without residual, scaling or
 * amax, and with fp32 or bf16 output only:
 *
 *     D[i][j] = act(alpha * (A x B)[i][j] + beta * C[i][j] + bias[j])
 *
 * "Tiled matrix multiplication" ("Implementation notes"; "Efficiency",
 * epilogue fusion): bias, activation and the narrowing to bf16 happen while
 * the tile is still in registers, which saves a full read and write of the
 * output.  A, B, lda, ldb as in gemm_bf16gemm.  C: M x N fp32 (ldc), read only
 * when beta != 0 (may be NULL otherwise).  bias: N fp32 values, or NULL for
 * none.  act: a gemm_act_t.  D: M x N output of type d_type (a gemm_out_t),
 * leading dimension ldd >= max(1, N), 4-byte aligned for fp32 and 2-byte for
 * bf16; D may be C itself only when d_type is GEMM_OUT_F32 and ldd == ldc,
 * otherwise D must not overlap A, B, C or bias.  The same tensor-core kernels
 * as gemm_bf16gemm run (including the decode kernel for small M); operands
 * the TMA engine cannot describe are staged as in gemm_bf16gemm_fused; an
 * unknown act or a d_type other than GEMM_OUT_F32 and GEMM_OUT_BF16 returns
 * GEMM_ERR_INVALID_VALUE.  K == 0 or alpha == 0: D = act(beta*C +
 * bias).  Error bound: the bf16 GEMM's bound on the pre-activation value,
 * times the activation's largest slope (1 for none and ReLU, 1.13 for GELU),
 * plus the bf16 rounding of D when d_type is GEMM_OUT_BF16.
 */
gemm_status_t gemm_bf16gemm_epilogue(int64_t M, int64_t N, int64_t K, float alpha,
                                     const void *A, int64_t lda,
                                     const void *B, int64_t ldb,
                                     float beta, const float *C, int64_t ldc,
                                     const float *bias, int act,
                                     void *D, int64_t ldd, int d_type, void *stream);

/*
 * gemm_bf16gemm_decode_static -- the decode-shaped bf16 GEMM of gemm_bf16gemm
 * (M <= 16; same arguments, same kernel, same results) for callers that must
 * not allocate device memory: for example a serving process that reserves all
 * of its device memory at start-up and allows no allocation on its request
 * path, or code that runs inside a memory allocator's own callbacks, where
 * calling cudaMalloc again is not allowed.  The GEMM pages have no
 * counterpart of this entry point; it exists for such callers only.
 *
 * Instead of allocating its split-K scratch (partial sums and per-column-group
 * arrival counters) the call uses one fixed array of 4 MiB that the library
 * holds on every device it is loaded onto, until the process exits.  It calls
 * no cudaMalloc or cudaFree.  Limit: the array holds the partial sums of
 * up to twice as many 128-column groups as the device has SMs, so
 * N <= 256 x SMs (N <= 38,912 on a 152-SM GB300; any K).  Larger N returns
 * GEMM_ERR_UNSUPPORTED, as do M > 16 and operands the TMA engine cannot
 * describe (base not 16-byte aligned, or a row pitch that is not a multiple
 * of 16 bytes) -- use gemm_bf16gemm for those.  M == 0 or N == 0 does
 * nothing; K == 0 or alpha == 0 computes C <- beta*C.
 *
 * The array is used only when the column groups outnumber the SMs
 * (N > 128 x SMs); fewer groups run with no scratch at all, as in
 * gemm_bf16gemm.  Every call on a device shares that one array, and a call
 * that uses it first clears its counters (an asynchronous memset on
 * `stream`).  Calls whose
 * work overlaps on the GPU -- on different streams, or from different host
 * threads -- race on the array and give wrong results: serialise them.  The
 * first call on each device looks up the array's device address (once, with
 * that device current); make that first call before any stream capture.
 */
gemm_status_t gemm_bf16gemm_decode_static(int64_t M, int64_t N, int64_t K, float alpha,
                                          const void *A, int64_t lda,
                                          const void *B, int64_t ldb,
                                          float beta, float *C, int64_t ldc, void *stream);

/*
 * gemm_release_stream -- frees the scratch and staging buffers the library
 * keeps for `stream` on the current device (see Memory above), stream-ordered
 * after the work already queued on that stream; a later call on the stream
 * allocates them again.  Call it before destroying a stream that has run
 * GEMMs, so that the buffers do not outlive it.  Returns GEMM_OK (also when
 * the stream has none), GEMM_ERR_INVALID_VALUE while the stream is being
 * captured, GEMM_ERR_LAUNCH if a free could not be queued.
 */
gemm_status_t gemm_release_stream(void *stream);

/* Static, NUL-terminated description of a status code (never NULL). */
const char *gemm_status_string(gemm_status_t status);

/*
 * gemm_check_device_error -- synchronise `stream`, then read and clear the
 * current device's error word, which the kernels set when one of their
 * bounded waits (on an mbarrier or on another CTA) runs out.  Returns
 * GEMM_ERR_DEVICE_TIMEOUT if it was set, GEMM_ERR_LAUNCH if the
 * synchronisation itself failed, else GEMM_OK.  When the word was set, a
 * launch that gave up may have left split-K arrival counters non-zero on
 * whichever stream it ran: the call then synchronises the whole device
 * (every stream's GEMMs finish first) and resets the counters of every
 * stream's scratch, so that later split launches start clean.
 */
gemm_status_t gemm_check_device_error(void *stream);

/* Free the scratch and staging buffers of every stream on every device
 * (see Memory above).  Call with no GEMM in flight. */
gemm_status_t gemm_shutdown(void);

/* Kernel paths a call can take (reported by gemm_select_path). */
typedef enum {
    GEMM_PATH_NONE = 0,           /* M == 0 or N == 0: nothing launched     */
    GEMM_PATH_SCALE_C = 1,        /* alpha == 0 or K == 0: C <- beta*C      */
    GEMM_PATH_SIMT_TMA = 2,       /* fp32 CUDA-core kernel, TMA operands    */
    GEMM_PATH_SIMT_GENERIC = 3,   /* fp32 CUDA-core kernel, generic loads   */
    GEMM_PATH_TC_BF16 = 4,        /* bf16 tensor-core (tcgen05) kernel,
                                     one CTA per 128x256 tile (M <= 128,
                                     and small problems: see below)        */
    GEMM_PATH_TC_DECODE = 5,      /* bf16 tensor-core split-K decode kernel */
    GEMM_PATH_SIMT_BF16 = 6,      /* bf16 operands TMA cannot describe:
                                     widened to fp32 on the CUDA cores     */
    GEMM_PATH_TC_BF16_PAIR = 7,   /* bf16 tensor-core kernel on CTA pairs:
                                     two SMs per 256x256 tile (M > 128,
                                     unless single CTAs: see below)        */
    GEMM_PATH_SIMT_STAGED = 8,    /* fp32 operands TMA cannot describe are
                                     first copied into an aligned staging
                                     buffer, then GEMM_PATH_SIMT_TMA       */
    GEMM_PATH_TC_STAGED = 9       /* bf16 operands TMA cannot describe are
                                     first copied into an aligned staging
                                     buffer, then the tcgen05 tile kernels
                                     (GEMM_PATH_TC_BF16 or _PAIR)          */
} gemm_path_t;

/*
 * gemm_select_path -- host-only: the kernel path a call with these arguments
 * takes.  `is_bf16` selects gemm_bf16gemm's rules instead of gemm_sgemm's.
 * Operands the TMA engine cannot describe are staged (GEMM_PATH_SIMT_STAGED,
 * GEMM_PATH_TC_STAGED) when the copy is cheap next to the GEMM: fp32 with at
 * least 2^31 FLOPs (2*M*N*K) and N >= 256 if A is copied, M >= 256 if B is;
 * bf16 with M > 16 and at least 2^24 FLOPs.  Otherwise GEMM_PATH_SIMT_GENERIC
 * or GEMM_PATH_SIMT_BF16 (also when the staging buffer cannot be allocated).
 * Between the two bf16 tile kernels it reports the one automatic dispatch
 * runs on the current device (CTA pairs for large problems -- at least 128
 * tiles of 128 x 256 with K > 2048, or 256 with K > 512 -- unless the sweep's
 * table says otherwise); with no usable device, the one-CTA kernel for
 * M <= 128 and CTA pairs above.
 * Pointers are only inspected for alignment, never dereferenced.  Returns
 * GEMM_PATH_NONE (and writes nothing) for arguments the call would reject.
 */
gemm_path_t gemm_select_path(int is_bf16, int64_t M, int64_t N, int64_t K,
                             float alpha, const void *A, int64_t lda,
                             const void *B, int64_t ldb);

/*
 * gemm_split_parts -- host-only diagnostics: into how many k-ranges the tile
 * kernel for an M x N x K problem cuts each work item of the persistent
 * grid's last round ("A GEMM Kernel, Step by Step": the partial last wave of
 * "The fringe and the last wave", filled by the split-K of "What is left").
 * 1 means no item is split.  Under the stream-K tail (GEMM_SPLIT_STREAM)
 * the tail items are cut into differing numbers of k-ranges; the largest is
 * reported.  `is_bf16`
 * selects gemm_bf16gemm's tensor-core tile kernels instead of gemm_sgemm's
 * CUDA-core kernel; the decode kernel (bf16, small M) plans its
 * own split and reports 1 here.  Returns 0 for negative sizes or when there
 * is no usable sm_103a device (the plan depends on its SM count).
 */
int gemm_split_parts(int is_bf16, int64_t M, int64_t N, int64_t K);

/*
 * Launch configurations of the tile kernels ("A GEMM Kernel, Step by Step",
 * "Six parameters, found by search": the best tiling depends on the card and
 * the shape, so it is searched for rather than derived).  Tile sizes, stages
 * and warp layout are fixed per kernel at build time; what can change per
 * call is which kernel runs, how the last round's work items are cut along k
 * and the raster order.  Automatic dispatch takes these from a table written
 * by an offline sweep on this GPU (dense_gemm_12_gb300/tune.py), keyed by
 * ceil(log2) of M, N and K, and falls back to a cost model for shapes the
 * table does not hold.
 */
typedef enum {
    GEMM_KERNEL_AUTO = 0,        /* the library chooses                        */
    GEMM_KERNEL_SINGLE_CTA = 1,  /* one CTA per tile: the CUDA-core kernel's
                                    128 x 128 tiles (fp32), the tcgen05
                                    kernel's 128 x 256 tiles (bf16)            */
    GEMM_KERNEL_CTA_PAIR = 2,    /* bf16 only: two CTAs of a cluster per
                                    256 x 256 tile (tcgen05 cta_group::2)      */
    GEMM_KERNEL_WIDE = 3         /* fp32 only: the CUDA-core kernel on
                                    128 x 256 tiles (8 x 16 values per thread:
                                    fewer shared-memory reads per FMA, half
                                    as many tiles)                             */
} gemm_kernel_t;

/* gemm_config_t.split value: stream-K tail.  The k-blocks of all work items
 * past the last whole round are dealt out evenly to the persistent workers
 * (CTAs, or CTA pairs) in contiguous ranges that may cross an item boundary;
 * each item's partial sums are added in k order by the last range to finish
 * it.  bf16: used when those k-blocks are at least as many as the workers,
 * else the equal split of the cost model runs instead. */
#define GEMM_SPLIT_STREAM (-1)

typedef struct {
    int kernel;   /* a gemm_kernel_t                                          */
    int split;    /* k-ranges per work item of the persistent grid's last
                     round: 0 = automatic, 1 = none, 2..8 (capped at one
                     k-block per range), or GEMM_SPLIT_STREAM                 */
    int group_m;  /* raster order: work items walk column by column through
                     groups of this many item rows; 0 = automatic, 1..64     */
} gemm_config_t;

/*
 * gemm_sgemm_config / gemm_bf16gemm_config -- gemm_sgemm / gemm_bf16gemm with
 * the launch configuration pinned by cfg (cfg == NULL or all fields 0: the
 * same as the plain call).  The result is the same GEMM within the same bound
 * for every configuration (bit-identical where the sums are exact).  A pinned
 * bf16 kernel always runs the tcgen05 tile kernels, also for small M (the
 * decode kernel runs only under GEMM_KERNEL_AUTO).  The fp32 path has two
 * tile widths (GEMM_KERNEL_SINGLE_CTA: 128 x 128, GEMM_KERNEL_WIDE:
 * 128 x 256); GEMM_KERNEL_CTA_PAIR is invalid there, and GEMM_KERNEL_WIDE
 * is invalid for bf16.  The fields are ignored on
 * the paths without tiles (M, N, K or alpha zero: nothing to configure).
 * Errors: fields out of range give
 * GEMM_ERR_INVALID_VALUE; otherwise as the plain calls.  Operands that TMA
 * cannot describe are staged as in the plain calls; unstaged, bf16 ones run
 * on the CUDA cores (128 x 128 tiles), where only split and group_m apply,
 * and fp32 ones always on 128 x 128 tiles.
 */
gemm_status_t gemm_sgemm_config(int64_t M, int64_t N, int64_t K, float alpha,
                                const float *A, int64_t lda,
                                const float *B, int64_t ldb,
                                float beta, float *C, int64_t ldc,
                                const gemm_config_t *cfg, void *stream);
gemm_status_t gemm_bf16gemm_config(int64_t M, int64_t N, int64_t K, float alpha,
                                   const void *A, int64_t lda,
                                   const void *B, int64_t ldb,
                                   float beta, float *C, int64_t ldc,
                                   const gemm_config_t *cfg, void *stream);

/*
 * gemm_get_config -- host-only: the configuration automatic dispatch uses for
 * an M x N x K problem on the current device (every field resolved; for the
 * bf16 shapes of the decode kernel, kernel is GEMM_KERNEL_AUTO and the other
 * fields 0: the decode kernel plans itself).  *from_table (may be NULL) is
 * set to 1 when the entry came from the sweep's table, 0 for the cost model.
 * Errors: out == NULL or negative sizes: GEMM_ERR_INVALID_VALUE; no usable
 * sm_103a device: GEMM_ERR_UNSUPPORTED.
 */
gemm_status_t gemm_get_config(int is_bf16, int64_t M, int64_t N, int64_t K,
                              gemm_config_t *out, int *from_table);

/*
 * gemm_get_model_config -- as gemm_get_config, but the configuration the
 * cost model alone chooses, ignoring the sweep's table (the baseline the
 * sweep measures table entries against).
 */
gemm_status_t gemm_get_model_config(int is_bf16, int64_t M, int64_t N, int64_t K,
                                    gemm_config_t *out);

/*
 * gemm_split_cluster -- host-side diagnostics for gemm_sgemm / gemm_bf16gemm
 * (and their _config forms) with operands the TMA engine can describe: when
 * every tile of the problem runs in the first round and each is cut into
 * S = 2..8 k-ranges, the S CTAs of a tile form a thread-block cluster and add
 * their partial sums through distributed shared memory, in k order, instead
 * of through the stream's global-memory workspace (the same sums, so the same
 * bits; no scratch is needed, also inside a stream capture).  That needs the
 * 128-wide fp32 tile or the single-CTA bf16 kernel (128 x 256 tiles), and
 * all the clusters resident at once on the device.  `is_bf16` selects
 * gemm_bf16gemm's rules (its decode kernel, which plans its own clusters,
 * reports 1).  Returns S when this configuration (`cfg`, or nullptr for
 * automatic dispatch) runs so, 1 when it does not, 0 for invalid sizes or
 * fields or when there is no usable sm_103a device.  The pages' kernels have
 * no counterpart: their split-K partials meet in global memory ("A GEMM
 * Kernel, Step by Step", "What is left").
 */
int gemm_split_cluster(int is_bf16, int64_t M, int64_t N, int64_t K, const gemm_config_t *cfg);

/*
 * Tile and wave quantization of a launch ("A GEMM Kernel, Step by Step",
 * "The fringe and the last wave"; "Tiled matrix multiplication",
 * "Complexity and constants", wave quantization).
 */
typedef struct {
    int64_t tiles_m;        /* ceil(M / BM)                                 */
    int64_t tiles_n;        /* ceil(N / BN)                                 */
    int64_t tiles;          /* tiles_m * tiles_n                            */
    int64_t covered_m;      /* tiles_m * BM: rows the tile grid covers      */
    int64_t covered_n;      /* tiles_n * BN                                 */
    double useful_fraction; /* (M * N) / (covered_m * covered_n)            */
    int64_t per_wave;       /* num_sms * ctas_per_sm                        */
    int64_t waves;          /* ceil(tiles / per_wave)                       */
    double wave_efficiency; /* tiles / (waves * per_wave)                   */
} gemm_quantization_t;

/*
 * gemm_quantization -- host-only, pure arithmetic: fill `out` for an M x N
 * output cut into BM x BN tiles on `num_sms` multiprocessors holding
 * `ctas_per_sm` blocks each.  Returns GEMM_ERR_INVALID_VALUE for negative
 * sizes or non-positive tile sizes / slots or a NULL `out`.  For M == 0 or
 * N == 0 the fractions are 1 and the counts 0.
 */
gemm_status_t gemm_quantization(int64_t M, int64_t N, int64_t BM, int64_t BN,
                                int64_t num_sms, int64_t ctas_per_sm,
                                gemm_quantization_t *out);

/* Library version, major * 10000 + minor * 100 + patch. */
int gemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM12_H */
