/*
 * gemm_gb300.h -- dense matrix multiply C = alpha * A * B + beta * C on one
 * NVIDIA GB300 (sm_103a).  C ABI of libgemm_gb300.so.
 *
 * The operation is the general GEMM of "Blackwell BF16 GEMM ..." (lshu.cn),
 * section 1.1 (C = alpha*A*B + beta*C), in the two precisions the pages
 * treat:
 *   - gemm_f32:  FP32 SGEMM on the CUDA cores, as in "CUDA hand-written
 *     SGEMM: 0.4 -> 10.23 TFLOPS" (gtnt.cn), sections 1.1-7.1.  Every
 *     product and sum is an IEEE fp32 fused multiply-add; nothing is rounded
 *     through TF32.
 *   - gemm_bf16: BF16 operands, FP32 accumulation in the tensor cores, one
 *     final conversion to BF16 (or an FP32 store), as in "Blackwell BF16
 *     GEMM ...", sections 1.2, 2.1-2.3 and 6.3.
 *
 * Layout.  All matrices are row-major.  A is M x K with row pitch lda >= K,
 * B is K x N with row pitch ldb >= N, C is M x N with row pitch ldc >= N.
 * Pitches count elements, not bytes.
 *
 * Memory and ownership.  A, B and C are DEVICE pointers owned by the caller
 * (for example torch tensors); the library never frees or retains them.
 * Pointers need only element alignment.  The fast paths (TMA, 16-byte
 * vectors) are taken when base addresses are 16-byte aligned and
 * pitch * element size is a multiple of 16 bytes; otherwise a slower
 * generic GPU kernel runs.  There is no CPU fallback.
 *
 * Semantics (the BLAS conventions):
 *   - M == 0 or N == 0: nothing is done.
 *   - beta == 0: C is not read (it may hold NaN or garbage).
 *   - alpha == 0 or K == 0: A and B are not read; C = beta * C.
 *   - C must not overlap A or B (checked by address range).
 *   - BF16 outputs are rounded to nearest, ties to even; overflow gives inf.
 *   - For a given call configuration results are bit-for-bit reproducible
 *     from run to run (no floating-point atomics).
 *
 * Streams and errors.  Calls enqueue work on `stream` (a cudaStream_t; NULL
 * is the legacy default stream) and return without synchronising.  The
 * return value is a gemm_status_t: argument errors are found on the host
 * before anything is launched; GEMM_ERR_CUDA means a CUDA call failed at
 * launch.  Device-side faults of the pipeline (a wait that ran past its
 * time limit) are recorded in a per-device status word that
 * gemm_get_device_status() returns.  The library keeps a little
 * per-device state: the status word and, for launches that split K, one
 * fp32 workspace per stream, allocated on first use and grown (which
 * synchronises the device) when a launch needs more than any before it on
 * that stream; gemm_shutdown() frees it.
 *
 * Thread safety: calls may come from several host threads.  Per-device
 * state is created and grown under a lock.  A split-K workspace belongs to
 * a stream, so calls that enqueue on the same stream from several threads
 * at once must be ordered by the caller (as any work on one stream must
 * be); gemm_shutdown() must not overlap other calls.  The host-buffer entry
 * points run one at a time per process.  Encoded TMA descriptors are cached
 * per thread.  The configuration knobs are process-wide and apply to calls
 * that start after the change.
 */
#ifndef GEMM_GB300_H
#define GEMM_GB300_H

#include <stdint.h>

/* The library is built with hidden visibility; only these are exported. */
#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = -1,        /* negative size, unknown enum, bad key */
    GEMM_ERR_NULLPTR = -2,            /* a matrix that must be read/written is NULL */
    GEMM_ERR_BAD_LD = -3,             /* lda < max(1,K), ldb < max(1,N) or ldc < max(1,N)
                                         (transposed operands: lda < max(1,M), ldb < max(1,K)) */
    GEMM_ERR_UNSUPPORTED_DEVICE = -4, /* current device is not compute capability 10.3 */
    GEMM_ERR_CUDA = -5,               /* a CUDA runtime/driver call failed */
    GEMM_ERR_DEVICE_TIMEOUT = -6,     /* a pipeline wait on the GPU ran out of time */
    GEMM_ERR_ALIAS = -7,              /* C overlaps A, B or the bias */
    GEMM_ERR_TOO_LARGE = -8,          /* a dimension or pitch exceeds 2^31 - 1 */
    GEMM_ERR_SCRATCH_LIMIT = -9,      /* gemm_bf16_noalloc: the call needs more split-K
                                         scratch than its static maximum */
    GEMM_ERR_DEVICE_CHECK = -10       /* debug build only (libgemm_gb300_debug.so): a
                                         device-side check of an index, a copy's
                                         coordinates or a shared/tensor-memory range
                                         failed and the access was skipped */
} gemm_status_t;

typedef enum {
    GEMM_OUT_BF16 = 0,  /* C holds bf16 (uint16 bit patterns) */
    GEMM_OUT_F32 = 1    /* C holds fp32 */
} gemm_out_t;

/*
 * FP32 SGEMM: C = alpha * A * B + beta * C, all fp32, on the CUDA cores.
 * Source: "CUDA hand-written SGEMM: 0.4 -> 10.23 TFLOPS" (gtnt.cn),
 * section 1.1 (C = A*B, row-major) generalised by "Blackwell BF16 GEMM ..."
 * section 1.1 (alpha, beta).
 *   M, N, K     sizes, >= 0
 *   A, lda      device fp32, M x K, pitch lda
 *   B, ldb      device fp32, K x N, pitch ldb
 *   C, ldc      device fp32, M x N, pitch ldc; read only if beta != 0
 *   stream      cudaStream_t to enqueue on
 * Returns GEMM_OK or a gemm_status_t error; on error nothing is launched.
 */
GEMM_API int gemm_f32(int64_t M, int64_t N, int64_t K, float alpha,
             const float *A, int64_t lda, const float *B, int64_t ldb,
             float beta, float *C, int64_t ldc, void *stream);

/*
 * BF16 GEMM with FP32 accumulation on the tcgen05 tensor cores:
 * C = alpha * A * B + beta * C, accumulated in fp32, alpha/beta applied in
 * fp32, then stored as bf16 (round to nearest even) or fp32.
 * Source: "Blackwell BF16 GEMM ..." (lshu.cn), sections 1.1-1.2 (operation,
 * bf16 format, fp32 accumulation), 2.2-2.3 (TMA-fed asynchronous pipeline),
 * 4.3 and 6.2 (tails), 6.3 (the accumulator must be fp32).
 *   A, lda      device bf16 (uint16 bits), M x K, pitch lda
 *   B, ldb      device bf16 (uint16 bits), K x N, pitch ldb
 *   C, ldc      device, M x N, pitch ldc, element type c_type; it is both
 *               the beta input and the output
 *   c_type      GEMM_OUT_BF16 or GEMM_OUT_F32
 * Returns GEMM_OK or a gemm_status_t error; on error nothing is launched.
 */
GEMM_API int gemm_bf16(int64_t M, int64_t N, int64_t K, float alpha,
              const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
              float beta, void *C, int64_t ldc, int c_type, void *stream);

/* Activation of the fused epilogue. */
typedef enum {
    GEMM_ACT_NONE = 0,
    GEMM_ACT_RELU = 1,      /* max(x, 0) */
    GEMM_ACT_GELU_TANH = 2  /* 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */
} gemm_act_t;

/*
 * Options of the extended entry points: operand layouts and a fused
 * epilogue.  A zero-initialised struct means "no transposes, no epilogue".
 *   trans_a    0: A is M x K row-major (lda >= K);
 *              1: the caller stores A^T, K x M row-major (lda >= M)
 *   trans_b    0: B is K x N row-major (ldb >= N);
 *              1: the caller stores B^T, N x K row-major (ldb >= K)
 *   bias       NULL, or a device vector of N values added to every row
 *   bias_type  GEMM_OUT_BF16 or GEMM_OUT_F32: element type of bias
 *   act        gemm_act_t
 */
typedef struct {
    int trans_a;
    int trans_b;
    const void *bias;
    int bias_type;
    int act;
} gemm_opts_t;

/*
 * Extended GEMMs with transposed operands and a fused epilogue:
 *     C = act(alpha * op(A) * op(B) + bias) + beta * C
 * op(X) is X or, with trans_x, the transpose of the stored matrix.  The
 * activation comes first and beta * C (a residual) is added after it, the
 * order of the fused "GELU, then residual add" kernel of the "Z-Turbo"
 * tuning page (lanjinlin.com.cn), section 2.1; "Blackwell BF16 GEMM ..."
 * (lshu.cn), section 3.3, names GELU and residual as epilogue fusions, and
 * section 5.1 the transposed GEMMs of training.  The epilogue runs in fp32:
 * v = act(fmaf(alpha, acc, bias)), then out = v + beta * C with beta * C
 * rounded first (as in the plain epilogue fmaf(alpha, acc, beta * C)), then
 * the single conversion to C's type.  opts == NULL (or all zero) gives
 * exactly gemm_bf16 / gemm_f32.  Same memory, stream and error rules as the
 * plain entry points; additionally bias must not overlap C
 * (GEMM_ERR_ALIAS), and an unknown act or bias_type is GEMM_ERR_INVALID_ARG.
 */
GEMM_API int gemm_bf16_ex(int64_t M, int64_t N, int64_t K, float alpha,
                          const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                          float beta, void *C, int64_t ldc, int c_type,
                          const gemm_opts_t *opts, void *stream);
GEMM_API int gemm_f32_ex(int64_t M, int64_t N, int64_t K, float alpha,
                         const float *A, int64_t lda, const float *B, int64_t ldb,
                         float beta, float *C, int64_t ldc, const gemm_opts_t *opts,
                         void *stream);

/*
 * Strided batched GEMMs: for i = 0 .. batch-1,
 *     C_i = act(alpha * op(A_i) * op(B_i) + bias) + beta * C_i
 * with A_i = A + i * stride_a, B_i = B + i * stride_b, C_i = C + i * stride_c
 * (strides in elements).  "Blackwell BF16 GEMM ..." (lshu.cn), section 3.1,
 * lists grouped / batched GEMM among the cuBLASLt capabilities a GEMM
 * library covers; this is the strided form of BLAS.  Every matrix has the
 * same M, N, K, pitches, layouts (opts) and bias.
 *   batch      >= 0 (0: nothing is done)
 *   stride_a   >= 0; 0 shares one A among all products (likewise stride_b)
 *   stride_c   C matrices must not overlap: stride_c * element size at least
 *              the span of one C (else GEMM_ERR_ALIAS)
 * The whole batch runs as one launch; the tensor-core and TMA kernels take
 * it when pitches and nonzero batch strides are multiples of 16 bytes and a
 * nonzero stride is at least one matrix's span, otherwise the generic
 * kernel.  C must not overlap any A, B or bias byte the batch reads
 * (GEMM_ERR_ALIAS); negative strides are GEMM_ERR_INVALID_ARG.  Otherwise
 * the rules of gemm_bf16_ex / gemm_f32_ex.
 */
GEMM_API int gemm_bf16_batched(int64_t batch, int64_t M, int64_t N, int64_t K, float alpha,
                               const uint16_t *A, int64_t lda, int64_t stride_a,
                               const uint16_t *B, int64_t ldb, int64_t stride_b, float beta,
                               void *C, int64_t ldc, int64_t stride_c, int c_type,
                               const gemm_opts_t *opts, void *stream);
GEMM_API int gemm_f32_batched(int64_t batch, int64_t M, int64_t N, int64_t K, float alpha,
                              const float *A, int64_t lda, int64_t stride_a, const float *B,
                              int64_t ldb, int64_t stride_b, float beta, float *C, int64_t ldc,
                              int64_t stride_c, const gemm_opts_t *opts, void *stream);

/*
 * One problem of a grouped GEMM: C = alpha * op(A) * op(B) + beta * C with
 * its own sizes, operands, pitches (elements) and scalars.  A and B are bf16
 * (uint16 bits) for gemm_bf16_grouped and fp32 for gemm_f32_grouped; C has
 * the call's output type.
 */
typedef struct {
    int64_t M, N, K;
    const void *A;
    int64_t lda;
    const void *B;
    int64_t ldb;
    void *C;
    int64_t ldc;
    float alpha, beta;
} gemm_group_t;

/*
 * Grouped GEMMs: `count` problems of different shapes and operands in one
 * call ("Blackwell BF16 GEMM ..." (lshu.cn), section 3.1, lists grouped
 * GEMM among the capabilities of a GEMM library).  groups is a HOST array of
 * count gemm_group_t (read during the call only).  Each problem follows the
 * rules of gemm_bf16 / gemm_f32 (pitches, NULL pointers, beta == 0 leaves C
 * unread, alpha == 0 or K == 0 gives beta * C, empty problems do nothing);
 * opts may select transposed layouts (trans_a / trans_b apply to every
 * problem) but no bias or activation (GEMM_ERR_INVALID_ARG).  Because the
 * problems run concurrently, no problem's C may overlap any other
 * problem's A, B or C, and none its own A or B (GEMM_ERR_ALIAS); A and B
 * may be shared between problems.
 * Problems whose operands TMA can fetch (16-byte aligned bases, pitches in
 * multiples of 16 bytes; FP32 also row-major) run in ONE persistent launch
 * per 64 problems over the union of their output tiles (the tcgen05 kernel
 * for bf16, the TMA SGEMM for fp32); the others run one call each.
 * The grouped launch never splits K; results meet the same tolerances as
 * the single calls (and on integer-valued inputs are exact either way).
 * Returns GEMM_OK or a gemm_status_t error; argument errors are reported
 * before anything is launched.
 */
GEMM_API int gemm_bf16_grouped(int64_t count, const gemm_group_t *groups, int c_type,
                               const gemm_opts_t *opts, void *stream);
GEMM_API int gemm_f32_grouped(int64_t count, const gemm_group_t *groups,
                              const gemm_opts_t *opts, void *stream);

/*
 * Host-buffer GEMMs: the same products with A, B and C in HOST memory
 * (pinned memory gives the full copy bandwidth; pageable memory works).  The
 * library copies B and then A (and C when beta != 0) to the device in row
 * blocks, computes each block as soon as its rows have landed and copies it
 * back while the next computes (copy-in, compute and copy-out streams of a
 * per-device pipeline), and returns when C holds the result.  Device staging
 * buffers are library-owned, allocated on first use, grown when a call needs
 * more and kept until gemm_shutdown().  One host-buffer call runs at a time
 * (others wait).  Argument rules as gemm_f32 / gemm_bf16 (C may not overlap
 * A or B in host memory); a device pipeline fault returns
 * GEMM_ERR_DEVICE_TIMEOUT, as gemm_get_device_status() would.
 */
GEMM_API int gemm_f32_host(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                           int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                           int64_t ldc);
GEMM_API int gemm_bf16_host(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t *A,
                            int64_t lda, const uint16_t *B, int64_t ldb, float beta, void *C,
                            int64_t ldc, int c_type);

/*
 * Several host-buffer GEMMs in one call.  The products run in order through
 * the pipeline above: the copies of product i + 1 are enqueued right behind
 * those of product i, so they travel while product i computes, and the call
 * returns once every C holds its result.  (A sequence of gemm_*_host calls
 * cannot overlap this way: each returns only when its C is back.)  Each
 * product follows the rules of gemm_f32_host / gemm_bf16_host; in addition
 * no product's C may overlap an operand or the C of another product of the
 * batch (GEMM_ERR_ALIAS): products that feed one another need separate calls.
 * At most GEMM_HOST_BATCH_MAX products; count == 0 does nothing.  The pages
 * have no counterpart (their GEMMs start from device memory).
 */
enum { GEMM_HOST_F32 = 0, GEMM_HOST_BF16 = 1 };
#define GEMM_HOST_BATCH_MAX 64
typedef struct {
    int dtype;    /* GEMM_HOST_F32: fp32 A, B, C; GEMM_HOST_BF16: bf16 A, B */
    int c_type;   /* GEMM_HOST_BF16 only: GEMM_OUT_BF16 or GEMM_OUT_F32 */
    int64_t M, N, K;
    float alpha, beta;
    const void *A;
    int64_t lda;  /* elements, row-major M x K */
    const void *B;
    int64_t ldb;  /* elements, row-major K x N */
    void *C;
    int64_t ldc;  /* elements, row-major M x N */
} gemm_host_op_t;
GEMM_API int gemm_host_batch(int64_t count, const gemm_host_op_t *ops);

/*
 * Allocation-free BF16 GEMM.  The source pages have no counterpart: this is
 * an interface for callers that cannot call cudaMalloc at all, for example
 * code that runs inside a host whose device memory is fully owned by its own
 * arena or caching allocator (a plugin, a framework extension) and may not
 * allocate around it, or latency-critical code that cannot accept the
 * implicit device synchronisation an allocation can cause.
 *
 * Same operation, arguments, layout and results as gemm_bf16 (same kernel,
 * same split choice), except that the split-K scratch lives in a statically
 * sized device array compiled into the library instead of a workspace the
 * library allocates:
 *   - the array holds GEMM_NOALLOC_SCRATCH_BYTES (32 MiB) and is reserved on
 *     every GPU that loads its module, until the process exits;
 *   - a call whose split-K partials need more than the array offers (at
 *     most 4096 output tiles and about 32 MiB of fp32 partials) returns
 *     GEMM_ERR_SCRATCH_LIMIT and launches nothing; the automatic split
 *     choice stays well inside the limit, a large forced "split_k" may not;
 *   - A and B must be TMA-compatible (16-byte aligned bases, lda and ldb
 *     multiples of 8), else GEMM_ERR_INVALID_ARG;
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first
 *     call before any stream capture on that device;
 *   - every call shares the one array and clears the part that must start
 *     at zero (the split-K tile counters) on `stream` before its kernel;
 *     calls whose executions overlap on the GPU (different streams, no
 *     ordering between them) race on the array and give wrong results;
 *   - a pipeline wait that runs out of time is recorded in the array's
 *     fault record, not in the status word gemm_get_device_status reads;
 *     the kernel still returns and leaves that call's output incomplete.
 *     The record keeps the first fault since it was last read:
 *     gemm_noalloc_get_status below reports and clears it.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define GEMM_NOALLOC_SCRATCH_BYTES (32u << 20)
GEMM_API int gemm_bf16_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                               const uint16_t *A, int64_t lda, const uint16_t *B,
                               int64_t ldb, float beta, void *C, int64_t ldc, int c_type,
                               void *stream);

/*
 * Status of gemm_bf16_noalloc calls on the current device, for the same
 * callers (it allocates nothing either; the source pages have no
 * counterpart).  Synchronises `stream` (make it the stream, or the last of
 * the streams, the calls ran on), reads the static array's fault record and
 * returns GEMM_OK if no wait ran out since the record was last read, else
 * GEMM_ERR_DEVICE_TIMEOUT (GEMM_ERR_DEVICE_CHECK for a failed check of the
 * debug build) and clears the record.  fault_info (may be NULL)
 * receives the fault's details in the layout of
 * gemm_get_device_fault_info, or 0.  GEMM_ERR_CUDA if a CUDA call failed.
 * Like the first gemm_bf16_noalloc call, the first use on a device looks up
 * the array's address and should come before any stream capture.
 */
GEMM_API int gemm_noalloc_get_status(void *stream, int64_t *fault_info);

/*
 * Synchronises `stream`, then returns and clears the current device's
 * pipeline status: GEMM_OK, or GEMM_ERR_DEVICE_TIMEOUT if a kernel since the
 * last call gave up on a wait (its output is then incomplete), or, in the
 * debug build (libgemm_gb300_debug.so, loaded when the environment variable
 * GEMM_GB300_DEBUG is 1), GEMM_ERR_DEVICE_CHECK if a device-side check of an
 * index, a copy coordinate or a memory range failed (the checked access was
 * skipped; the output is then incomplete).  Returns GEMM_ERR_CUDA if the
 * synchronisation itself failed.
 */
GEMM_API int gemm_get_device_status(void *stream);

/*
 * Details of the last recorded device fault (0 if none): bits 0-7 the role
 * (1 producer, 2 MMA issuer, 3 epilogue, 4 FP32 kernel, 5 a debug-build
 * check), bits 8-15 the pipeline stage (for a check: its site, 1 a load of
 * A, 2 a load of B, 3 a store of C, 4 tensor-memory columns, 5 a split-K
 * workspace index, 6 an MMA operand's shared-memory range), bits 16-47 the
 * tile index.  Does not clear it.
 */
GEMM_API int64_t gemm_get_device_fault_info(void);

/* A static, human-readable name for a gemm_status_t. */
GEMM_API const char *gemm_status_string(int status);

/*
 * 1 in the debug build (libgemm_gb300_debug.so, compiled with GEMM_DEBUG=1,
 * whose kernels check the indices, copy coordinates and shared/tensor-memory
 * ranges they compute and report a failed check as GEMM_ERR_DEVICE_CHECK),
 * 0 in the release build.  Needs no GPU.  Part of the library's own
 * test support (compute-sanitizer is not available to its tests); the source
 * pages have no counterpart.
 */
GEMM_API int gemm_debug_checks(void);

/*
 * Tuning and debugging knobs (process-wide).  Keys:
 *   "watchdog_ms"   time limit of one pipeline wait on the GPU, ms (default 2000)
 *   "force_path"    0 auto, 1 force the non-TMA kernels (cp.async SGEMM,
 *                   generic BF16 kernel),
 *                   2 force the tcgen05 kernel (fails on misaligned input)
 *   "fault_inject"  1: the next tcgen05 or FP32 TMA launch withholds one
 *                   pipeline stage so its waits run out (tests the
 *                   watchdog); resets itself
 *   "split_k"       0 auto, else the number of K slices for the tcgen05 kernel
 *   "bf16_tile_n"   0 auto, else 128 or 256 (tcgen05 tile width)
 *   "tail_split_off" 1: leave the tiles of the last partial wave whole;
 *                   0 (default) cuts them: into narrower sub-tiles
 *                   (tcgen05 kernels) or along K (FP32 TMA kernel)
 *   "stream_k"      1: when a tcgen05 GEMM has few tiles and a long K, deal
 *                   all K iterations out to the SMs in equal ranges
 *                   (stream-K); 0 (default): equal K slices per tile
 *   "raster_group"  0 auto, else the number of M-blocks (128 rows, or 256
 *                   for CTA pairs) per raster band of the tcgen05 kernel
 *   "cta_pair"      0 auto, 1 single-CTA tcgen05 kernel only, 2 always the
 *                   CTA-pair (2-SM, cta_group::2) kernel
 *   "pair_limit"    0 all resident pairs, else at most this many CTA pairs
 *                   (leaves SMs free for other work; tests use it to reach
 *                   the tail paths at small sizes)
 *   "stage_pairs"   tcgen05 kernels: 0 (default) every tile runs its K
 *                   blocks two at a time (one barrier wait and eight MMAs per
 *                   pair of stages; the single-CTA kernel only when its ring
 *                   has six or more stages), 1 on the CTA-pair kernel only its
 *                   narrower tail tiles, 2 none
 *   "kpair_maps_off" 0 (default): where the shape allows, the CTA-pair
 *                   kernel fills two stages with one TMA copy per operand
 *                   (boxes spanning two 64-deep K blocks); 1: one copy per
 *                   64-deep box
 * Returns GEMM_OK or GEMM_ERR_INVALID_ARG for an unknown key or value.
 */
GEMM_API int gemm_set_config(const char *key, int64_t value);
GEMM_API int gemm_get_config(const char *key, int64_t *value);

/*
 * Name of the kernel the last successful gemm_* call on this host thread
 * launched ("sgemm_tma", "sgemm_simt", "bf16_tcgen05", "bf16_simt", "scale_c",
 * "sgemm_tma_grouped", "bf16_tcgen05_grouped", "bf16_grouped_mixed" or
 * "f32_grouped_mixed" (a grouped call that also ran single calls),
 * "none").
 */
GEMM_API const char *gemm_last_kernel(void);

/* Frees the per-device state of the current device.  Safe to call twice. */
GEMM_API int gemm_shutdown(void);

/*
 * Library ABI version, currently 2.  Version 2 keeps every version-1 entry
 * point and structure unchanged and adds gemm_bf16_grouped /
 * gemm_f32_grouped, gemm_host_batch (gemm_host_op_t), gemm_noalloc_get_status,
 * gemm_debug_checks and the status GEMM_ERR_DEVICE_CHECK.
 */
GEMM_API int gemm_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_GB300_H */
