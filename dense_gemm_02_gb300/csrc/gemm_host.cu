// Host-buffer entry points (gemm_f32_host, gemm_bf16_host, and
// gemm_host_batch for several products in one pipeline): operands in host
// memory, results back in host memory when the call returns.  The copies are
// pipelined with the GEMM on three streams of a per-device pipeline:
//
//   copy-in   B (whole), then A (and C when beta != 0) in row blocks
//   compute   the device GEMM of each row block once B and its A block
//             have landed (the same library kernels as gemm_f32/gemm_bf16)
//   copy-out  each C row block as soon as it is computed
//
// so the transfer of block i+1 and the return of block i-1 overlap the
// computation of block i.  Device staging buffers (A, B, C with row pitches
// rounded up to 16 bytes, so the TMA kernels take them) are one library
// allocation per device, grown on demand and kept until gemm_shutdown.
// Every numeric step runs in the device kernels; this file only moves
// memory and orders streams.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "gemm_gb300.h"
#include "internal.h"

namespace gemm {
namespace {

std::mutex g_host_mu;  // the pipeline state of a device serves one call at a time

constexpr int kMaxBlocks = 8;

int64_t round_up(int64_t x, int64_t q) { return (x + q - 1) / q * q; }

// Events one product's pipeline uses (B landed, then per row block: A landed,
// C computed).
constexpr size_t kEventsPerOp = 1 + 2 * kMaxBlocks;

// Creates the device's pipeline on first use and grows its events (n_ops
// products' worth) and its staging buffer.
int host_pipe(DeviceState *st, size_t bytes, size_t n_ops, HostPipe **out) {
    if (!st->host) {
        auto hp = std::make_unique<HostPipe>();
        for (cudaStream_t *s : {&hp->in, &hp->compute, &hp->out})
            if (cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) != cudaSuccess)
                return GEMM_ERR_CUDA;
        st->host = std::move(hp);
    }
    HostPipe *hp = st->host.get();
    while (hp->events.size() < n_ops * kEventsPerOp) {
        cudaEvent_t e;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
            return GEMM_ERR_CUDA;
        hp->events.push_back(e);
    }
    if (hp->bytes < bytes) {
        if (hp->buf && cudaFree(hp->buf) != cudaSuccess) return GEMM_ERR_CUDA;
        hp->buf = nullptr;
        hp->bytes = 0;
        if (cudaMalloc(&hp->buf, bytes) != cudaSuccess) return GEMM_ERR_CUDA;
        hp->bytes = bytes;
    }
    *out = hp;
    return GEMM_OK;
}

// Copies `rows` rows of `width_bytes` between pitched buffers on `s` (one
// linear copy when both sides are packed).
bool copy_rows(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width_bytes,
               size_t rows, cudaMemcpyKind kind, cudaStream_t s) {
    if (rows == 0 || width_bytes == 0) return true;
    if (dpitch == width_bytes && spitch == width_bytes)
        return cudaMemcpyAsync(dst, src, width_bytes * rows, kind, s) == cudaSuccess;
    return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width_bytes, rows, kind, s) == cudaSuccess;
}

// One product of a host-buffer call, with its staging plan: device pitches
// (rows padded to 16 bytes so the TMA kernels apply), byte offsets of its
// staged A, B and C in the pipeline's buffer, and its row blocks.
struct HostOp {
    bool f32;    // fp32 A, B, C; else bf16 A, B and C of c_type
    int c_type;  // bf16 products: GEMM_OUT_BF16 or GEMM_OUT_F32
    int64_t M, N, K;
    float alpha, beta;
    const void *A;
    int64_t lda;
    const void *B;
    int64_t ldb;
    void *C;
    int64_t ldc;
    // plan
    size_t ab_esz, c_esz;
    bool reads_ab;
    int64_t lda_d, ldb_d, ldc_d;
    size_t a_off, b_off, c_off, bytes;
    int64_t nblk, mb;
};

// Fills in the plan of `op` (staging offsets from `base`).  Row blocks are
// multiples of 256 rows (the CTA-pair tile height), each at least `waves`
// waves of 128 x 128 tiles over the SMs: smaller blocks overlap more of the
// copies but run the GEMM less efficiently.  Measured on GB300: the FP32
// 4096^3 GEMM takes 2.13 ms whole, 2.2 ms in two blocks, 2.41 ms in three
// and 2.64 ms in eight, so the compute-bound FP32 path asks for three waves;
// the BF16 path, bound by the copies, for one.  At most kMaxBlocks.
void plan_op(HostOp &op, int sm_count, size_t base) {
    op.ab_esz = op.f32 ? 4 : 2;
    op.c_esz = (op.f32 || op.c_type == GEMM_OUT_F32) ? 4 : 2;
    op.reads_ab = op.alpha != 0.f && op.K > 0;
    const int64_t qa = 16 / (int64_t)op.ab_esz, qc = 16 / (int64_t)op.c_esz;
    op.lda_d = round_up(std::max<int64_t>(op.K, 1), qa);
    op.ldb_d = round_up(std::max<int64_t>(op.N, 1), qa);
    op.ldc_d = round_up(std::max<int64_t>(op.N, 1), qc);
    const size_t a_bytes = op.reads_ab ? (size_t)round_up(op.M * op.lda_d * op.ab_esz, 256) : 0;
    const size_t b_bytes = op.reads_ab ? (size_t)round_up(op.K * op.ldb_d * op.ab_esz, 256) : 0;
    const size_t c_bytes = (size_t)round_up(op.M * op.ldc_d * op.c_esz, 256);
    op.a_off = base;
    op.b_off = base + a_bytes;
    op.c_off = base + a_bytes + b_bytes;
    op.bytes = a_bytes + b_bytes + c_bytes;
    const int64_t waves = op.f32 ? 3 : 1;
    const int64_t min_rows = round_up(
        waves * (int64_t)sm_count * 128 * 128 / std::max<int64_t>(op.N, 128), 256);
    int64_t nblk = std::min<int64_t>(kMaxBlocks, std::max<int64_t>(1, op.M / min_rows));
    op.mb = round_up((op.M + nblk - 1) / nblk, 256);
    op.nblk = (op.M + op.mb - 1) / op.mb;
}

// The device GEMM of rows [r0, r0 + m) of `op` on the staged operands.
int device_gemm(const HostOp &op, char *buf, int64_t r0, int64_t m, cudaStream_t s) {
    const char *dA = op.reads_ab ? buf + op.a_off + r0 * op.lda_d * op.ab_esz : nullptr;
    const char *dB = op.reads_ab ? buf + op.b_off : nullptr;
    char *dC = buf + op.c_off + r0 * op.ldc_d * op.c_esz;
    if (op.f32)
        return gemm_f32(m, op.N, op.K, op.alpha, reinterpret_cast<const float *>(dA), op.lda_d,
                        reinterpret_cast<const float *>(dB), op.ldb_d, op.beta,
                        reinterpret_cast<float *>(dC), op.ldc_d, s);
    return gemm_bf16(m, op.N, op.K, op.alpha, reinterpret_cast<const uint16_t *>(dA), op.lda_d,
                     reinterpret_cast<const uint16_t *>(dB), op.ldb_d, op.beta, dC, op.ldc_d,
                     op.c_type, s);
}

// Enqueues the pipeline of one planned product; events ev[0 .. 2 * nblk] are
// its own.  Returns at the first failing call.
int enqueue_op(const HostOp &op, HostPipe *hp, const cudaEvent_t *ev) {
    char *buf = static_cast<char *>(hp->buf);
    const size_t ab = op.ab_esz, ce = op.c_esz;
    if (op.reads_ab &&
        !copy_rows(buf + op.b_off, op.ldb_d * ab, op.B, op.ldb * ab, op.N * ab, op.K,
                   cudaMemcpyHostToDevice, hp->in))
        return GEMM_ERR_CUDA;
    if (cudaEventRecord(ev[0], hp->in) != cudaSuccess ||
        cudaStreamWaitEvent(hp->compute, ev[0], 0) != cudaSuccess)
        return GEMM_ERR_CUDA;
    for (int64_t i = 0; i < op.nblk; ++i) {
        const int64_t r0 = i * op.mb, m = std::min(op.mb, op.M - r0);
        cudaEvent_t eIn = ev[1 + 2 * i], eOut = ev[2 + 2 * i];
        if (op.reads_ab &&
            !copy_rows(buf + op.a_off + r0 * op.lda_d * ab, op.lda_d * ab,
                       static_cast<const char *>(op.A) + r0 * op.lda * ab, op.lda * ab, op.K * ab,
                       m, cudaMemcpyHostToDevice, hp->in))
            return GEMM_ERR_CUDA;
        if (op.beta != 0.f &&
            !copy_rows(buf + op.c_off + r0 * op.ldc_d * ce, op.ldc_d * ce,
                       static_cast<const char *>(op.C) + r0 * op.ldc * ce, op.ldc * ce,
                       op.N * ce, m, cudaMemcpyHostToDevice, hp->in))
            return GEMM_ERR_CUDA;
        if (cudaEventRecord(eIn, hp->in) != cudaSuccess ||
            cudaStreamWaitEvent(hp->compute, eIn, 0) != cudaSuccess)
            return GEMM_ERR_CUDA;
        const int r = device_gemm(op, buf, r0, m, hp->compute);
        if (r != GEMM_OK) return r;
        if (cudaEventRecord(eOut, hp->compute) != cudaSuccess ||
            cudaStreamWaitEvent(hp->out, eOut, 0) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (!copy_rows(static_cast<char *>(op.C) + r0 * op.ldc * ce, op.ldc * ce,
                       buf + op.c_off + r0 * op.ldc_d * ce, op.ldc_d * ce, op.N * ce, m,
                       cudaMemcpyDeviceToHost, hp->out))
            return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

// Runs `count` validated products through one pipeline, in order: the
// copies of product i + 1 are enqueued behind those of product i, so they
// overlap its GEMMs, and the call returns once every C is in host memory.
int run_ops(HostOp *ops, size_t count) {
    std::lock_guard<std::mutex> lock(g_host_mu);
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != GEMM_OK) return rc;
    size_t bytes = 0;
    for (size_t i = 0; i < count; ++i) {
        plan_op(ops[i], st->sm_count, bytes);
        bytes += ops[i].bytes;
    }
    HostPipe *hp = nullptr;
    if ((rc = host_pipe(st, bytes, count, &hp)) != GEMM_OK) return rc;
    for (size_t i = 0; i < count && rc == GEMM_OK; ++i)
        rc = enqueue_op(ops[i], hp, hp->events.data() + i * kEventsPerOp);
    if (rc != GEMM_OK) {
        // Copies and GEMMs enqueued before the failure may still be running,
        // some writing the caller's C: let them finish before the caller gets
        // its buffers back.  Their own errors are not reported over rc.
        cudaStreamSynchronize(hp->in);
        cudaStreamSynchronize(hp->compute);
        cudaStreamSynchronize(hp->out);
        cudaGetLastError();
        return rc;
    }
    if (cudaStreamSynchronize(hp->out) != cudaSuccess) return GEMM_ERR_CUDA;
    // A pipeline wait that ran out of time on the device shows here.
    return gemm_get_device_status(hp->compute);
}

// Argument checks of one product (as the single-product entry points):
// GEMM_OK, an error, or 1 for nothing to do (M == 0 or N == 0).
int check_op(const HostOp &op) {
    if (!op.f32 && op.c_type != GEMM_OUT_BF16 && op.c_type != GEMM_OUT_F32)
        return GEMM_ERR_INVALID_ARG;
    const size_t ab = op.f32 ? 4 : 2, ce = (op.f32 || op.c_type == GEMM_OUT_F32) ? 4 : 2;
    return validate_gemm_args(op.M, op.N, op.K, op.alpha, op.A, op.lda, ab, op.B, op.ldb, ab,
                              op.beta, op.C, op.ldc, ce);
}

}  // namespace
}  // namespace gemm

using namespace gemm;

extern "C" int gemm_f32_host(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                             int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                             int64_t ldc) {
    HostOp op{true, GEMM_OUT_F32, M, N, K, alpha, beta, A, lda, B, ldb, C, ldc};
    const int rc = check_op(op);
    if (rc == 1) return GEMM_OK;
    if (rc != GEMM_OK) return rc;
    return run_ops(&op, 1);
}

extern "C" int gemm_bf16_host(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t *A,
                              int64_t lda, const uint16_t *B, int64_t ldb, float beta, void *C,
                              int64_t ldc, int c_type) {
    HostOp op{false, c_type, M, N, K, alpha, beta, A, lda, B, ldb, C, ldc};
    const int rc = check_op(op);
    if (rc == 1) return GEMM_OK;
    if (rc != GEMM_OK) return rc;
    return run_ops(&op, 1);
}

extern "C" int gemm_host_batch(int64_t count, const gemm_host_op_t *ops) {
    if (count < 0 || count > GEMM_HOST_BATCH_MAX) return GEMM_ERR_INVALID_ARG;
    if (count == 0) return GEMM_OK;
    if (!ops) return GEMM_ERR_NULLPTR;
    std::vector<HostOp> run;
    run.reserve((size_t)count);
    for (int64_t i = 0; i < count; ++i) {
        const gemm_host_op_t &o = ops[i];
        if (o.dtype != GEMM_HOST_F32 && o.dtype != GEMM_HOST_BF16) return GEMM_ERR_INVALID_ARG;
        HostOp op{o.dtype == GEMM_HOST_F32, o.dtype == GEMM_HOST_F32 ? GEMM_OUT_F32 : o.c_type,
                  o.M, o.N, o.K, o.alpha, o.beta, o.A, o.lda, o.B, o.ldb, o.C, o.ldc};
        const int rc = check_op(op);
        if (rc == 1) continue;
        if (rc != GEMM_OK) return rc;
        run.push_back(op);
    }
    // No product's C may meet any operand or result of another: the copies of
    // later products run while earlier ones compute and write back.
    for (size_t i = 0; i < run.size(); ++i) {
        const HostOp &x = run[i];
        const size_t xce = (x.f32 || x.c_type == GEMM_OUT_F32) ? 4 : 2;
        const size_t xc = span_bytes(x.M, x.N, x.ldc, xce);
        for (size_t j = 0; j < run.size(); ++j) {
            if (j == i) continue;
            const HostOp &y = run[j];
            const size_t yab = y.f32 ? 4 : 2, yce = (y.f32 || y.c_type == GEMM_OUT_F32) ? 4 : 2;
            const bool y_ab = y.alpha != 0.f && y.K > 0;
            if (ranges_overlap(x.C, xc, y.C, span_bytes(y.M, y.N, y.ldc, yce)) ||
                (y_ab && (ranges_overlap(x.C, xc, y.A, span_bytes(y.M, y.K, y.lda, yab)) ||
                          ranges_overlap(x.C, xc, y.B, span_bytes(y.K, y.N, y.ldb, yab)))))
                return GEMM_ERR_ALIAS;
        }
    }
    if (run.empty()) return GEMM_OK;
    return run_ops(run.data(), run.size());
}
