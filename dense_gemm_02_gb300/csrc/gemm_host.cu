// Host-buffer entry points (gemm_f32_host, gemm_bf16_host): operands in host
// memory, result back in host memory when the call returns.  The copies are
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

// Creates the device's pipeline on first use and grows its staging buffer.
int host_pipe(DeviceState *st, size_t bytes, HostPipe **out) {
    if (!st->host) {
        auto hp = std::make_unique<HostPipe>();
        for (cudaStream_t *s : {&hp->in, &hp->compute, &hp->out})
            if (cudaStreamCreateWithFlags(s, cudaStreamNonBlocking) != cudaSuccess)
                return GEMM_ERR_CUDA;
        hp->events.resize(1 + 2 * kMaxBlocks);
        for (cudaEvent_t &e : hp->events)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
                return GEMM_ERR_CUDA;
        st->host = std::move(hp);
    }
    HostPipe *hp = st->host.get();
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

// The pipelined host GEMM.  `device_gemm(m, A, lda, B, ldb, C, ldc,
// stream)` runs the device GEMM of m rows with the staged B; `waves` is the
// least work per row block, in waves of 128 x 128 tiles over the SMs.
template <typename DeviceGemm>
int run_host(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
             size_t ab_esz, const void *B, int64_t ldb, float beta, void *C, int64_t ldc,
             size_t c_esz, int64_t waves, DeviceGemm device_gemm) {
    std::lock_guard<std::mutex> lock(g_host_mu);
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != GEMM_OK) return rc;
    const bool reads_ab = alpha != 0.f && K > 0;
    // Device pitches: rows padded to 16 bytes so the TMA kernels apply.
    const int64_t lda_d = round_up(std::max<int64_t>(K, 1), 16 / (int64_t)ab_esz);
    const int64_t ldb_d = round_up(std::max<int64_t>(N, 1), 16 / (int64_t)ab_esz);
    const int64_t ldc_d = round_up(std::max<int64_t>(N, 1), 16 / (int64_t)c_esz);
    const size_t a_bytes = reads_ab ? (size_t)round_up(M * lda_d * ab_esz, 256) : 0;
    const size_t b_bytes = reads_ab ? (size_t)round_up(K * ldb_d * ab_esz, 256) : 0;
    const size_t c_bytes = (size_t)round_up(M * ldc_d * c_esz, 256);
    HostPipe *hp = nullptr;
    if ((rc = host_pipe(st, a_bytes + b_bytes + c_bytes, &hp)) != GEMM_OK) return rc;
    char *dA = static_cast<char *>(hp->buf);
    char *dB = dA + a_bytes;
    char *dC = dB + b_bytes;

    // Row blocks, multiples of 256 rows (the CTA-pair tile height), each at
    // least `waves` waves of 128 x 128 tiles: smaller blocks overlap more of
    // the copies but run the GEMM less efficiently.  Measured on GB300: the
    // FP32 4096^3 GEMM takes 2.13 ms whole, 2.2 ms in two blocks, 2.41 ms in
    // three and 2.64 ms in eight, so the compute-bound FP32 path asks for
    // three waves; the BF16 path, bound by the copies, for one.  At most
    // kMaxBlocks.
    const int64_t min_rows =
        round_up(waves * (int64_t)st->sm_count * 128 * 128 / std::max<int64_t>(N, 128), 256);
    int64_t nblk = std::min<int64_t>(kMaxBlocks, std::max<int64_t>(1, M / min_rows));
    const int64_t mb = round_up((M + nblk - 1) / nblk, 256);
    nblk = (M + mb - 1) / mb;

    // Enqueues the whole pipeline; returns at the first failing call.
    auto enqueue = [&]() -> int {
        cudaEvent_t eB = hp->events[0];
        if (reads_ab) {
            if (!copy_rows(dB, ldb_d * ab_esz, B, ldb * ab_esz, N * ab_esz, K,
                           cudaMemcpyHostToDevice, hp->in))
                return GEMM_ERR_CUDA;
        }
        if (cudaEventRecord(eB, hp->in) != cudaSuccess ||
            cudaStreamWaitEvent(hp->compute, eB, 0) != cudaSuccess)
            return GEMM_ERR_CUDA;
        for (int64_t i = 0; i < nblk; ++i) {
            const int64_t r0 = i * mb, m = std::min(mb, M - r0);
            cudaEvent_t eIn = hp->events[1 + 2 * i], eOut = hp->events[2 + 2 * i];
            if (reads_ab &&
                !copy_rows(dA + r0 * lda_d * ab_esz, lda_d * ab_esz,
                           static_cast<const char *>(A) + r0 * lda * ab_esz, lda * ab_esz,
                           K * ab_esz, m, cudaMemcpyHostToDevice, hp->in))
                return GEMM_ERR_CUDA;
            if (beta != 0.f &&
                !copy_rows(dC + r0 * ldc_d * c_esz, ldc_d * c_esz,
                           static_cast<const char *>(C) + r0 * ldc * c_esz, ldc * c_esz,
                           N * c_esz, m, cudaMemcpyHostToDevice, hp->in))
                return GEMM_ERR_CUDA;
            if (cudaEventRecord(eIn, hp->in) != cudaSuccess ||
                cudaStreamWaitEvent(hp->compute, eIn, 0) != cudaSuccess)
                return GEMM_ERR_CUDA;
            const int r = device_gemm(m, reads_ab ? dA + r0 * lda_d * ab_esz : nullptr, lda_d,
                                      dB, ldb_d, dC + r0 * ldc_d * c_esz, ldc_d, hp->compute);
            if (r != GEMM_OK) return r;
            if (cudaEventRecord(eOut, hp->compute) != cudaSuccess ||
                cudaStreamWaitEvent(hp->out, eOut, 0) != cudaSuccess)
                return GEMM_ERR_CUDA;
            if (!copy_rows(static_cast<char *>(C) + r0 * ldc * c_esz, ldc * c_esz,
                           dC + r0 * ldc_d * c_esz, ldc_d * c_esz, N * c_esz, m,
                           cudaMemcpyDeviceToHost, hp->out))
                return GEMM_ERR_CUDA;
        }
        return GEMM_OK;
    };
    if ((rc = enqueue()) != GEMM_OK) {
        // Copies and GEMMs of earlier blocks may still be running, some
        // writing the caller's C: let them finish before the caller gets
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

}  // namespace
}  // namespace gemm

using namespace gemm;

extern "C" int gemm_f32_host(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                             int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                             int64_t ldc) {
    int rc = validate_gemm_args(M, N, K, alpha, A, lda, 4, B, ldb, 4, beta, C, ldc, 4);
    if (rc == 1) return GEMM_OK;
    if (rc != GEMM_OK) return rc;
    return run_host(M, N, K, alpha, A, lda, 4, B, ldb, beta, C, ldc, 4, 3,
                    [&](int64_t m, const char *dA, int64_t lda_d, const char *dB, int64_t ldb_d,
                        char *dC, int64_t ldc_d, cudaStream_t s) {
                        return gemm_f32(m, N, K, alpha, reinterpret_cast<const float *>(dA),
                                        lda_d, reinterpret_cast<const float *>(dB), ldb_d, beta,
                                        reinterpret_cast<float *>(dC), ldc_d, s);
                    });
}

extern "C" int gemm_bf16_host(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t *A,
                              int64_t lda, const uint16_t *B, int64_t ldb, float beta, void *C,
                              int64_t ldc, int c_type) {
    if (c_type != GEMM_OUT_BF16 && c_type != GEMM_OUT_F32) return GEMM_ERR_INVALID_ARG;
    const size_t c_esz = c_type == GEMM_OUT_F32 ? 4 : 2;
    int rc = validate_gemm_args(M, N, K, alpha, A, lda, 2, B, ldb, 2, beta, C, ldc, c_esz);
    if (rc == 1) return GEMM_OK;
    if (rc != GEMM_OK) return rc;
    return run_host(M, N, K, alpha, A, lda, 2, B, ldb, beta, C, ldc, c_esz, 1,
                    [&](int64_t m, const char *dA, int64_t lda_d, const char *dB, int64_t ldb_d,
                        char *dC, int64_t ldc_d, cudaStream_t s) {
                        return gemm_bf16(m, N, K, alpha, reinterpret_cast<const uint16_t *>(dA),
                                         lda_d, reinterpret_cast<const uint16_t *>(dB), ldb_d,
                                         beta, dC, ldc_d, c_type, s);
                    });
}
