// C-ABI front end of libgemm_gb300.so (declared in include/gemm_gb300.h):
// argument checking, per-device state, configuration knobs, dispatch to the
// kernels, and the device fault word.  Every numeric step runs on the GPU;
// this file only validates and launches.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gemm_gb300.h"
#include "internal.h"

namespace gemm {
namespace {

std::atomic<int64_t> g_watchdog_ms{2000};
std::atomic<int64_t> g_force_path{0};
std::atomic<int64_t> g_fault_inject{0};
std::atomic<int64_t> g_split_k{0};
std::atomic<int64_t> g_bf16_tile_n{0};
std::atomic<int64_t> g_tail_split_off{0};
std::atomic<int64_t> g_raster_group{0};
std::atomic<int64_t> g_cta_pair{0};
std::atomic<int64_t> g_last_fault{0};

std::mutex g_state_mu;
DeviceState g_state[kMaxDevices];

thread_local const char *t_last_kernel = "none";

constexpr int64_t kMaxDim = 0x7fffffffLL;

bool ranges_overlap(const void *a, size_t a_bytes, const void *b, size_t b_bytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + b_bytes && b0 < a0 + a_bytes;
}

// Bytes spanned by a rows x cols row-major matrix with pitch ld.
size_t span_bytes(int64_t rows, int64_t cols, int64_t ld, size_t esz) {
    if (rows <= 0 || cols <= 0) return 0;
    return (size_t)((rows - 1) * ld + cols) * esz;
}

}  // namespace

int validate_gemm_args(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
                       size_t a_esz, const void *B, int64_t ldb, size_t b_esz, float beta,
                       const void *C, int64_t ldc, size_t c_esz) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim || lda > kMaxDim || ldb > kMaxDim ||
        ldc > kMaxDim)
        return GEMM_ERR_TOO_LARGE;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
        return GEMM_ERR_BAD_LD;
    if (M == 0 || N == 0) return 1;
    if (!C) return GEMM_ERR_NULLPTR;
    const bool reads_ab = (alpha != 0.f) && K > 0;
    if (reads_ab) {
        if (!A || !B) return GEMM_ERR_NULLPTR;
        const size_t cb = span_bytes(M, N, ldc, c_esz);
        if (ranges_overlap(C, cb, A, span_bytes(M, K, lda, a_esz)) ||
            ranges_overlap(C, cb, B, span_bytes(K, N, ldb, b_esz)))
            return GEMM_ERR_ALIAS;
    }
    (void)beta;
    return GEMM_OK;
}

int device_state(DeviceState **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_state_mu);
    DeviceState &st = g_state[dev];
    if (st.device < 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED_DEVICE;
        unsigned long long *fw = nullptr;
        if (cudaMalloc(&fw, sizeof(*fw)) != cudaSuccess) return GEMM_ERR_CUDA;
        if (cudaMemset(fw, 0, sizeof(*fw)) != cudaSuccess) {
            cudaFree(fw);
            return GEMM_ERR_CUDA;
        }
        st.fault_word = fw;
        st.sm_count = sms;
        st.device = dev;
    }
    *out = &st;
    return GEMM_OK;
}

int ensure_splitk_workspace(DeviceState *st, size_t ws_bytes, size_t n_counters) {
    std::lock_guard<std::mutex> lock(g_state_mu);
    if (st->splitk_ws_bytes < ws_bytes) {
        // Stream-ordered work may still read the old buffer.
        if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
        if (st->splitk_ws) cudaFree(st->splitk_ws);
        st->splitk_ws = nullptr;
        st->splitk_ws_bytes = 0;
        if (cudaMalloc(&st->splitk_ws, ws_bytes) != cudaSuccess) return GEMM_ERR_CUDA;
        st->splitk_ws_bytes = ws_bytes;
    }
    if (st->splitk_counters_n < n_counters) {
        if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
        if (st->splitk_counters) cudaFree(st->splitk_counters);
        st->splitk_counters = nullptr;
        st->splitk_counters_n = 0;
        if (cudaMalloc(&st->splitk_counters, n_counters * sizeof(unsigned)) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (cudaMemset(st->splitk_counters, 0, n_counters * sizeof(unsigned)) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
        st->splitk_counters_n = n_counters;
    }
    return GEMM_OK;
}

RuntimeConfig runtime_config() {
    return RuntimeConfig{g_watchdog_ms.load(), g_force_path.load(), g_fault_inject.load(),
                         g_split_k.load(),      g_bf16_tile_n.load(), g_tail_split_off.load(),
                         g_raster_group.load(), g_cta_pair.load()};
}

void consume_fault_inject() { g_fault_inject.store(0); }

void set_last_kernel(const char *name) { t_last_kernel = name; }

}  // namespace gemm

using namespace gemm;

extern "C" int gemm_f32(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                        int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                        int64_t ldc, void *stream) {
    int rc = validate_gemm_args(M, N, K, alpha, A, lda, 4, B, ldb, 4, beta, C, ldc, 4);
    if (rc == 1) {
        set_last_kernel("none");
        return GEMM_OK;
    }
    if (rc != GEMM_OK) return rc;
    DeviceState *st = nullptr;
    if ((rc = device_state(&st)) != GEMM_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (alpha == 0.f || K == 0) {
        e = launch_scale_c((int)M, (int)N, beta, C, ldc, true, s);
        set_last_kernel("scale_c");
    } else {
        // TMA needs 16-byte aligned bases and pitches that are multiples of
        // 16 bytes (4 floats); other operands take the cp.async kernel.
        const bool tma_ok = ((reinterpret_cast<uintptr_t>(A) & 15) == 0) &&
                            ((reinterpret_cast<uintptr_t>(B) & 15) == 0) && (lda % 4 == 0) &&
                            (ldb % 4 == 0);
        if (tma_ok && runtime_config().force_path != 1) {
            rc = launch_sgemm_tma(st, (int)M, (int)N, (int)K, alpha, A, lda, B, ldb, beta, C,
                                  ldc, s);
            if (rc == GEMM_OK) set_last_kernel("sgemm_tma");
            return rc;
        }
        e = launch_sgemm_simt((int)M, (int)N, (int)K, alpha, A, lda, B, ldb, beta, C, ldc, s);
        set_last_kernel("sgemm_simt");
    }
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

extern "C" int gemm_bf16(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t *A,
                         int64_t lda, const uint16_t *B, int64_t ldb, float beta, void *C,
                         int64_t ldc, int c_type, void *stream) {
    if (c_type != GEMM_OUT_BF16 && c_type != GEMM_OUT_F32) return GEMM_ERR_INVALID_ARG;
    const bool c_f32 = (c_type == GEMM_OUT_F32);
    int rc = validate_gemm_args(M, N, K, alpha, A, lda, 2, B, ldb, 2, beta, C, ldc, c_f32 ? 4 : 2);
    if (rc == 1) {
        set_last_kernel("none");
        return GEMM_OK;
    }
    if (rc != GEMM_OK) return rc;
    DeviceState *st = nullptr;
    if ((rc = device_state(&st)) != GEMM_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (alpha == 0.f || K == 0) {
        set_last_kernel("scale_c");
        return launch_scale_c((int)M, (int)N, beta, C, ldc, c_f32, s) == cudaSuccess
                   ? GEMM_OK
                   : GEMM_ERR_CUDA;
    }
    // TMA needs 16-byte aligned bases and row pitches that are multiples of
    // 16 bytes (8 bf16 elements).
    const bool tma_ok = ((reinterpret_cast<uintptr_t>(A) & 15) == 0) &&
                        ((reinterpret_cast<uintptr_t>(B) & 15) == 0) && (lda % 8 == 0) &&
                        (ldb % 8 == 0);
    const int64_t force = runtime_config().force_path;
    if (force == 2 && !tma_ok) return GEMM_ERR_INVALID_ARG;
    if (tma_ok && force != 1) {
        rc = launch_bf16_tcgen05(st, (int)M, (int)N, (int)K, alpha, A, lda, B, ldb, beta, C, ldc,
                                 c_f32, s);
        if (rc == GEMM_OK) set_last_kernel("bf16_tcgen05");
        return rc;
    }
    const cudaError_t e = launch_gemm_simt_generic((int)M, (int)N, (int)K, alpha, A, lda, B, ldb,
                                                   beta, C, ldc, true, c_f32, s);
    if (e == cudaSuccess) set_last_kernel("bf16_simt");
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

extern "C" int gemm_get_device_status(void *stream) {
    DeviceState *st = nullptr;
    int rc = device_state(&st);
    if (rc != GEMM_OK) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GEMM_ERR_CUDA;
    unsigned long long word = 0;
    if (cudaMemcpy(&word, st->fault_word, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (word == 0) return GEMM_OK;
    g_last_fault.store((int64_t)(word & ~kFaultFlag));
    if (cudaMemset(st->fault_word, 0, sizeof(word)) != cudaSuccess) return GEMM_ERR_CUDA;
    // A kernel that gave up may have left split-K tile counters mid-count.
    {
        std::lock_guard<std::mutex> lock(g_state_mu);
        if (st->splitk_counters &&
            cudaMemset(st->splitk_counters, 0, st->splitk_counters_n * sizeof(unsigned)) !=
                cudaSuccess)
            return GEMM_ERR_CUDA;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
    return GEMM_ERR_DEVICE_TIMEOUT;
}

extern "C" int64_t gemm_get_device_fault_info(void) { return g_last_fault.load(); }

extern "C" const char *gemm_status_string(int status) {
    switch (status) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG: invalid argument";
        case GEMM_ERR_NULLPTR: return "GEMM_ERR_NULLPTR: required pointer is NULL";
        case GEMM_ERR_BAD_LD: return "GEMM_ERR_BAD_LD: leading dimension too small";
        case GEMM_ERR_UNSUPPORTED_DEVICE:
            return "GEMM_ERR_UNSUPPORTED_DEVICE: needs a compute capability 10.3 GPU";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: a CUDA call failed";
        case GEMM_ERR_DEVICE_TIMEOUT:
            return "GEMM_ERR_DEVICE_TIMEOUT: a GPU pipeline wait ran out of time";
        case GEMM_ERR_ALIAS: return "GEMM_ERR_ALIAS: C overlaps A or B";
        case GEMM_ERR_TOO_LARGE: return "GEMM_ERR_TOO_LARGE: dimension exceeds 2^31-1";
        case GEMM_ERR_SCRATCH_LIMIT:
            return "GEMM_ERR_SCRATCH_LIMIT: needs more split-K scratch than the static maximum";
        default: return "unknown gemm status";
    }
}

extern "C" int gemm_set_config(const char *key, int64_t value) {
    if (!key) return GEMM_ERR_INVALID_ARG;
    if (!strcmp(key, "watchdog_ms")) {
        if (value < 1 || value > 600000) return GEMM_ERR_INVALID_ARG;
        g_watchdog_ms.store(value);
    } else if (!strcmp(key, "force_path")) {
        if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
        g_force_path.store(value);
    } else if (!strcmp(key, "fault_inject")) {
        if (value < 0 || value > 1) return GEMM_ERR_INVALID_ARG;
        g_fault_inject.store(value);
    } else if (!strcmp(key, "split_k")) {
        if (value < 0 || value > 64) return GEMM_ERR_INVALID_ARG;
        g_split_k.store(value);
    } else if (!strcmp(key, "bf16_tile_n")) {
        if (value != 0 && value != 128 && value != 256) return GEMM_ERR_INVALID_ARG;
        g_bf16_tile_n.store(value);
    } else if (!strcmp(key, "tail_split_off")) {
        if (value < 0 || value > 1) return GEMM_ERR_INVALID_ARG;
        g_tail_split_off.store(value);
    } else if (!strcmp(key, "raster_group")) {
        if (value < 0 || value > 1024) return GEMM_ERR_INVALID_ARG;
        g_raster_group.store(value);
    } else if (!strcmp(key, "cta_pair")) {
        if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
        g_cta_pair.store(value);
    } else {
        return GEMM_ERR_INVALID_ARG;
    }
    return GEMM_OK;
}

extern "C" int gemm_get_config(const char *key, int64_t *value) {
    if (!key || !value) return GEMM_ERR_INVALID_ARG;
    if (!strcmp(key, "watchdog_ms")) *value = g_watchdog_ms.load();
    else if (!strcmp(key, "force_path")) *value = g_force_path.load();
    else if (!strcmp(key, "fault_inject")) *value = g_fault_inject.load();
    else if (!strcmp(key, "split_k")) *value = g_split_k.load();
    else if (!strcmp(key, "bf16_tile_n")) *value = g_bf16_tile_n.load();
    else if (!strcmp(key, "tail_split_off")) *value = g_tail_split_off.load();
    else if (!strcmp(key, "raster_group")) *value = g_raster_group.load();
    else if (!strcmp(key, "cta_pair")) *value = g_cta_pair.load();
    else return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

extern "C" const char *gemm_last_kernel(void) { return t_last_kernel; }

extern "C" int gemm_shutdown(void) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GEMM_OK;
    std::lock_guard<std::mutex> lock(g_state_mu);
    DeviceState &st = g_state[dev];
    if (st.device < 0) return GEMM_OK;
    if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
    if (st.fault_word) cudaFree(st.fault_word);
    if (st.splitk_ws) cudaFree(st.splitk_ws);
    if (st.splitk_counters) cudaFree(st.splitk_counters);
    st = DeviceState{};
    return GEMM_OK;
}

extern "C" int gemm_abi_version(void) { return 1; }
