// C-ABI front end of libgemm_gb300.so (declared in include/gemm_gb300.h):
// argument checking, per-device state, configuration knobs, dispatch to the
// kernels, and the device fault word.  Every numeric step runs on the GPU;
// this file only validates and launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

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
std::atomic<int64_t> g_stream_k{0};
std::atomic<int64_t> g_pair_limit{0};
std::atomic<int64_t> g_stage_pairs{0};
std::atomic<int64_t> g_kpair_maps_off{0};
std::atomic<int64_t> g_last_fault{0};

std::mutex g_state_mu;
DeviceState g_state[kMaxDevices];

thread_local const char *t_last_kernel = "none";

constexpr int64_t kMaxDim = 0x7fffffffLL;

}  // namespace

int validate_gemm_args(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
                       size_t a_esz, const void *B, int64_t ldb, size_t b_esz, float beta,
                       const void *C, int64_t ldc, size_t c_esz) {
    return validate_gemm_args_ex(M, N, K, alpha, A, lda, a_esz, false, B, ldb, b_esz, false, beta,
                                 C, ldc, c_esz);
}

int validate_gemm_args_ex(int64_t M, int64_t N, int64_t K, float alpha, const void *A,
                          int64_t lda, size_t a_esz, bool trans_a, const void *B, int64_t ldb,
                          size_t b_esz, bool trans_b, float beta, const void *C, int64_t ldc,
                          size_t c_esz) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim || lda > kMaxDim || ldb > kMaxDim ||
        ldc > kMaxDim)
        return GEMM_ERR_TOO_LARGE;
    // Stored shapes: A is M x K (K x M when transposed), B is K x N (N x K).
    const int64_t a_rows = trans_a ? K : M, a_cols = trans_a ? M : K;
    const int64_t b_rows = trans_b ? N : K, b_cols = trans_b ? K : N;
    if (lda < (a_cols > 1 ? a_cols : 1) || ldb < (b_cols > 1 ? b_cols : 1) ||
        ldc < (N > 1 ? N : 1))
        return GEMM_ERR_BAD_LD;
    if (M == 0 || N == 0) return 1;
    if (!C) return GEMM_ERR_NULLPTR;
    const bool reads_ab = (alpha != 0.f) && K > 0;
    if (reads_ab) {
        if (!A || !B) return GEMM_ERR_NULLPTR;
        const size_t cb = span_bytes(M, N, ldc, c_esz);
        if (ranges_overlap(C, cb, A, span_bytes(a_rows, a_cols, lda, a_esz)) ||
            ranges_overlap(C, cb, B, span_bytes(b_rows, b_cols, ldb, b_esz)))
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

int stream_workspace(DeviceState *st, cudaStream_t stream, size_t ws_bytes, size_t n_counters,
                     Workspace **out) {
    std::lock_guard<std::mutex> lock(g_state_mu);
    Workspace *w = nullptr;
    for (auto &p : st->workspaces)
        if (p->stream == stream) w = p.get();
    if (!w) {
        st->workspaces.push_back(std::make_unique<Workspace>());
        w = st->workspaces.back().get();
        w->stream = stream;
    }
    if (w->ws_bytes < ws_bytes) {
        // Work already queued on this stream may still read the old buffer.
        if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
        if (w->ws) cudaFree(w->ws);
        w->ws = nullptr;
        w->ws_bytes = 0;
        if (cudaMalloc(&w->ws, ws_bytes) != cudaSuccess) return GEMM_ERR_CUDA;
        w->ws_bytes = ws_bytes;
    }
    if (w->counters_n < n_counters) {
        if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
        if (w->counters) cudaFree(w->counters);
        w->counters = nullptr;
        w->counters_n = 0;
        if (cudaMalloc(&w->counters, n_counters * sizeof(unsigned)) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (cudaMemset(w->counters, 0, n_counters * sizeof(unsigned)) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
        w->counters_n = n_counters;
    }
    *out = w;
    return GEMM_OK;
}

RuntimeConfig runtime_config() {
    return RuntimeConfig{g_watchdog_ms.load(), g_force_path.load(), g_fault_inject.load(),
                         g_split_k.load(),      g_bf16_tile_n.load(), g_tail_split_off.load(),
                         g_raster_group.load(), g_cta_pair.load(), g_stream_k.load(),
                         g_pair_limit.load(),   g_stage_pairs.load(), g_kpair_maps_off.load()};
}

void consume_fault_inject() { g_fault_inject.store(0); }

void set_last_kernel(const char *name) { t_last_kernel = name; }

}  // namespace gemm

namespace gemm {
namespace {

// Checks the public options and converts them.  A NULL opts gives the
// plain layouts and epilogue.
int convert_opts(const gemm_opts_t *opts, GemmOpts *out) {
    *out = GemmOpts{};
    if (!opts) return GEMM_OK;
    if ((opts->trans_a != 0 && opts->trans_a != 1) || (opts->trans_b != 0 && opts->trans_b != 1))
        return GEMM_ERR_INVALID_ARG;
    if (opts->act != GEMM_ACT_NONE && opts->act != GEMM_ACT_RELU &&
        opts->act != GEMM_ACT_GELU_TANH)
        return GEMM_ERR_INVALID_ARG;
    if (opts->bias_type != GEMM_OUT_BF16 && opts->bias_type != GEMM_OUT_F32)
        return GEMM_ERR_INVALID_ARG;
    out->trans_a = opts->trans_a;
    out->trans_b = opts->trans_b;
    out->bias = opts->bias;
    out->bias_f32 = (opts->bias_type == GEMM_OUT_F32) ? 1 : 0;
    out->act = opts->act;
    return GEMM_OK;
}

bool has_epilogue(const GemmOpts &o) { return o.bias != nullptr || o.act != GEMM_ACT_NONE; }

// Strided-batch checks, after the per-matrix ones: non-negative strides; C
// matrices that do not overlap one another; C clear of every A, B and bias
// byte the batch reads.
int check_batch(const GemmOpts &o, int64_t M, int64_t N, int64_t K, float alpha, const void *A,
                int64_t lda, size_t a_esz, const void *B, int64_t ldb, size_t b_esz,
                const void *C, int64_t ldc, size_t c_esz) {
    if (o.batch <= 1) return GEMM_OK;
    if (o.stride_a < 0 || o.stride_b < 0 || o.stride_c < 0) return GEMM_ERR_INVALID_ARG;
    if (o.batch > kMaxDim || o.stride_a > (int64_t(1) << 40) || o.stride_b > (int64_t(1) << 40) ||
        o.stride_c > (int64_t(1) << 40))
        return GEMM_ERR_TOO_LARGE;
    const size_t c_one = span_bytes(M, N, ldc, c_esz);
    if ((size_t)o.stride_c * c_esz < c_one) return GEMM_ERR_ALIAS;  // C matrices overlap
    const size_t c_all = (size_t)(o.batch - 1) * o.stride_c * c_esz + c_one;
    if (alpha != 0.f && K > 0) {
        const int64_t a_rows = o.trans_a ? K : M, a_cols = o.trans_a ? M : K;
        const int64_t b_rows = o.trans_b ? N : K, b_cols = o.trans_b ? K : N;
        const size_t a_all = (size_t)(o.batch - 1) * o.stride_a * a_esz +
                             span_bytes(a_rows, a_cols, lda, a_esz);
        const size_t b_all = (size_t)(o.batch - 1) * o.stride_b * b_esz +
                             span_bytes(b_rows, b_cols, ldb, b_esz);
        if (ranges_overlap(C, c_all, A, a_all) || ranges_overlap(C, c_all, B, b_all))
            return GEMM_ERR_ALIAS;
    }
    if (o.bias && ranges_overlap(C, c_all, o.bias, (size_t)N * (o.bias_f32 ? 4 : 2)))
        return GEMM_ERR_ALIAS;
    return GEMM_OK;
}

// Whether A and B (in their stored layouts, over the batch) can be fetched by
// TMA: 16-byte aligned bases, pitches and batch strides that are multiples
// of 16 bytes.
bool tma_operands_ok(const GemmOpts &o, int64_t M, int64_t N, int64_t K, const void *A,
                     int64_t lda, const void *B, int64_t ldb, size_t esz) {
    const int64_t q = 16 / (int64_t)esz;
    if ((reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15) ||
        lda % q || ldb % q)
        return false;
    const int64_t a_rows = o.trans_a ? K : M, b_rows = o.trans_b ? N : K;
    return tma_batch_stride_ok(o.batch, o.stride_a * (int64_t)esz, a_rows * lda * (int64_t)esz) &&
           tma_batch_stride_ok(o.batch, o.stride_b * (int64_t)esz, b_rows * ldb * (int64_t)esz);
}

// The same options for a launch that reads neither A nor B.
GemmOpts without_ab(const GemmOpts &o) {
    GemmOpts r = o;
    r.stride_a = r.stride_b = 0;
    return r;
}

// Shared by the plain and extended FP32 entry points.
int run_f32(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
            const float *B, int64_t ldb, float beta, float *C, int64_t ldc, const GemmOpts &o,
            void *stream) {
    int rc = validate_gemm_args_ex(M, N, K, alpha, A, lda, 4, o.trans_a, B, ldb, 4, o.trans_b,
                                   beta, C, ldc, 4);
    if (rc == 1) {
        set_last_kernel("none");
        return GEMM_OK;
    }
    if (rc != GEMM_OK) return rc;
    if (o.bias && ranges_overlap(C, span_bytes(M, N, ldc, 4), o.bias,
                                 (size_t)N * (o.bias_f32 ? 4 : 2)))
        return GEMM_ERR_ALIAS;
    if ((rc = check_batch(o, M, N, K, alpha, A, lda, 4, B, ldb, 4, C, ldc, 4)) != GEMM_OK)
        return rc;
    DeviceState *st = nullptr;
    if ((rc = device_state(&st)) != GEMM_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool epi = has_epilogue(o);
    cudaError_t e;
    if (alpha == 0.f || K == 0) {
        if (!epi) {
            e = launch_scale_c((int)M, (int)N, beta, C, ldc, true, o.batch, o.stride_c, s);
            set_last_kernel("scale_c");
        } else {  // act(bias) + beta * C: the generic kernel with an empty K loop
            const GemmOpts oc = without_ab(o);
            e = launch_gemm_simt_generic((int)M, (int)N, 0, alpha, nullptr, 1, nullptr, 1, beta,
                                         C, ldc, false, true, &oc, s);
            set_last_kernel("f32_simt");
        }
        return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }
    // TMA needs 16-byte aligned bases and pitches (and batch strides) that
    // are multiples of 16 bytes (4 floats).  Row-major operands take the
    // TMA kernel (or, one matrix without an epilogue, the cp.async kernel);
    // transposed ones, and others, the generic kernel.
    const bool tma_ok = tma_operands_ok(o, M, N, K, A, lda, B, ldb, 4);
    const bool row_major = !o.trans_a && !o.trans_b;
    if (row_major && tma_ok && runtime_config().force_path != 1) {
        rc = launch_sgemm_tma(st, (int)M, (int)N, (int)K, alpha, A, lda, B, ldb, beta, C, ldc,
                              &o, s);
        if (rc == GEMM_OK) set_last_kernel("sgemm_tma");
        return rc;
    }
    if (row_major && !epi && o.batch == 1) {
        e = launch_sgemm_simt((int)M, (int)N, (int)K, alpha, A, lda, B, ldb, beta, C, ldc, s);
        set_last_kernel("sgemm_simt");
    } else {
        e = launch_gemm_simt_generic((int)M, (int)N, (int)K, alpha, A, lda, B, ldb, beta, C, ldc,
                                     false, true, &o, s);
        set_last_kernel("f32_simt");
    }
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// Shared by the plain and extended BF16 entry points.
int run_bf16(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t *A, int64_t lda,
             const uint16_t *B, int64_t ldb, float beta, void *C, int64_t ldc, int c_type,
             const GemmOpts &o, void *stream) {
    if (c_type != GEMM_OUT_BF16 && c_type != GEMM_OUT_F32) return GEMM_ERR_INVALID_ARG;
    const bool c_f32 = (c_type == GEMM_OUT_F32);
    const size_t c_esz = c_f32 ? 4 : 2;
    int rc = validate_gemm_args_ex(M, N, K, alpha, A, lda, 2, o.trans_a, B, ldb, 2, o.trans_b,
                                   beta, C, ldc, c_esz);
    if (rc == 1) {
        set_last_kernel("none");
        return GEMM_OK;
    }
    if (rc != GEMM_OK) return rc;
    if (o.bias && ranges_overlap(C, span_bytes(M, N, ldc, c_esz), o.bias,
                                 (size_t)N * (o.bias_f32 ? 4 : 2)))
        return GEMM_ERR_ALIAS;
    if ((rc = check_batch(o, M, N, K, alpha, A, lda, 2, B, ldb, 2, C, ldc, c_esz)) != GEMM_OK)
        return rc;
    DeviceState *st = nullptr;
    if ((rc = device_state(&st)) != GEMM_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (alpha == 0.f || K == 0) {
        cudaError_t e;
        if (!has_epilogue(o)) {
            e = launch_scale_c((int)M, (int)N, beta, C, ldc, c_f32, o.batch, o.stride_c, s);
            set_last_kernel("scale_c");
        } else {  // act(bias) + beta * C: the generic kernel with an empty K loop
            const GemmOpts oc = without_ab(o);
            e = launch_gemm_simt_generic((int)M, (int)N, 0, alpha, nullptr, 1, nullptr, 1, beta,
                                         C, ldc, true, c_f32, &oc, s);
            set_last_kernel("bf16_simt");
        }
        return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    }
    // TMA needs 16-byte aligned bases and row pitches (and batch strides)
    // that are multiples of 16 bytes (8 bf16 elements), in either stored
    // layout.
    const bool tma_ok = tma_operands_ok(o, M, N, K, A, lda, B, ldb, 2);
    const int64_t force = runtime_config().force_path;
    if (force == 2 && !tma_ok) return GEMM_ERR_INVALID_ARG;
    if (tma_ok && force != 1) {
        rc = launch_bf16_tcgen05(st, (int)M, (int)N, (int)K, alpha, A, lda, B, ldb, beta, C, ldc,
                                 c_f32, &o, s);
        if (rc == GEMM_OK) set_last_kernel("bf16_tcgen05");
        return rc;
    }
    const cudaError_t e = launch_gemm_simt_generic((int)M, (int)N, (int)K, alpha, A, lda, B, ldb,
                                                   beta, C, ldc, true, c_f32, &o, s);
    if (e == cudaSuccess) set_last_kernel("bf16_simt");
    return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// Grouped GEMMs.  Every problem is checked as a single call would be; then
// the problems, which run concurrently, must not write what another one
// reads or writes: a C region may overlap no other region of the call
// (operands that are only read, such as a weight matrix shared by several
// problems, may overlap each other).  Checked by sorting the regions by
// start address and sweeping once.
int check_group_overlap(int64_t count, const gemm_group_t *g, const GemmOpts &o, size_t ab_esz,
                        size_t c_esz) {
    struct Region {
        uintptr_t lo, hi;
        bool write;
    };
    std::vector<Region> r;
    r.reserve((size_t)count * 3);
    for (int64_t i = 0; i < count; ++i) {
        const gemm_group_t &x = g[i];
        if (x.M == 0 || x.N == 0) continue;
        const size_t cb = span_bytes(x.M, x.N, x.ldc, c_esz);
        r.push_back({reinterpret_cast<uintptr_t>(x.C), reinterpret_cast<uintptr_t>(x.C) + cb, true});
        if (x.alpha != 0.f && x.K > 0) {
            const int64_t a_rows = o.trans_a ? x.K : x.M, a_cols = o.trans_a ? x.M : x.K;
            const int64_t b_rows = o.trans_b ? x.N : x.K, b_cols = o.trans_b ? x.K : x.N;
            const size_t ab = span_bytes(a_rows, a_cols, x.lda, ab_esz);
            const size_t bb = span_bytes(b_rows, b_cols, x.ldb, ab_esz);
            r.push_back({reinterpret_cast<uintptr_t>(x.A), reinterpret_cast<uintptr_t>(x.A) + ab,
                         false});
            r.push_back({reinterpret_cast<uintptr_t>(x.B), reinterpret_cast<uintptr_t>(x.B) + bb,
                         false});
        }
    }
    std::sort(r.begin(), r.end(), [](const Region &a, const Region &b) { return a.lo < b.lo; });
    uintptr_t end_w = 0, end_any = 0;  // furthest end of earlier written / any regions
    for (const Region &x : r) {
        if (x.hi <= x.lo) continue;
        if (x.lo < end_w || (x.write && x.lo < end_any)) return GEMM_ERR_ALIAS;
        if (x.write) end_w = std::max(end_w, x.hi);
        end_any = std::max(end_any, x.hi);
    }
    return GEMM_OK;
}

int run_grouped(bool bf16, int64_t count, const gemm_group_t *groups, int c_type,
                const gemm_opts_t *opts, void *stream) {
    GemmOpts o;
    int rc = convert_opts(opts, &o);
    if (rc != GEMM_OK) return rc;
    if (has_epilogue(o)) return GEMM_ERR_INVALID_ARG;  // plain epilogue only
    if (bf16 && c_type != GEMM_OUT_BF16 && c_type != GEMM_OUT_F32) return GEMM_ERR_INVALID_ARG;
    if (count < 0) return GEMM_ERR_INVALID_ARG;
    if (count > kMaxDim) return GEMM_ERR_TOO_LARGE;
    if (count == 0) {
        set_last_kernel("none");
        return GEMM_OK;
    }
    if (!groups) return GEMM_ERR_NULLPTR;
    const size_t ab_esz = bf16 ? 2 : 4;
    const bool c_f32 = !bf16 || c_type == GEMM_OUT_F32;
    const size_t c_esz = c_f32 ? 4 : 2;
    for (int64_t i = 0; i < count; ++i) {
        const gemm_group_t &x = groups[i];
        rc = validate_gemm_args_ex(x.M, x.N, x.K, x.alpha, x.A, x.lda, ab_esz, o.trans_a, x.B,
                                   x.ldb, ab_esz, o.trans_b, x.beta, x.C, x.ldc, c_esz);
        if (rc != GEMM_OK && rc != 1) return rc;
    }
    if ((rc = check_group_overlap(count, groups, o, ab_esz, c_esz)) != GEMM_OK) return rc;
    DeviceState *st = nullptr;
    if ((rc = device_state(&st)) != GEMM_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool force_other = runtime_config().force_path == 1;
    // Problems the grouped kernels take, and the rest one call at a time.
    std::vector<GroupProblem> fast;
    bool singles = false;  // some problem ran as a single call
    for (int64_t i = 0; i < count; ++i) {
        const gemm_group_t &x = groups[i];
        if (x.M == 0 || x.N == 0) continue;
        const bool tma = tma_operands_ok(o, x.M, x.N, x.K, x.A, x.lda, x.B, x.ldb, ab_esz);
        const bool ok = x.alpha != 0.f && x.K > 0 && tma && !force_other &&
                        (bf16 || (!o.trans_a && !o.trans_b));
        if (ok) {
            fast.push_back(GroupProblem{x.M, x.N, x.K, x.A, x.lda, x.B, x.ldb, x.C, x.ldc,
                                        x.alpha, x.beta});
            continue;
        }
        rc = bf16 ? run_bf16(x.M, x.N, x.K, x.alpha, static_cast<const uint16_t *>(x.A), x.lda,
                             static_cast<const uint16_t *>(x.B), x.ldb, x.beta, x.C, x.ldc,
                             c_type, o, stream)
                  : run_f32(x.M, x.N, x.K, x.alpha, static_cast<const float *>(x.A), x.lda,
                            static_cast<const float *>(x.B), x.ldb, x.beta,
                            static_cast<float *>(x.C), x.ldc, o, stream);
        if (rc != GEMM_OK) return rc;
        singles = true;
    }
    for (size_t i0 = 0; i0 < fast.size(); i0 += kMaxGroupsPerLaunch) {
        const int n = (int)std::min<size_t>(kMaxGroupsPerLaunch, fast.size() - i0);
        rc = bf16 ? launch_bf16_tcgen05_grouped(st, n, fast.data() + i0, c_f32, o.trans_a,
                                                o.trans_b, s)
                  : launch_sgemm_tma_grouped(st, n, fast.data() + i0, s);
        if (rc != GEMM_OK) return rc;
    }
    if (singles && !fast.empty())
        set_last_kernel(bf16 ? "bf16_grouped_mixed" : "f32_grouped_mixed");
    else if (!fast.empty())
        set_last_kernel(bf16 ? "bf16_tcgen05_grouped" : "sgemm_tma_grouped");
    else if (!singles)
        set_last_kernel("none");
    return GEMM_OK;
}

}  // namespace
}  // namespace gemm

using namespace gemm;

extern "C" int gemm_bf16_grouped(int64_t count, const gemm_group_t *groups, int c_type,
                                 const gemm_opts_t *opts, void *stream) {
    return run_grouped(true, count, groups, c_type, opts, stream);
}

extern "C" int gemm_f32_grouped(int64_t count, const gemm_group_t *groups,
                                const gemm_opts_t *opts, void *stream) {
    return run_grouped(false, count, groups, GEMM_OUT_F32, opts, stream);
}

extern "C" int gemm_f32(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                        int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                        int64_t ldc, void *stream) {
    GemmOpts o;
    convert_opts(nullptr, &o);
    return run_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, o, stream);
}

extern "C" int gemm_f32_ex(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                           int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                           int64_t ldc, const gemm_opts_t *opts, void *stream) {
    GemmOpts o;
    const int rc = convert_opts(opts, &o);
    if (rc != GEMM_OK) return rc;
    return run_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, o, stream);
}

extern "C" int gemm_bf16(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t *A,
                         int64_t lda, const uint16_t *B, int64_t ldb, float beta, void *C,
                         int64_t ldc, int c_type, void *stream) {
    GemmOpts o;
    convert_opts(nullptr, &o);
    return run_bf16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, c_type, o, stream);
}

extern "C" int gemm_bf16_ex(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t *A,
                            int64_t lda, const uint16_t *B, int64_t ldb, float beta, void *C,
                            int64_t ldc, int c_type, const gemm_opts_t *opts, void *stream) {
    GemmOpts o;
    const int rc = convert_opts(opts, &o);
    if (rc != GEMM_OK) return rc;
    return run_bf16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, c_type, o, stream);
}

extern "C" int gemm_bf16_batched(int64_t batch, int64_t M, int64_t N, int64_t K, float alpha,
                                 const uint16_t *A, int64_t lda, int64_t stride_a,
                                 const uint16_t *B, int64_t ldb, int64_t stride_b, float beta,
                                 void *C, int64_t ldc, int64_t stride_c, int c_type,
                                 const gemm_opts_t *opts, void *stream) {
    GemmOpts o;
    int rc = convert_opts(opts, &o);
    if (rc != GEMM_OK) return rc;
    if (batch < 0) return GEMM_ERR_INVALID_ARG;
    if (batch == 0) {
        set_last_kernel("none");
        return GEMM_OK;
    }
    o.batch = batch;
    o.stride_a = stride_a;
    o.stride_b = stride_b;
    o.stride_c = stride_c;
    return run_bf16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, c_type, o, stream);
}

extern "C" int gemm_f32_batched(int64_t batch, int64_t M, int64_t N, int64_t K, float alpha,
                                const float *A, int64_t lda, int64_t stride_a, const float *B,
                                int64_t ldb, int64_t stride_b, float beta, float *C, int64_t ldc,
                                int64_t stride_c, const gemm_opts_t *opts, void *stream) {
    GemmOpts o;
    int rc = convert_opts(opts, &o);
    if (rc != GEMM_OK) return rc;
    if (batch < 0) return GEMM_ERR_INVALID_ARG;
    if (batch == 0) {
        set_last_kernel("none");
        return GEMM_OK;
    }
    o.batch = batch;
    o.stride_a = stride_a;
    o.stride_b = stride_b;
    o.stride_c = stride_c;
    return run_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, o, stream);
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
        for (auto &w : st->workspaces)
            if (w->counters &&
                cudaMemset(w->counters, 0, w->counters_n * sizeof(unsigned)) != cudaSuccess)
                return GEMM_ERR_CUDA;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
    return fault_status(word);
}

extern "C" int64_t gemm_get_device_fault_info(void) { return g_last_fault.load(); }

extern "C" int gemm_debug_checks(void) { return GEMM_DEBUG ? 1 : 0; }

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
        case GEMM_ERR_ALIAS: return "GEMM_ERR_ALIAS: C overlaps A, B or the bias";
        case GEMM_ERR_TOO_LARGE: return "GEMM_ERR_TOO_LARGE: dimension exceeds 2^31-1";
        case GEMM_ERR_SCRATCH_LIMIT:
            return "GEMM_ERR_SCRATCH_LIMIT: needs more split-K scratch than the static maximum";
        case GEMM_ERR_DEVICE_CHECK:
            return "GEMM_ERR_DEVICE_CHECK: a debug-build device check failed (access skipped)";
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
    } else if (!strcmp(key, "stream_k")) {
        if (value < 0 || value > 1) return GEMM_ERR_INVALID_ARG;
        g_stream_k.store(value);
    } else if (!strcmp(key, "pair_limit")) {
        if (value < 0 || value > 1024) return GEMM_ERR_INVALID_ARG;
        g_pair_limit.store(value);
    } else if (!strcmp(key, "stage_pairs")) {
        if (value < 0 || value > 2) return GEMM_ERR_INVALID_ARG;
        g_stage_pairs.store(value);
    } else if (!strcmp(key, "kpair_maps_off")) {
        if (value < 0 || value > 1) return GEMM_ERR_INVALID_ARG;
        g_kpair_maps_off.store(value);
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
    else if (!strcmp(key, "stream_k")) *value = g_stream_k.load();
    else if (!strcmp(key, "pair_limit")) *value = g_pair_limit.load();
    else if (!strcmp(key, "stage_pairs")) *value = g_stage_pairs.load();
    else if (!strcmp(key, "kpair_maps_off")) *value = g_kpair_maps_off.load();
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
    for (auto &w : st.workspaces) {
        if (w->ws) cudaFree(w->ws);
        if (w->counters) cudaFree(w->counters);
    }
    if (st.host) {
        for (cudaEvent_t e : st.host->events) cudaEventDestroy(e);
        for (cudaStream_t s : {st.host->in, st.host->compute, st.host->out})
            if (s) cudaStreamDestroy(s);
        if (st.host->buf) cudaFree(st.host->buf);
    }
    st = DeviceState{};
    return GEMM_OK;
}

extern "C" int gemm_abi_version(void) { return 2; }
