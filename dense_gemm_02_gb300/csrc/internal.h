// Internal interfaces between the C-ABI front end (gemm_api.cu) and the
// kernel translation units.  Nothing here is part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <memory>
#include <mutex>
#include <vector>

#include "gemm_gb300.h"

namespace gemm {

constexpr int kMaxDevices = 64;

// One-time setup per device (function attributes, occupancy queries) that
// several host threads may reach at once: the first caller on a device runs
// `init` (0 = success) under a lock while the others wait; a failed setup
// is tried again by the next call.  Returns init's result, or 0 once done.
class PerDeviceOnce {
  public:
    template <class F>
    int run(int device, F &&init) {
        if (device < 0 || device >= kMaxDevices) return -1;
        if (done_[device].load(std::memory_order_acquire)) return 0;
        std::lock_guard<std::mutex> lock(mu_);
        if (done_[device].load(std::memory_order_relaxed)) return 0;
        const int rc = init();
        if (rc == 0) done_[device].store(true, std::memory_order_release);
        return rc;
    }

  private:
    std::mutex mu_;
    std::atomic<bool> done_[kMaxDevices] = {};
};

// Device fault word layout (written once per fault by the first failing
// thread with atomicCAS; 0 means no fault).
constexpr unsigned long long kFaultFlag = 1ull << 63;
enum FaultRole : unsigned {
    kRoleProducer = 1,
    kRoleMma = 2,
    kRoleEpilogue = 3,
    kRoleSimt = 4,
    kRoleCheck = 5  // a debug-build check failed; the stage byte holds its CheckSite
};

__host__ __device__ constexpr unsigned long long fault_code(unsigned role, unsigned stage,
                                                            unsigned tile) {
    return kFaultFlag | (unsigned long long)(role & 0xff) |
           ((unsigned long long)(stage & 0xff) << 8) |
           ((unsigned long long)tile << 16);
}

// Status a nonzero fault word reports: GEMM_ERR_DEVICE_CHECK for a failed
// debug-build check, else GEMM_ERR_DEVICE_TIMEOUT (a wait ran out).
inline int fault_status(unsigned long long word) {
    return (word & 0xff) == kRoleCheck ? GEMM_ERR_DEVICE_CHECK : GEMM_ERR_DEVICE_TIMEOUT;
}

// Debug build (compiled with GEMM_DEBUG=1 into libgemm_gb300_debug.so):
// device-side checks of the indices, copy coordinates and shared- and
// tensor-memory ranges the kernels compute.  A failed check records
// kRoleCheck and its site in the fault word (the first fault wins) and its
// caller skips the access it guards; waits that depended on that access then
// run out and the kernel leaves through its usual watchdog path.  In the
// release build every check is the constant true and compiles away.
#ifndef GEMM_DEBUG
#define GEMM_DEBUG 0
#endif
enum CheckSite : unsigned {
    kSiteLoadA = 1,      // a TMA load of A: x coordinate alignment, destination range
    kSiteLoadB = 2,      // the same for B
    kSiteStoreC = 3,     // a TMA store of C: x coordinate alignment, staging range
    kSiteTmem = 4,       // an accumulator's tensor-memory columns
    kSiteWorkspace = 5,  // a split-K partial tile or counter index
    kSiteSmemDesc = 6    // an MMA operand's shared-memory range
};

#if defined(__CUDACC__)
__device__ __forceinline__ bool debug_check(unsigned long long *fault_word, bool ok,
                                            unsigned site, unsigned tile) {
#if GEMM_DEBUG
    if (!ok) atomicCAS(fault_word, 0ull, fault_code(kRoleCheck, site, tile));
    return ok;
#else
    (void)fault_word;
    (void)ok;
    (void)site;
    (void)tile;
    return true;
#endif
}
#endif

// Split-K workspace of one stream: fp32 partial tiles and one uint32
// counter per split tile (each counter is back at zero after every launch).
// Launches on one stream run in order, so they may share it; launches on
// different streams may overlap and get different workspaces.
struct Workspace {
    cudaStream_t stream = nullptr;
    float *ws = nullptr;
    size_t ws_bytes = 0;
    unsigned *counters = nullptr;
    size_t counters_n = 0;
};

// State of the host-buffer entry points on one device: copy-in, compute and
// copy-out streams, their events, and one device staging allocation for A,
// B and C, grown on demand and kept.
struct HostPipe {
    cudaStream_t in = nullptr, compute = nullptr, out = nullptr;
    std::vector<cudaEvent_t> events;
    void *buf = nullptr;
    size_t bytes = 0;
};

// Per-device library state, created on the first call on a device.
struct DeviceState {
    int device = -1;
    int sm_count = 0;
    unsigned long long *fault_word = nullptr;  // device, 8 bytes
    std::vector<std::unique_ptr<Workspace>> workspaces;  // one per stream used
    std::unique_ptr<HostPipe> host;                      // gemm_*_host, on first use
};

// Returns the state of the current device (creating it), or an error.
int device_state(DeviceState **out);

// The workspace of `stream` on st's device, grown to hold ws_bytes of
// partials and n_counters counters (new counters zeroed).  Growing
// synchronises the device; it happens only when a launch needs more than
// any earlier one on that stream.
int stream_workspace(DeviceState *st, cudaStream_t stream, size_t ws_bytes, size_t n_counters,
                     Workspace **out);

struct RuntimeConfig {
    int64_t watchdog_ms;
    int64_t force_path;
    int64_t fault_inject;
    int64_t split_k;
    int64_t bf16_tile_n;
    int64_t tail_split_off;
    int64_t raster_group;
    int64_t cta_pair;
    int64_t stream_k;
    int64_t pair_limit;
    int64_t stage_pairs;
    int64_t kpair_maps_off;
};
RuntimeConfig runtime_config();
void consume_fault_inject();

void set_last_kernel(const char *name);

// Output-tile order shared by the kernels: tiles are walked in bands of
// `group` M-blocks, N-blocks varying slowest within a band, so that CTAs
// running at the same time reuse the same A rows and B columns in L2.
constexpr int kRasterGroup = 8;
__host__ __device__ __forceinline__ void grouped_tile_coords(int tile, int num_m, int num_n,
                                                             int group_m, int &m_blk,
                                                             int &n_blk) {
    const int per_group = group_m * num_n;
    const int group = tile / per_group;
    const int first_m = group * group_m;
    const int gm = (num_m - first_m < group_m) ? num_m - first_m : group_m;
    const int r = tile - group * per_group;
    m_blk = first_m + r % gm;
    n_blk = r / gm;
}

// Encodes a 3-D tiled tensor map (cuTensorMapEncodeTiled through the
// runtime's driver entry point) over `depth` matrices depth_stride_bytes
// apart, each `outer` rows of `inner` contiguous elements, `pitch_bytes`
// between rows; boxes of box_inner x box_outer x 1.  depth <= 1 is one
// matrix (the stride is then ignored).  Out-of-range reads return zero.
// False if the driver call failed.
bool encode_tensor_map_3d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                          uint64_t inner, uint64_t outer, uint64_t depth, uint64_t pitch_bytes,
                          uint64_t depth_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle swizzle);

// Whether a strided batch can be fetched by 3-D TMA: one matrix, or a batch
// stride (bytes) that is 0 (shared matrix) or a multiple of 16 no smaller
// than one matrix's span.
inline bool tma_batch_stride_ok(int64_t batch, int64_t stride_bytes, int64_t span_bytes) {
    return batch <= 1 || stride_bytes == 0 ||
           (stride_bytes % 16 == 0 && stride_bytes >= span_bytes);
}

// ---- kernel launchers (return cudaSuccess or the launch error) ----

// Operand layouts, fused epilogue and strided batch of the extended entry
// points (host side): trans_a: A stored K x M; trans_b: B stored N x K;
// bias: nullptr or N values (fp32 when bias_f32, else bf16); act: a
// gemm_act_t; batch matrices, matrix i at A + i * stride_a (elements; 0
// shares one matrix among all), likewise B and C.  A null GemmOpts pointer
// means one row-major product with the plain epilogue.
struct GemmOpts {
    int trans_a = 0, trans_b = 0;
    const void *bias = nullptr;
    int bias_f32 = 0;
    int act = 0;
    int64_t batch = 1;
    int64_t stride_a = 0, stride_b = 0, stride_c = 0;
};

cudaError_t launch_sgemm_simt(int M, int N, int K, float alpha, const float *A, int64_t lda,
                              const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                              cudaStream_t stream);

// FP32 SGEMM fed by TMA.  Needs 16-byte aligned A/B bases and lda, ldb
// multiples of 4.  Returns a gemm_status_t.
int launch_sgemm_tma(DeviceState *st, int M, int N, int K, float alpha, const float *A,
                     int64_t lda, const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                     const GemmOpts *opts, cudaStream_t stream);

// Generic SIMT GEMM for any alignment and layout; bf16_in selects bf16
// operands, c_f32 selects an fp32 (else bf16) C.  K == 0 (with any A, B)
// gives C = act(bias) + beta * C.
cudaError_t launch_gemm_simt_generic(int M, int N, int K, float alpha, const void *A,
                                     int64_t lda, const void *B, int64_t ldb, float beta,
                                     void *C, int64_t ldc, bool bf16_in, bool c_f32,
                                     const GemmOpts *opts, cudaStream_t stream);

// C = beta * C (C = 0 without reading it when beta == 0), for `batch`
// matrices stride_c elements apart.
cudaError_t launch_scale_c(int M, int N, float beta, void *C, int64_t ldc, bool c_f32,
                           int64_t batch, int64_t stride_c, cudaStream_t stream);

// Whether the byte ranges [a, a + a_bytes) and [b, b + b_bytes) meet.
inline bool ranges_overlap(const void *a, size_t a_bytes, const void *b, size_t b_bytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + b_bytes && b0 < a0 + a_bytes;
}

// Bytes spanned by a rows x cols row-major matrix with pitch ld.
inline size_t span_bytes(int64_t rows, int64_t cols, int64_t ld, size_t esz) {
    if (rows <= 0 || cols <= 0) return 0;
    return (size_t)((rows - 1) * ld + cols) * esz;
}

// Host-side argument checks shared by the entry points.  Returns GEMM_OK,
// an error, or 1 for "valid, nothing to do" (M == 0 or N == 0).
int validate_gemm_args(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
                       size_t a_esz, const void *B, int64_t ldb, size_t b_esz, float beta,
                       const void *C, int64_t ldc, size_t c_esz);
// The same with stored layouts: trans_a means A is stored K x M (lda >=
// max(1, M)), trans_b that B is stored N x K (ldb >= max(1, K)).
int validate_gemm_args_ex(int64_t M, int64_t N, int64_t K, float alpha, const void *A,
                          int64_t lda, size_t a_esz, bool trans_a, const void *B, int64_t ldb,
                          size_t b_esz, bool trans_b, float beta, const void *C, int64_t ldc,
                          size_t c_esz);

// One problem of a grouped GEMM (host side): C = alpha * op(A) * op(B) +
// beta * C with its own sizes, pointers and pitches (elements).
struct GroupProblem {
    int64_t M, N, K;
    const void *A;
    int64_t lda;
    const void *B;
    int64_t ldb;
    void *C;
    int64_t ldc;
    float alpha, beta;
};
// Groups one grouped launch can carry: their tensor maps and sizes travel in
// the kernel's parameters (up to 32 KiB), not in a device buffer.
constexpr int kMaxGroupsPerLaunch = 64;

// Grouped FP32 SGEMM on the TMA kernel: one launch over every tile of
// `count` (<= kMaxGroupsPerLaunch) problems, all with 16-byte aligned A/B
// bases, lda and ldb multiples of 4, M, N, K > 0 and alpha != 0.  Returns a
// gemm_status_t.
int launch_sgemm_tma_grouped(DeviceState *st, int count, const GroupProblem *g,
                             cudaStream_t stream);
// Grouped BF16 tcgen05 GEMM: one persistent launch over the union of the
// problems' output tiles, in the layouts trans_a / trans_b select (shared by
// all problems); the same preconditions with 16-byte aligned pitches (in
// elements: multiples of 8).  Returns a gemm_status_t.
int launch_bf16_tcgen05_grouped(DeviceState *st, int count, const GroupProblem *g, bool c_f32,
                                int trans_a, int trans_b, cudaStream_t stream);

// Split-K storage supplied by the caller instead of the library workspace.
struct ExternalScratch {
    float *ws;                       // fp32 partial tiles
    size_t ws_bytes;
    unsigned *counters;              // one per output tile; cleared before each launch
    size_t counters_n;
    unsigned long long *fault_word;  // pipeline fault record
};

// Same kernel as launch_bf16_tcgen05 with split-K storage from `ext`; never
// allocates.  GEMM_ERR_SCRATCH_LIMIT if the chosen split needs more.
int launch_bf16_tcgen05_external(int device, int sm_count, const ExternalScratch &ext, int M,
                                 int N, int K, float alpha, const uint16_t *A, int64_t lda,
                                 const uint16_t *B, int64_t ldb, float beta, void *C,
                                 int64_t ldc, bool c_f32, const GemmOpts *opts,
                                 cudaStream_t stream);

// BF16 tcgen05 GEMM.  Requires 16-byte aligned A/B bases and lda, ldb
// multiples of 8 (in whichever layout opts selects).  Returns a
// gemm_status_t.
int launch_bf16_tcgen05(DeviceState *st, int M, int N, int K, float alpha, const uint16_t *A,
                        int64_t lda, const uint16_t *B, int64_t ldb, float beta, void *C,
                        int64_t ldc, bool c_f32, const GemmOpts *opts, cudaStream_t stream);

}  // namespace gemm
