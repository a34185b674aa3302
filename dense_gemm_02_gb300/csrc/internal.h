// Internal interfaces between the C-ABI front end (gemm_api.cu) and the
// kernel translation units.  Nothing here is part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_gb300.h"

namespace gemm {

constexpr int kMaxDevices = 64;

// Device fault word layout (written once per fault by the first failing
// thread with atomicCAS; 0 means no fault).
constexpr unsigned long long kFaultFlag = 1ull << 63;
enum FaultRole : unsigned { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3, kRoleSimt = 4 };

__host__ __device__ constexpr unsigned long long fault_code(unsigned role, unsigned stage,
                                                            unsigned tile) {
    return kFaultFlag | (unsigned long long)(role & 0xff) |
           ((unsigned long long)(stage & 0xff) << 8) |
           ((unsigned long long)tile << 16);
}

// Per-device library state, created on the first call on a device.
struct DeviceState {
    int device = -1;
    int sm_count = 0;
    unsigned long long *fault_word = nullptr;  // device, 8 bytes
    // split-K workspace: fp32 partial tiles, then one uint32 counter per tile
    float *splitk_ws = nullptr;
    size_t splitk_ws_bytes = 0;
    unsigned *splitk_counters = nullptr;
    size_t splitk_counters_n = 0;
};

// Returns the state of the current device (creating it), or an error.
int device_state(DeviceState **out);

// Grows the split-K workspace of `st` to hold ws_bytes of partials and n
// counters (zeroed).  Synchronous; only called outside the hot loop.
int ensure_splitk_workspace(DeviceState *st, size_t ws_bytes, size_t n_counters);

struct RuntimeConfig {
    int64_t watchdog_ms;
    int64_t force_path;
    int64_t fault_inject;
    int64_t split_k;
    int64_t bf16_tile_n;
    int64_t tail_split_off;
    int64_t raster_group;
    int64_t cta_pair;
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

// Encodes a 2-D tiled tensor map (cuTensorMapEncodeTiled through the
// runtime's driver entry point): `inner` contiguous elements per row,
// `outer` rows, `pitch_bytes` between rows, boxes of box_inner x box_outer.
// Out-of-range reads return zero.  False if the driver call failed.
bool encode_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                          uint64_t inner, uint64_t outer, uint64_t pitch_bytes,
                          uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

// ---- kernel launchers (return cudaSuccess or the launch error) ----

cudaError_t launch_sgemm_simt(int M, int N, int K, float alpha, const float *A, int64_t lda,
                              const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                              cudaStream_t stream);

// FP32 SGEMM fed by TMA.  Needs 16-byte aligned A/B bases and lda, ldb
// multiples of 4.  Returns a gemm_status_t.
int launch_sgemm_tma(DeviceState *st, int M, int N, int K, float alpha, const float *A,
                     int64_t lda, const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                     cudaStream_t stream);

// Generic SIMT GEMM for any alignment; a_bf16/b_bf16 select bf16 operands,
// c_f32 selects an fp32 (else bf16) C.
cudaError_t launch_gemm_simt_generic(int M, int N, int K, float alpha, const void *A,
                                     int64_t lda, const void *B, int64_t ldb, float beta,
                                     void *C, int64_t ldc, bool bf16_in, bool c_f32,
                                     cudaStream_t stream);

// C = beta * C (C = 0 without reading it when beta == 0).
cudaError_t launch_scale_c(int M, int N, float beta, void *C, int64_t ldc, bool c_f32,
                           cudaStream_t stream);

// Host-side argument checks shared by the entry points.  Returns GEMM_OK,
// an error, or 1 for "valid, nothing to do" (M == 0 or N == 0).
int validate_gemm_args(int64_t M, int64_t N, int64_t K, float alpha, const void *A, int64_t lda,
                       size_t a_esz, const void *B, int64_t ldb, size_t b_esz, float beta,
                       const void *C, int64_t ldc, size_t c_esz);

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
                                 int64_t ldc, bool c_f32, cudaStream_t stream);

// BF16 tcgen05 GEMM.  Requires 16-byte aligned A/B bases and lda, ldb
// multiples of 8.  Returns a gemm_status_t.
int launch_bf16_tcgen05(DeviceState *st, int M, int N, int K, float alpha, const uint16_t *A,
                        int64_t lda, const uint16_t *B, int64_t ldb, float beta, void *C,
                        int64_t ldc, bool c_f32, cudaStream_t stream);

}  // namespace gemm
