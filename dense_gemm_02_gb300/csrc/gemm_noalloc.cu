// gemm_bf16_noalloc: the BF16 tcgen05 GEMM for callers that cannot
// allocate device memory.  The split-K scratch (fault record, tile counters,
// fp32 partial tiles) is a file-scope device array compiled into the
// library, so no call ever allocates; the source pages have no counterpart.
//
// Host code cannot use the array's name as a device address (in host code it
// is a host-side stand-in), so the first call on each device, with that
// device current, asks the runtime for the array's device address once and
// keeps it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "gemm_gb300.h"
#include "internal.h"

namespace gemm {
namespace {

constexpr size_t kScratchBytes = GEMM_NOALLOC_SCRATCH_BYTES;
constexpr size_t kFaultOffset = 0;          // 8-byte fault record
constexpr size_t kCountersOffset = 256;     // one uint32 per output tile
constexpr size_t kMaxTiles = 4096;
constexpr size_t kPartialsOffset = kCountersOffset + kMaxTiles * sizeof(unsigned);  // 16640
static_assert(kPartialsOffset % 256 == 0, "partials must stay 256-byte aligned");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct ScratchSlot {
    std::once_flag once;
    int status = GEMM_ERR_CUDA;
    int sm_count = 0;
    unsigned char *base = nullptr;  // device address of g_noalloc_scratch
};
ScratchSlot g_slots[kMaxDevices];

// Once per device, with that device current: compute capability check, SM
// count, and the device address of the scratch array.
int scratch_for_current_device(int *device, ScratchSlot **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    ScratchSlot &slot = g_slots[dev];
    std::call_once(slot.once, [&slot, dev] {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            slot.status = GEMM_ERR_CUDA;
            return;
        }
        if (major != 10 || minor != 3) {
            slot.status = GEMM_ERR_UNSUPPORTED_DEVICE;
            return;
        }
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            slot.status = GEMM_ERR_CUDA;
            return;
        }
        // The fault record starts clear; afterwards only
        // gemm_noalloc_get_status clears it, so a fault stays visible
        // until the caller has asked.
        if (cudaMemset(static_cast<unsigned char *>(ptr) + kFaultOffset, 0,
                       sizeof(unsigned long long)) != cudaSuccess) {
            slot.status = GEMM_ERR_CUDA;
            return;
        }
        slot.base = static_cast<unsigned char *>(ptr);
        slot.sm_count = sms;
        slot.status = GEMM_OK;
    });
    *device = dev;
    *out = &slot;
    return slot.status;
}

}  // namespace
}  // namespace gemm

using namespace gemm;

extern "C" int gemm_bf16_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                 const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                                 float beta, void *C, int64_t ldc, int c_type, void *stream) {
    if (c_type != GEMM_OUT_BF16 && c_type != GEMM_OUT_F32) return GEMM_ERR_INVALID_ARG;
    const bool c_f32 = (c_type == GEMM_OUT_F32);
    int rc = validate_gemm_args(M, N, K, alpha, A, lda, 2, B, ldb, 2, beta, C, ldc,
                                c_f32 ? 4 : 2);
    if (rc == 1) return GEMM_OK;
    if (rc != GEMM_OK) return rc;
    int device = -1;
    ScratchSlot *slot = nullptr;
    if ((rc = scratch_for_current_device(&device, &slot)) != GEMM_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (alpha == 0.f || K == 0)
        return launch_scale_c((int)M, (int)N, beta, C, ldc, c_f32, 1, 0, s) == cudaSuccess
                   ? GEMM_OK
                   : GEMM_ERR_CUDA;
    const bool tma_ok = ((reinterpret_cast<uintptr_t>(A) & 15) == 0) &&
                        ((reinterpret_cast<uintptr_t>(B) & 15) == 0) && (lda % 8 == 0) &&
                        (ldb % 8 == 0);
    if (!tma_ok) return GEMM_ERR_INVALID_ARG;
    ExternalScratch ext;
    ext.fault_word = reinterpret_cast<unsigned long long *>(slot->base + kFaultOffset);
    ext.counters = reinterpret_cast<unsigned *>(slot->base + kCountersOffset);
    ext.counters_n = kMaxTiles;
    ext.ws = reinterpret_cast<float *>(slot->base + kPartialsOffset);
    ext.ws_bytes = kScratchBytes - kPartialsOffset;
    return launch_bf16_tcgen05_external(device, slot->sm_count, ext, (int)M, (int)N, (int)K,
                                        alpha, A, lda, B, ldb, beta, C, ldc, c_f32, nullptr, s);
}

extern "C" int gemm_noalloc_get_status(void *stream, int64_t *fault_info) {
    if (fault_info) *fault_info = 0;
    int device = -1;
    ScratchSlot *slot = nullptr;
    int rc = scratch_for_current_device(&device, &slot);
    if (rc != GEMM_OK) return rc;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return GEMM_ERR_CUDA;
    // An 8-byte read into the caller's stack and, if it held a fault, an
    // 8-byte clear: plain copies, nothing allocated.
    unsigned long long word = 0;
    void *rec = slot->base + kFaultOffset;
    if (cudaMemcpy(&word, rec, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (word == 0) return GEMM_OK;
    if (fault_info) *fault_info = (int64_t)(word & ~kFaultFlag);
    if (cudaMemset(rec, 0, sizeof(word)) != cudaSuccess) return GEMM_ERR_CUDA;
    return fault_status(word);
}
