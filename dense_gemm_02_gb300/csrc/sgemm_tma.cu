// FP32 SGEMM on the CUDA cores fed by TMA: C = alpha * A * B + beta * C.
//
// Same method as sgemm_simt.cu ("CUDA hand-written SGEMM: 0.4 -> 10.23
// TFLOPS" (gtnt.cn): shared-memory tiling with a sliding K window, bank-
// conflict-free shared memory, 16-byte vector fragments, a register-blocked
// outer product, a multi-buffered load pipeline), with the load path moved
// off the compute warps, which is the largest non-FFMA cost of that kernel:
//
//   * One thread issues two TMA boxes per 32-deep K step: A (128 rows x 32,
//     K-major, 128-byte swizzle) and B (32 rows x 128 columns).  Out-of-range
//     rows, columns and K are zero-filled by the TMA, so the loop carries no
//     bounds checks.  Three 32 KiB stages, two CTAs per SM.
//   * Each stage completes on an mbarrier; every thread waits on it with a
//     time limit, and one __syncthreads_or per step both frees the previous
//     stage for the next TMA and votes on abort, so all threads leave the
//     loop together if a wait ever runs out.
//   * Warp tile 64 x 32 (8 x 4 threads), 8 x 8 outputs per thread.  A thread
//     owns rows tm + 8i, so every row it reads has the same swizzle phase
//     (row & 7 == tm): its A fragment for four K values is one LDS.128 per
//     row, the eight tm threads of a warp hit eight different bank groups,
//     and no per-load address arithmetic is needed beyond one XOR per four
//     K values.  B fragments are LDS.128 broadcasts of 64 contiguous bytes.
//   * The outer product uses the packed FP32 FMA of sm_100 (__ffma2_rn: two
//     fp32 fused multiply-adds per instruction, each exactly fmaf), with
//     accumulator pairs along N and the A value broadcast, so the FP32 pipe
//     is fed at half the instruction issue rate.  Results are bit-identical to
//     scalar fmaf in the same order.
//   * CUDA-core FP32 only (no tensor-core or TF32 instruction).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx_sm100.cuh"

namespace gemm {
namespace {

using namespace ptx;

constexpr int TBM = 128, TBN = 128, TBK = 32, TSTAGES = 3, TTHREADS = 256;
constexpr int TA_BYTES = TBM * TBK * 4;  // 16 KiB, rows of 128 bytes, swizzled
constexpr int TB_BYTES = TBK * TBN * 4;  // 16 KiB, rows of 512 bytes
constexpr int TSTAGE_BYTES = TA_BYTES + TB_BYTES;
constexpr int TOFF_BAR = TSTAGES * TSTAGE_BYTES;
constexpr int TSMEM_ALLOC = TOFF_BAR + 64 + 1024;  // barriers, then alignment slack

struct TmaParams {
    int M, N, K;
    float alpha, beta;
    float *C;
    long long ldc;
    int c_vec;
    int num_m_blk, num_n_blk;
    unsigned long long *fault_word;
    unsigned long long timeout_ns;
};

__global__ void __launch_bounds__(TTHREADS, 2)
    sgemm_tma_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const TmaParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + TOFF_BAR);
    volatile int *never = reinterpret_cast<volatile int *>(full + TSTAGES);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 2, wn = warp & 3;  // 2 x 4 warps, warp tile 64 x 32
    const int tm = lane >> 2, tn = lane & 3;  // 8 x 4 threads, thread tile 8 x 8

    int m_blk, n_blk;
    grouped_tile_coords(blockIdx.x, p.num_m_blk, p.num_n_blk, kRasterGroup, m_blk, n_blk);
    const int m0 = m_blk * TBM, n0 = n_blk * TBN;
    const int KT = (p.K + TBK - 1) / TBK;

    if (tid == 0) {
        for (int s = 0; s < TSTAGES; ++s) mbar_init(&full[s], 1);
        *never = 0;
        fence_barrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    __syncthreads();

    auto issue = [&](int kt) {
        const int s = kt % TSTAGES;
        uint8_t *st = smem + s * TSTAGE_BYTES;
        mbar_arrive_expect_tx(&full[s], TSTAGE_BYTES);
        tma_load_2d(st, &tmA, &full[s], kt * TBK, m0);
        tma_load_2d(st + TA_BYTES, &tmB, &full[s], n0, kt * TBK);
    };
    int issued = 0;
    if (tid == 0)
        for (; issued < TSTAGES - 1 && issued < KT; ++issued) issue(issued);

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    // Byte offsets of this thread's fragments inside a stage.
    const uint32_t a_row_off = (uint32_t)(wm * 64 + tm) * 128u;  // + i * 1024 for row tm + 8i
    const uint32_t b_col_off = (uint32_t)TA_BYTES + (uint32_t)(wn * 32 + tn * 4) * 4u;

    int kt = 0, s = 0;
    uint32_t ph = 0;
    bool failed = false;
#pragma unroll 1
    for (; kt < KT; ++kt) {
        const bool ok = mbar_wait(&full[s], ph, never, p.timeout_ns);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        // Every thread is past step kt-1, so its stage may be refilled.
        if (tid == 0 && issued < KT) issue(issued++);
        const uint8_t *st = smem + s * TSTAGE_BYTES;
#pragma unroll
        for (int c = 0; c < TBK / 4; ++c) {
            // 16-byte chunk c (K values 4c..4c+3) of each row, after the
            // 128-byte swizzle: chunk position c ^ (row & 7) = c ^ tm.
            const uint8_t *ap = st + a_row_off + (uint32_t)((c ^ tm) << 4);
            float4 a[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = *reinterpret_cast<const float4 *>(ap + i * 1024);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const uint8_t *bp = st + b_col_off + (uint32_t)(c * 4 + k4) * (TBN * 4);
                const float4 b0 = *reinterpret_cast<const float4 *>(bp);
                const float4 b1 = *reinterpret_cast<const float4 *>(bp + 64);
                const float2 bq[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                                      make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float av = k4 == 0 ? a[i].x : k4 == 1 ? a[i].y : k4 == 2 ? a[i].z : a[i].w;
                    const float2 apr = make_float2(av, av);
                    // Packed FP32 FMA: two IEEE fp32 fused multiply-adds per
                    // instruction (per component exactly fmaf), halving the
                    // issue slots the outer product needs.
#pragma unroll
                    for (int jp = 0; jp < 4; ++jp) {
                        const float2 r = __ffma2_rn(
                            apr, bq[jp], make_float2(acc[i][2 * jp], acc[i][2 * jp + 1]));
                        acc[i][2 * jp] = r.x;
                        acc[i][2 * jp + 1] = r.y;
                    }
                }
            }
        }
        if (++s == TSTAGES) {
            s = 0;
            ph ^= 1u;
        }
    }

    if (failed) {
        if (tid == 0) {
            atomicCAS(p.fault_word, 0ull, fault_code(kRoleSimt, (unsigned)(kt % TSTAGES),
                                                     (unsigned)blockIdx.x));
            // Let the copies still in flight land before the CTA exits.
            for (int j = kt; j < issued; ++j)
                mbar_wait(&full[j % TSTAGES], (uint32_t)((j / TSTAGES) & 1), never, p.timeout_ns,
                          true);
        }
        return;
    }

    // Epilogue: C = alpha * acc + beta * C (C unread when beta == 0); row
    // wm*64 + tm + 8i, columns wn*32 + tn*4 + {0..3} and +16.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = m0 + wm * 64 + tm + 8 * i;
        if (row >= p.M) continue;
        float *crow = p.C + (long long)row * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = n0 + wn * 32 + tn * 4 + 16 * h;
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = p.alpha * acc[i][4 * h + j];
            if (p.c_vec && col + 3 < p.N) {
                float4 *dst = reinterpret_cast<float4 *>(crow + col);
                if (p.beta != 0.f) {
                    const float4 c = *dst;
                    v[0] = fmaf(p.alpha, acc[i][4 * h + 0], p.beta * c.x);
                    v[1] = fmaf(p.alpha, acc[i][4 * h + 1], p.beta * c.y);
                    v[2] = fmaf(p.alpha, acc[i][4 * h + 2], p.beta * c.z);
                    v[3] = fmaf(p.alpha, acc[i][4 * h + 3], p.beta * c.w);
                }
                *dst = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (col + j < p.N) {
                        if (p.beta != 0.f)
                            v[j] = fmaf(p.alpha, acc[i][4 * h + j], p.beta * crow[col + j]);
                        crow[col + j] = v[j];
                    }
                }
            }
        }
    }
}

}  // namespace

int launch_sgemm_tma(DeviceState *st, int M, int N, int K, float alpha, const float *A,
                     int64_t lda, const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                     cudaStream_t stream) {
    static bool attr_done[kMaxDevices] = {};
    if (!attr_done[st->device]) {
        if (cudaFuncSetAttribute(sgemm_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TSMEM_ALLOC) != cudaSuccess)
            return GEMM_ERR_CUDA;
        attr_done[st->device] = true;
    }
    alignas(64) CUtensorMap ta, tb;
    if (!encode_tensor_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, A, (uint64_t)K, (uint64_t)M,
                              (uint64_t)lda * 4, TBK, TBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, B, (uint64_t)N, (uint64_t)K,
                              (uint64_t)ldb * 4, TBN, TBK, CU_TENSOR_MAP_SWIZZLE_NONE))
        return GEMM_ERR_CUDA;
    TmaParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.C = C;
    p.ldc = ldc;
    p.c_vec = ((reinterpret_cast<uintptr_t>(C) & 15) == 0) && (ldc % 4 == 0);
    p.num_m_blk = (M + TBM - 1) / TBM;
    p.num_n_blk = (N + TBN - 1) / TBN;
    p.fault_word = st->fault_word;
    p.timeout_ns = (unsigned long long)runtime_config().watchdog_ms * 1000000ull;
    const long long tiles = (long long)p.num_m_blk * p.num_n_blk;
    if (tiles > 0x7fffffffLL) return GEMM_ERR_TOO_LARGE;
    sgemm_tma_kernel<<<(unsigned)tiles, TTHREADS, TSMEM_ALLOC, stream>>>(ta, tb, p);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace gemm
