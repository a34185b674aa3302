// Generic GPU paths that accept any pitch and any element alignment:
//   * gemm_simt_generic: C = act(alpha*op(A)*op(B) + bias) + beta*C with
//     fp32 or bf16 operands in either layout (op(X) = X or X^T) and an fp32
//     or bf16 C, on the CUDA cores with fp32 accumulation.  It serves BF16
//     inputs whose rows cannot be fetched by TMA (pitch not a multiple of 8
//     elements, or a base that is not 16-byte aligned) and FP32 operands in
//     transposed layouts.  The product of two bf16 values is exact in fp32,
//     so the arithmetic is the same fp32 accumulation as on the tensor
//     cores, in another order.
//   * scale_c: C = beta * C for alpha == 0 or K == 0 (C is written without
//     being read when beta == 0).
// The tiling follows the plain shared-memory scheme of "CUDA shared memory
// optimisation" (hdetylss.com), section 3.2, with bounds-checked,
// zero-filled loads at the edges as in the "Z-Turbo" tuning page
// (lanjinlin.com.cn), section 3.1.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "epilogue.cuh"
#include "internal.h"

namespace gemm {
namespace {

constexpr int GB = 64, GK = 16, GTHREADS = 256;

struct GenericParams {
    int M, N, K;
    float alpha, beta;
    const void *A;
    const void *B;
    void *C;
    long long lda, ldb, ldc;
    int trans_a, trans_b;  // A stored K x M / B stored N x K
    EpiParams epi;
    long long batch, stride_a, stride_b, stride_c;  // matrix i at X + i * stride_x
};

template <bool BF16>
__device__ __forceinline__ float load_in(const void *p, long long idx) {
    if constexpr (BF16) {
        const uint16_t bits = static_cast<const uint16_t *>(p)[idx];
        return __uint_as_float(static_cast<uint32_t>(bits) << 16);
    } else {
        return static_cast<const float *>(p)[idx];
    }
}

template <bool F32OUT>
__device__ __forceinline__ float load_c(const void *p, long long idx) {
    if constexpr (F32OUT) {
        return static_cast<const float *>(p)[idx];
    } else {
        const uint16_t bits = static_cast<const uint16_t *>(p)[idx];
        return __uint_as_float(static_cast<uint32_t>(bits) << 16);
    }
}

template <bool F32OUT>
__device__ __forceinline__ void store_c(void *p, long long idx, float v) {
    if constexpr (F32OUT) {
        static_cast<float *>(p)[idx] = v;
    } else {
        static_cast<__nv_bfloat16 *>(p)[idx] = __float2bfloat16_rn(v);
    }
}

// 64 x 64 output tile, 256 threads, 4 x 4 outputs per thread.
template <bool BF16IN, bool F32OUT>
__global__ void __launch_bounds__(GTHREADS) gemm_simt_generic_kernel(const GenericParams p,
                                                                      int num_m_blk,
                                                                      int num_n_blk) {
    __shared__ float As[GK][GB + 4];  // transposed: As[k][m]
    __shared__ float Bs[GK][GB + 4];
    int m_blk, n_blk;
    grouped_tile_coords(blockIdx.x, num_m_blk, num_n_blk, kRasterGroup, m_blk, n_blk);
    const int m0 = m_blk * GB, n0 = n_blk * GB;
    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    // Matrices blockIdx.y, blockIdx.y + gridDim.y, ... of the batch.
    for (long long bi = blockIdx.y; bi < p.batch; bi += gridDim.y) {
        const void *Ab = static_cast<const char *>(p.A) + bi * p.stride_a * (BF16IN ? 2 : 4);
        const void *Bb = static_cast<const char *>(p.B) + bi * p.stride_b * (BF16IN ? 2 : 4);
        void *Cb = static_cast<char *>(p.C) + bi * p.stride_c * (F32OUT ? 4 : 2);

        float acc[4][4] = {};
        for (int k0 = 0; k0 < p.K; k0 += GK) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int idx = tid + GTHREADS * i;  // 0..1023
                // Consecutive threads take consecutive addresses of whichever
                // index is contiguous in memory.
                {
                    const int k = p.trans_a ? idx >> 6 : idx & 15;
                    const int m = p.trans_a ? idx & 63 : idx >> 4;
                    const int gm = m0 + m, gk = k0 + k;
                    const long long off =
                        p.trans_a ? (long long)gk * p.lda + gm : (long long)gm * p.lda + gk;
                    As[k][m] = (gm < p.M && gk < p.K) ? load_in<BF16IN>(Ab, off) : 0.f;
                }
                {
                    const int n = p.trans_b ? idx >> 4 : idx & 63;
                    const int k = p.trans_b ? idx & 15 : idx >> 6;
                    const int gk = k0 + k, gn = n0 + n;
                    const long long off =
                        p.trans_b ? (long long)gn * p.ldb + gk : (long long)gk * p.ldb + gn;
                    Bs[k][n] = (gk < p.K && gn < p.N) ? load_in<BF16IN>(Bb, off) : 0.f;
                }
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < GK; ++kk) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = m0 + ty + 16 * i;
            if (row >= p.M) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = n0 + tx + 16 * j;
                if (col >= p.N) continue;
                const long long idx = (long long)row * p.ldc + col;
                const float c = (p.beta != 0.f) ? load_c<F32OUT>(Cb, idx) : 0.f;
                store_c<F32OUT>(Cb, idx, epi_finish(p.epi, p.alpha, p.beta, acc[i][j], col, c));
            }
        }
    }
}

template <bool F32OUT>
__global__ void scale_c_kernel(int M, int N, float beta, void *C, long long ldc, long long batch,
                               long long stride_c) {
    const long long total = (long long)M * N;
    for (long long bi = blockIdx.y; bi < batch; bi += gridDim.y) {
        void *Cb = static_cast<char *>(C) + bi * stride_c * (F32OUT ? 4 : 2);
        for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
             e += (long long)gridDim.x * blockDim.x) {
            const long long r = e / N, c = e - r * N;
            const long long idx = r * ldc + c;
            const float v = (beta == 0.f) ? 0.f : beta * load_c<F32OUT>(Cb, idx);
            store_c<F32OUT>(Cb, idx, v);
        }
    }
}

}  // namespace

cudaError_t launch_gemm_simt_generic(int M, int N, int K, float alpha, const void *A,
                                     int64_t lda, const void *B, int64_t ldb, float beta,
                                     void *C, int64_t ldc, bool bf16_in, bool c_f32,
                                     const GemmOpts *opts, cudaStream_t stream) {
    GenericParams p{M, N, K, alpha, beta, A, B, C, lda, ldb, ldc, 0, 0, EpiParams{}, 1, 0, 0, 0};
    if (opts) {
        p.trans_a = opts->trans_a ? 1 : 0;
        p.trans_b = opts->trans_b ? 1 : 0;
        p.epi.bias = opts->bias;
        p.epi.bias_f32 = opts->bias_f32 ? 1 : 0;
        p.epi.act = opts->act;
        p.epi.on = (opts->bias != nullptr || opts->act != 0) ? 1 : 0;
        p.batch = opts->batch;
        p.stride_a = opts->stride_a;
        p.stride_b = opts->stride_b;
        p.stride_c = opts->stride_c;
    }
    const int nm = (M + GB - 1) / GB, nn = (N + GB - 1) / GB;
    const long long tiles = (long long)nm * nn;
    if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const dim3 g((unsigned)tiles, (unsigned)(p.batch < 65535 ? p.batch : 65535), 1);
    if (bf16_in) {
        if (c_f32)
            gemm_simt_generic_kernel<true, true><<<g, GTHREADS, 0, stream>>>(p, nm, nn);
        else
            gemm_simt_generic_kernel<true, false><<<g, GTHREADS, 0, stream>>>(p, nm, nn);
    } else {
        if (c_f32)
            gemm_simt_generic_kernel<false, true><<<g, GTHREADS, 0, stream>>>(p, nm, nn);
        else
            gemm_simt_generic_kernel<false, false><<<g, GTHREADS, 0, stream>>>(p, nm, nn);
    }
    return cudaGetLastError();
}

cudaError_t launch_scale_c(int M, int N, float beta, void *C, int64_t ldc, bool c_f32,
                           int64_t batch, int64_t stride_c, cudaStream_t stream) {
    const long long total = (long long)M * N;
    long long blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    const dim3 g((unsigned)blocks, (unsigned)(batch < 65535 ? batch : 65535), 1);
    if (c_f32)
        scale_c_kernel<true><<<g, 256, 0, stream>>>(M, N, beta, C, ldc, batch, stride_c);
    else
        scale_c_kernel<false><<<g, 256, 0, stream>>>(M, N, beta, C, ldc, batch, stride_c);
    return cudaGetLastError();
}

}  // namespace gemm
