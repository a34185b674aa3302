// FP32 SGEMM on the CUDA cores: C = alpha * A * B + beta * C, all fp32.
//
// The method is the one of "CUDA hand-written SGEMM: 0.4 -> 10.23 TFLOPS"
// (gtnt.cn): output tiling with a sliding K window staged through shared
// memory (sections 3.1-3.2), row padding against bank conflicts (3.3),
// 16-byte vector transfers (4.1-4.2), a register-blocked outer product per
// thread (5.1-5.2) and a multi-buffered load pipeline (5.3, 7.2: cp.async).
// Re-designed for sm_103a:
//   * 128 x 128 x 16 CTA tile, 256 threads, 8 x 8 outputs per thread
//     (64 fp32 accumulators, no spills), two CTAs per SM.
//   * 4-stage cp.async ring, one __syncthreads per K step.
//   * A is transposed on its way into shared memory (4-byte cp.async, k
//     fastest for coalesced global reads) so that each thread reads its 8
//     A values as two 16-byte LDS.128; B keeps its row layout and is read
//     the same way.  The warp's 4 x 8 thread grid makes every LDS.128 a
//     broadcast of consecutive 16-byte chunks.
//   * Tails: out-of-range A/B elements are zero-filled by cp.async's
//     source-size operand; stores are predicated.  Any pitch works; B uses
//     16-byte copies only when its rows are 16-byte aligned.
//   * Pure FFMA: no tensor-core or TF32 instruction is involved.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace gemm {
namespace {

constexpr int BM = 128, BN = 128, BK = 16, STAGES = 4, THREADS = 256;
constexpr int AS_PITCH = BM + 4;  // floats per k-row of transposed A (16-byte aligned rows)
constexpr int BS_PITCH = BN;      // floats per k-row of B
constexpr int AS_STAGE = BK * AS_PITCH;
constexpr int BS_STAGE = BK * BS_PITCH;
constexpr int SMEM_BYTES = STAGES * (AS_STAGE + BS_STAGE) * 4;

struct SimtParams {
    int M, N, K;
    float alpha, beta;
    const float *A;
    const float *B;
    float *C;
    long long lda, ldb, ldc;
    int c_vec;  // C rows 16-byte aligned
    int num_m_blk, num_n_blk;
};

__device__ __forceinline__ void cp_async_4(float *dst, const float *src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_16(float *dst, const float *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Issues the copies of K-step kt into stage buffers As/Bs.
template <bool VEC_B>
__device__ __forceinline__ void load_stage(const SimtParams &p, float *As, float *Bs, int m0,
                                           int n0, int kt, int tid) {
    const int k0 = kt * BK;
    // A: 128 x 16 elements, k fastest across threads; stored transposed.
    {
        const int k = tid & 15;
        const int gk = k0 + k;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int m = (tid >> 4) + 16 * i;
            const int gm = m0 + m;
            const bool ok = gm < p.M && gk < p.K;
            const float *src = ok ? p.A + (long long)gm * p.lda + gk : p.A;
            cp_async_4(As + k * AS_PITCH + m, src, ok ? 4 : 0);
        }
    }
    if constexpr (VEC_B) {
        // B: 16 rows x 32 float4; partial float4s at the N edge copy only
        // their in-range bytes and zero-fill the rest.
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int k = (tid >> 5) + 8 * i;
            const int n4 = (tid & 31) * 4;
            const int gk = k0 + k, gn = n0 + n4;
            int bytes = 0;
            if (gk < p.K && gn < p.N) bytes = min(16, (p.N - gn) * 4);
            const float *src = bytes ? p.B + (long long)gk * p.ldb + gn : p.B;
            cp_async_16(Bs + k * BS_PITCH + n4, src, bytes);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = tid + THREADS * i;
            const int k = idx >> 7, n = idx & 127;
            const int gk = k0 + k, gn = n0 + n;
            const bool ok = gk < p.K && gn < p.N;
            const float *src = ok ? p.B + (long long)gk * p.ldb + gn : p.B;
            cp_async_4(Bs + k * BS_PITCH + n, src, ok ? 4 : 0);
        }
    }
}

template <bool VEC_B>
__global__ void __launch_bounds__(THREADS, 2) sgemm_simt_kernel(const SimtParams p) {
    extern __shared__ __align__(16) float smem[];
    float *As = smem;
    float *Bs = smem + STAGES * AS_STAGE;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 1, wn = warp & 1;  // 4 x 2 warps, warp tile 32 x 64
    const int tm = lane >> 3, tn = lane & 7;  // 4 x 8 threads, thread tile 8 x 8
    const int a_off = wm * 32 + tm * 4;       // rows a_off..+3 and a_off+16..+19
    const int b_off = wn * 64 + tn * 4;       // cols b_off..+3 and b_off+32..+35

    int m_blk, n_blk;
    grouped_tile_coords(blockIdx.x, p.num_m_blk, p.num_n_blk, kRasterGroup, m_blk, n_blk);
    const int m0 = m_blk * BM;
    const int n0 = n_blk * BN;
    const int KT = (p.K + BK - 1) / BK;

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < KT) load_stage<VEC_B>(p, As + s * AS_STAGE, Bs + s * BS_STAGE, m0, n0, s, tid);
        cp_async_commit();
    }

#pragma unroll 1
    for (int kt = 0; kt < KT; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        {
            const int nk = kt + STAGES - 1;
            if (nk < KT) {
                const int s = nk % STAGES;
                load_stage<VEC_B>(p, As + s * AS_STAGE, Bs + s * BS_STAGE, m0, n0, nk, tid);
            }
            cp_async_commit();
        }
        const int s = kt % STAGES;
        const float *as = As + s * AS_STAGE + a_off;
        const float *bs = Bs + s * BS_STAGE + b_off;
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4 *>(as + kk * AS_PITCH);
            const float4 a1 = *reinterpret_cast<const float4 *>(as + kk * AS_PITCH + 16);
            const float4 b0 = *reinterpret_cast<const float4 *>(bs + kk * BS_PITCH);
            const float4 b1 = *reinterpret_cast<const float4 *>(bs + kk * BS_PITCH + 32);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    cp_async_wait<0>();

    // Epilogue: C = alpha * acc + beta * C (C unread when beta == 0).
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = m0 + a_off + (i < 4 ? i : 12 + i);
        if (row >= p.M) continue;
        float *crow = p.C + (long long)row * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = n0 + b_off + 32 * h;
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

template <bool VEC_B>
cudaError_t launch_impl(const SimtParams &p, cudaStream_t stream) {
    // The shared-memory opt-in is a per-device function attribute.
    static PerDeviceOnce attrs;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (attrs.run(dev, [&e] {
            e = cudaFuncSetAttribute(sgemm_simt_kernel<VEC_B>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
            return e == cudaSuccess ? 0 : 1;
        }) != 0)
        return e;
    const long long tiles = (long long)p.num_m_blk * p.num_n_blk;
    if (tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    sgemm_simt_kernel<VEC_B><<<(unsigned)tiles, THREADS, SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sgemm_simt(int M, int N, int K, float alpha, const float *A, int64_t lda,
                              const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                              cudaStream_t stream) {
    SimtParams p;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.A = A;
    p.B = B;
    p.C = C;
    p.lda = lda;
    p.ldb = ldb;
    p.ldc = ldc;
    p.c_vec = ((reinterpret_cast<uintptr_t>(C) & 15) == 0) && (ldc % 4 == 0);
    p.num_m_blk = (M + BM - 1) / BM;
    p.num_n_blk = (N + BN - 1) / BN;
    const bool vec_b = ((reinterpret_cast<uintptr_t>(B) & 15) == 0) && (ldb % 4 == 0);
    return vec_b ? launch_impl<true>(p, stream) : launch_impl<false>(p, stream);
}

}  // namespace gemm
