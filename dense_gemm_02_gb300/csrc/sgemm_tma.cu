// FP32 SGEMM on the CUDA cores fed by TMA: C = alpha * A * B + beta * C, with
// the optional fused bias / activation epilogue of epilogue.cuh.
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

#include "epilogue.cuh"
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
    int fault_inject;  // test hook: block 0 never fills its first stage
    EpiParams epi;     // bias / activation of the fused epilogue
    // Partial-wave K split: blocks past tiles_main take one K slice
    // (kt_per_split 32-deep steps) of a tile split `splits` ways.
    int tiles_main, splits, kt_per_split;
    // Strided batch: tile t of the launch is tile t % tiles_per_batch of
    // matrix t / tiles_per_batch; a_bmul / b_bmul are 0 for a matrix shared
    // by the whole batch; C matrix i starts c_bstride elements after C.
    int tiles_per_batch, a_bmul, b_bmul;
    long long c_bstride;
    float *ws;           // fp32 partial tiles of the split tiles
    unsigned *counters;  // one per split tile
    int ws_tiles;        // split tiles the workspace covers (checked in the debug build)
};

// The work of one CTA: output tile (m_blk, n_blk) of matrix bidx of the
// batch, whole (slice < 0) or one K slice of split tile `tile`.  The plain
// and the grouped kernels both run it (force-inlined, so each compiles to
// its own straight-line kernel).
__device__ __forceinline__ void sgemm_cta(const CUtensorMap *tmA, const CUtensorMap *tmB,
                                          const TmaParams &p, int tile, int slice, int m_blk,
                                          int n_blk, int bidx) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + TOFF_BAR);
    volatile int *never = reinterpret_cast<volatile int *>(full + TSTAGES);
    volatile int *last_slice = never + 1;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 2, wn = warp & 3;  // 2 x 4 warps, warp tile 64 x 32
    const int tm = lane >> 2, tn = lane & 3;  // 8 x 4 threads, thread tile 8 x 8
    const int m0 = m_blk * TBM, n0 = n_blk * TBN;
    const int ab = bidx * p.a_bmul, bb = bidx * p.b_bmul;  // TMA batch coordinates
    const int KT_all = (p.K + TBK - 1) / TBK;
    const int kt0 = slice < 0 ? 0 : slice * p.kt_per_split;
    const int KT = slice < 0 ? KT_all : min(p.kt_per_split, KT_all - kt0);  // >= 1

    if (tid == 0) {
        for (int s = 0; s < TSTAGES; ++s) mbar_init(&full[s], 1);
        *never = 0;
        fence_barrier_init();
        prefetch_tensormap(tmA);
        prefetch_tensormap(tmB);
    }
    __syncthreads();

    auto issue = [&](int kt) {
        const int s = kt % TSTAGES;
        uint8_t *st = smem + s * TSTAGE_BYTES;
        mbar_arrive_expect_tx(&full[s], TSTAGE_BYTES);
        // Debug build: x coordinates a multiple of 4 fp32 elements (16 bytes).
        if (debug_check(p.fault_word, ((kt0 + kt) * TBK) % 4 == 0, kSiteLoadA, (unsigned)tile))
            tma_load_3d(st, tmA, &full[s], (kt0 + kt) * TBK, m0, ab);
        if (debug_check(p.fault_word, n0 % 4 == 0, kSiteLoadB, (unsigned)tile))
            tma_load_3d(st + TA_BYTES, tmB, &full[s], n0, (kt0 + kt) * TBK, bb);
    };
    int issued = 0;
    if (tid == 0)
        for (; issued < TSTAGES - 1 && issued < KT; ++issued)
            if (!(p.fault_inject && blockIdx.x == 0 && issued == 0)) issue(issued);

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
        // Plain polling here: all 256 threads wait on the stage, and a
        // suspend hint measured 1% slower for this kernel.
        const bool ok = mbar_wait(&full[s], ph, never, p.timeout_ns, false, 0);
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
                if (!(p.fault_inject && blockIdx.x == 0 && j == 0))
                    mbar_wait(&full[j % TSTAGES], (uint32_t)((j / TSTAGES) & 1), never,
                              p.timeout_ns, true);
        }
        return;
    }

    if (slice >= 0) {
        // Split tile: store this slice's partial sums (thread-major float4
        // columns, coalesced), count the slice in, and let the last slice to
        // arrive add all slices in the fixed order 0..splits-1, so the result
        // does not depend on which slice finishes last.
        const size_t split_tile = (size_t)(tile - p.tiles_main);
        if (!debug_check(p.fault_word, split_tile < (size_t)p.ws_tiles && slice < p.splits,
                         kSiteWorkspace, (unsigned)tile))
            return;
        float4 *base = reinterpret_cast<float4 *>(p.ws) + split_tile * p.splits * (16 * TTHREADS);
        float4 *mine = base + (size_t)slice * (16 * TTHREADS);
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                __stcg(mine + (2 * i + h) * TTHREADS + tid,
                       make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2],
                                   acc[i][4 * h + 3]));
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const unsigned old = atomicAdd(&p.counters[split_tile], 1u);
            *last_slice = (old == (unsigned)(p.splits - 1)) ? 1 : 0;
        }
        __syncthreads();
        if (!*last_slice) return;
        __threadfence();
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float4 v = __ldcg(base + (2 * i + h) * TTHREADS + tid);
#pragma unroll 1
                for (int sl = 1; sl < p.splits; ++sl) {
                    const float4 w = __ldcg(base + ((size_t)sl * 16 + 2 * i + h) * TTHREADS + tid);
                    v.x += w.x;
                    v.y += w.y;
                    v.z += w.z;
                    v.w += w.w;
                }
                acc[i][4 * h] = v.x;
                acc[i][4 * h + 1] = v.y;
                acc[i][4 * h + 2] = v.z;
                acc[i][4 * h + 3] = v.w;
            }
        if (tid == 0) p.counters[split_tile] = 0u;  // ready for the next launch
    }

    // Epilogue: C = act(alpha * acc + bias) + beta * C (C unread when
    // beta == 0; without bias and activation fmaf(alpha, acc, beta * C));
    // row wm*64 + tm + 8i, columns wn*32 + tn*4 + {0..3} and +16.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = m0 + wm * 64 + tm + 8 * i;
        if (row >= p.M) continue;
        float *crow = p.C + bidx * p.c_bstride + (long long)row * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int col = n0 + wn * 32 + tn * 4 + 16 * h;
            if (col >= p.N) continue;
            const bool vec = p.c_vec && col + 3 < p.N;
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            if (p.beta != 0.f) {
                if (vec) {
                    const float4 cv = *reinterpret_cast<const float4 *>(crow + col);
                    c[0] = cv.x, c[1] = cv.y, c[2] = cv.z, c[3] = cv.w;
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (col + j < p.N) c[j] = crow[col + j];
                }
            }
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                v[j] = epi_finish(p.epi, p.alpha, p.beta, acc[i][4 * h + j],
                                  col + j < p.N ? col + j : p.N - 1, c[j]);
            if (vec) {
                *reinterpret_cast<float4 *>(crow + col) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (col + j < p.N) crow[col + j] = v[j];
            }
        }
    }
}

__global__ void __launch_bounds__(TTHREADS, 2)
    sgemm_tma_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const TmaParams p) {
    // Blocks 0..tiles_main-1 compute whole tiles; each later block one K
    // slice of a tile of the partial last wave.
    int tile = blockIdx.x, slice = -1;
    if (tile >= p.tiles_main) {
        const int v = tile - p.tiles_main;
        tile = p.tiles_main + v / p.splits;
        slice = v - (v / p.splits) * p.splits;
    }
    const int bidx = tile / p.tiles_per_batch;
    int m_blk, n_blk;
    grouped_tile_coords(tile - bidx * p.tiles_per_batch, p.num_m_blk, p.num_n_blk, kRasterGroup,
                        m_blk, n_blk);
    sgemm_cta(&tmA, &tmB, p, tile, slice, m_blk, n_blk, bidx);
}

// Grouped GEMM: problem g owns launch tiles tile0[g] .. tile0[g+1] - 1; its
// A and B tensor maps and its whole parameter block travel in the kernel
// parameters (read from there where they are used, not held in registers).
struct SgGroupedParams {
    CUtensorMap ma[kMaxGroupsPerLaunch];
    CUtensorMap mb[kMaxGroupsPerLaunch];
    TmaParams tp[kMaxGroupsPerLaunch];
    int tile0[kMaxGroupsPerLaunch];
    int groups;
};

__global__ void __launch_bounds__(TTHREADS, 2)
    sgemm_tma_grouped_kernel(const __grid_constant__ SgGroupedParams gp) {
    // The problem of this block: the last one whose first tile is <= it
    // (every problem has at least one tile, so tile0 increases strictly).
    int g = 0;
    for (int i = 1; i < gp.groups; ++i)
        if (gp.tile0[i] <= (int)blockIdx.x) g = i;
    const TmaParams &q = gp.tp[g];
    const int t = (int)blockIdx.x - gp.tile0[g];
    int m_blk, n_blk;
    grouped_tile_coords(t, q.num_m_blk, q.num_n_blk, kRasterGroup, m_blk, n_blk);
    sgemm_cta(&gp.ma[g], &gp.mb[g], q, t, -1, m_blk, n_blk, 0);
}

}  // namespace

int launch_sgemm_tma_grouped(DeviceState *st, int count, const GroupProblem *g,
                             cudaStream_t stream) {
    static PerDeviceOnce attrs;
    if (attrs.run(st->device, [] {
            return cudaFuncSetAttribute(sgemm_tma_grouped_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        TSMEM_ALLOC) == cudaSuccess
                       ? 0
                       : 1;
        }) != 0)
        return GEMM_ERR_CUDA;
    if (count < 1 || count > kMaxGroupsPerLaunch) return GEMM_ERR_INVALID_ARG;
    static_assert(sizeof(SgGroupedParams) <= 32000, "kernel parameter space");
    // The parameter block is large; it lives on the heap of this thread.
    thread_local SgGroupedParams gp;
    long long tiles = 0;
    for (int i = 0; i < count; ++i) {
        const GroupProblem &x = g[i];
        if (!encode_tensor_map_3d(&gp.ma[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, x.A, (uint64_t)x.K,
                                  (uint64_t)x.M, 1, (uint64_t)x.lda * 4, 0, TBK, TBM,
                                  CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tensor_map_3d(&gp.mb[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, x.B, (uint64_t)x.N,
                                  (uint64_t)x.K, 1, (uint64_t)x.ldb * 4, 0, TBN, TBK,
                                  CU_TENSOR_MAP_SWIZZLE_NONE))
            return GEMM_ERR_CUDA;
        TmaParams &q = gp.tp[i];
        q = TmaParams{};
        q.M = (int)x.M;
        q.N = (int)x.N;
        q.K = (int)x.K;
        q.alpha = x.alpha;
        q.beta = x.beta;
        q.C = static_cast<float *>(x.C);
        q.ldc = x.ldc;
        q.c_vec = ((reinterpret_cast<uintptr_t>(x.C) & 15) == 0) && (x.ldc % 4 == 0);
        q.num_m_blk = (q.M + TBM - 1) / TBM;
        q.num_n_blk = (q.N + TBN - 1) / TBN;
        q.tiles_main = 0x7fffffff;  // whole tiles only
        q.splits = 1;
        q.tiles_per_batch = 0x7fffffff;
        gp.tile0[i] = (int)tiles;
        tiles += (long long)q.num_m_blk * q.num_n_blk;
        if (tiles > 0x7fffffffLL) return GEMM_ERR_TOO_LARGE;
    }
    gp.groups = count;
    const RuntimeConfig cfg = runtime_config();
    const int inject = cfg.fault_inject ? 1 : 0;
    if (inject) consume_fault_inject();
    for (int i = 0; i < count; ++i) {
        gp.tp[i].fault_word = st->fault_word;
        gp.tp[i].timeout_ns = (unsigned long long)cfg.watchdog_ms * 1000000ull;
        gp.tp[i].fault_inject = inject;
    }
    sgemm_tma_grouped_kernel<<<(unsigned)tiles, TTHREADS, TSMEM_ALLOC, stream>>>(gp);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

int launch_sgemm_tma(DeviceState *st, int M, int N, int K, float alpha, const float *A,
                     int64_t lda, const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                     const GemmOpts *opts, cudaStream_t stream) {
    static PerDeviceOnce attrs;
    if (attrs.run(st->device, [] {
            return cudaFuncSetAttribute(sgemm_tma_kernel,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        TSMEM_ALLOC) == cudaSuccess
                       ? 0
                       : 1;
        }) != 0)
        return GEMM_ERR_CUDA;
    const GemmOpts o = opts ? *opts : GemmOpts{};
    const int64_t batch = o.batch > 1 ? o.batch : 1;
    alignas(64) CUtensorMap ta, tb;
    if (!encode_tensor_map_3d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, A, (uint64_t)K, (uint64_t)M,
                              o.stride_a ? (uint64_t)batch : 1, (uint64_t)lda * 4,
                              (uint64_t)o.stride_a * 4, TBK, TBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tensor_map_3d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, B, (uint64_t)N, (uint64_t)K,
                              o.stride_b ? (uint64_t)batch : 1, (uint64_t)ldb * 4,
                              (uint64_t)o.stride_b * 4, TBN, TBK, CU_TENSOR_MAP_SWIZZLE_NONE))
        return GEMM_ERR_CUDA;
    TmaParams p{};
    p.epi.bias = o.bias;
    p.epi.bias_f32 = o.bias_f32 ? 1 : 0;
    p.epi.act = o.act;
    p.epi.on = (o.bias != nullptr || o.act != 0) ? 1 : 0;
    p.a_bmul = o.stride_a && batch > 1 ? 1 : 0;
    p.b_bmul = o.stride_b && batch > 1 ? 1 : 0;
    p.c_bstride = batch > 1 ? o.stride_c : 0;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.C = C;
    p.ldc = ldc;
    p.c_vec = ((reinterpret_cast<uintptr_t>(C) & 15) == 0) && (ldc % 4 == 0) &&
              (p.c_bstride % 4 == 0);
    p.num_m_blk = (M + TBM - 1) / TBM;
    p.num_n_blk = (N + TBN - 1) / TBN;
    p.fault_word = st->fault_word;
    p.timeout_ns = (unsigned long long)runtime_config().watchdog_ms * 1000000ull;
    p.fault_inject = runtime_config().fault_inject ? 1 : 0;
    if (p.fault_inject) consume_fault_inject();
    const long long tiles_per_batch = (long long)p.num_m_blk * p.num_n_blk;
    const long long tiles = tiles_per_batch * batch;
    if (tiles > 0x7fffffffLL) return GEMM_ERR_TOO_LARGE;
    p.tiles_per_batch = (int)tiles_per_batch;

    // Partial last wave.  The kernel is bound by the FP32 pipe, so an SM
    // finishes its tiles at about the same rate whether one or two CTAs
    // share it: what counts is the work per SM.  After the first
    // tiles - rem tiles (rem = tiles mod SMs) every SM has had the same
    // share; the last rem tiles would put one more whole tile on rem SMs
    // while the others idle.  Each of them is split along K into S slices
    // (at least four 32-deep K steps each, S <= 8) with S chosen to minimise
    // the busiest SM's extra work, ceil(rem * S / SMs) / S of a tile; the
    // slices meet in a workspace.  (4096^3 on 152 SMs: rem 112, S = 4, 0.75
    // of a tile instead of 1.)
    p.tiles_main = (int)tiles;
    p.splits = 1;
    p.kt_per_split = 0;
    p.ws = nullptr;
    p.counters = nullptr;
    p.ws_tiles = 0;
    const int KT = (K + TBK - 1) / TBK;
    const long long sms = st->sm_count;
    if (!runtime_config().tail_split_off && sms > 0) {
        const long long rem = tiles % sms;
        int best = 1;
        double best_t = rem ? 1.0 : 0.0;
        for (int S = 2; S <= 8 && S <= KT / 4 && rem; ++S) {
            const double t = (double)((rem * S + sms - 1) / sms) / S;
            if (t < best_t - 0.02) {
                best_t = t;
                best = S;
            }
        }
        if (best >= 2) {
            const int per = (KT + best - 1) / best;
            const int splits = (KT + per - 1) / per;  // no empty slice
            if (splits >= 2) {
                p.tiles_main = (int)(tiles - rem);
                p.splits = splits;
                p.kt_per_split = per;
            }
        }
    }
    const long long split_tiles = tiles - p.tiles_main;
    const long long units = p.tiles_main + split_tiles * p.splits;
    if (units > 0x7fffffffLL) return GEMM_ERR_TOO_LARGE;
    if (split_tiles > 0) {
        Workspace *w = nullptr;
        const size_t ws_bytes = (size_t)split_tiles * p.splits * TBM * TBN * sizeof(float);
        const int rc = stream_workspace(st, stream, ws_bytes, (size_t)split_tiles, &w);
        if (rc != GEMM_OK) return rc;
        p.ws = w->ws;
        p.counters = w->counters;
        p.ws_tiles = (int)split_tiles;
    }
    sgemm_tma_kernel<<<(unsigned)units, TTHREADS, TSMEM_ALLOC, stream>>>(ta, tb, p);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace gemm
