// BF16 GEMM with FP32 accumulation on the Blackwell tcgen05 tensor cores:
// C = alpha * A * B + beta * C, A (M x K) and B (K x N) row-major bf16,
// C bf16 or fp32.
//
// What the pages fix ("Blackwell BF16 GEMM ..." (lshu.cn)): BF16 operands
// with an FP32 accumulator converted back once at the end (sections 1.2,
// 6.3); a TMA-fed, mbarrier-synchronised asynchronous pipeline that keeps the
// tensor cores busy while the next tiles load (2.2-2.3); tiles of 128 rows
// with a K step of 64 (4.1-4.2); tails handled by predication (4.3, 6.2);
// split-K to bring more SMs to bear on small-M shapes ("CUDA hand-written
// SGEMM ..." (gtnt.cn) section 7.2, and the small-M discussion of the BF16
// page, section 5.2).  The design below is this library's own:
//
//   * Persistent CTAs (one per SM), each walking output tiles
//     (128 x BN, BN = 256 or 128) in grouped raster order.
//   * Warp roles: warp 0 lane 0 issues TMA loads into an S-stage shared
//     memory ring (A: one 64 x 128 box, K-major, 128-byte swizzle; B: BN/64
//     boxes of 64 x 64, N-major, 128-byte swizzle); warp 1 allocates tensor
//     memory and its lane 0 issues tcgen05.mma (M = 128, N = BN, K = 16)
//     into one of two TMEM accumulators; warps 2-5 drain the other
//     accumulator with tcgen05.ld, apply alpha/beta in fp32, convert and
//     store, so a tile's epilogue overlaps the next tile's main loop.
//   * Out-of-range rows/columns/K are zero-filled by TMA and masked at the
//     store.
//   * Split-K (small M x N): each (tile, K-slice) unit writes an fp32
//     partial tile to a workspace; the last unit of a tile to finish (an
//     atomic counter) sums the slices in slice order 0..S-1, so results are
//     bit-reproducible, then applies alpha/beta and stores.
//   * Every wait is bounded (see ptx_sm100.cuh); a wait that runs out records
//     a fault word, raises a CTA abort flag, lets in-flight copies and MMAs
//     finish, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx_sm100.cuh"

namespace gemm {
namespace {

using namespace ptx;

constexpr int TC_BM = 128;
constexpr int TC_BK = 64;            // bf16 elements in one 128-byte swizzle row
constexpr int TC_UMMA_K = 16;        // K of one kind::f16 MMA
constexpr int TC_THREADS = 192;      // 6 warps
constexpr int TC_EPI_THREADS = 128;  // warps 2-5
constexpr int TC_EPI_BAR = 1;        // named barrier id of the epilogue warps

template <int BN>
struct TcCfg {
    static constexpr int STAGES = (BN == 256) ? 4 : 6;
    static constexpr int A_BYTES = TC_BM * TC_BK * 2;  // 16 KiB
    static constexpr int B_BYTES = BN * TC_BK * 2;     // 32 KiB at BN = 256
    static constexpr int B_BOX_BYTES = 64 * TC_BK * 2; // one 64-column B box, 8 KiB
    static constexpr int STAGE_TX = A_BYTES + B_BYTES;
    static constexpr int B_BOXES = BN / 64;
    static constexpr int OFF_B = STAGES * A_BYTES;
    static constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 5;  // full, empty, tfull[2], tempty[2], drain
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;  // slack for 1024-byte alignment
    static constexpr int TMEM_COLS = 2 * BN;             // two fp32 accumulators
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
    static_assert(TMEM_COLS <= 512, "tensor memory budget");
};

struct TcParams {
    int M, N, K;
    int num_m_blk, num_n_blk, num_kb;
    int splits, kb_per_split;
    int num_units;
    float alpha, beta;
    void *C;
    long long ldc;
    int c_f32;
    int c_vec;
    float *ws;
    unsigned *counters;
    unsigned long long *fault_word;
    unsigned long long timeout_ns;
    int fault_inject;
};

// Shared-memory matrix descriptor of tcgen05 (PTX ISA, "matrix descriptor"):
// start address >> 4 in bits 0-13, leading-dimension byte offset >> 4 in
// 16-29, stride-dimension byte offset >> 4 in 32-45, the fixed value 1 in
// bits 46-48, base offset 0, swizzle mode in bits 61-63 (2 = 128-byte).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) |
           ((uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A bf16 (7-9 = 1), B bf16 (10-12 = 1), A K-major (bit 15 = 0), B MN-major
// (bit 16 = 1, B is row-major K x N), N >> 3 in bits 17-22, M >> 4 in 24-28.
template <int BN>
__host__ __device__ constexpr uint32_t idesc_bf16_f32() {
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(BN >> 3) << 17) |
           ((uint32_t)(TC_BM >> 4) << 24);
}

__device__ __forceinline__ void decode_unit(const TcParams &p, int u, int &tile, int &m_blk,
                                            int &n_blk, int &kb0, int &kb1) {
    tile = u / p.splits;
    const int split = u - tile * p.splits;
    grouped_tile_coords(tile, p.num_m_blk, p.num_n_blk, m_blk, n_blk);
    kb0 = split * p.kb_per_split;
    kb1 = min(kb0 + p.kb_per_split, p.num_kb);
}

__device__ __forceinline__ void record_fault(const TcParams &p, volatile int *abort_flag,
                                             unsigned role, unsigned stage, unsigned tile) {
    *abort_flag = 1;
    atomicCAS(p.fault_word, 0ull, fault_code(role, stage, tile));
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

// Stores 32 consecutive outputs of row gm starting at column gn:
// C = alpha * acc + beta * C, converted to C's type.
__device__ __forceinline__ void store_row_chunk(const TcParams &p, int gm, int gn,
                                                const float (&acc)[32]) {
    if (gm >= p.M) return;
    const float alpha = p.alpha, beta = p.beta;
    if (p.c_f32) {
        float *crow = static_cast<float *>(p.C) + (long long)gm * p.ldc;
        if (p.c_vec && gn + 32 <= p.N) {
            float4 *dst = reinterpret_cast<float4 *>(crow + gn);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float4 o = make_float4(alpha * acc[4 * j], alpha * acc[4 * j + 1],
                                       alpha * acc[4 * j + 2], alpha * acc[4 * j + 3]);
                if (beta != 0.f) {
                    const float4 c = dst[j];
                    o.x = fmaf(alpha, acc[4 * j], beta * c.x);
                    o.y = fmaf(alpha, acc[4 * j + 1], beta * c.y);
                    o.z = fmaf(alpha, acc[4 * j + 2], beta * c.z);
                    o.w = fmaf(alpha, acc[4 * j + 3], beta * c.w);
                }
                dst[j] = o;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (gn + j < p.N) {
                    float o = alpha * acc[j];
                    if (beta != 0.f) o = fmaf(alpha, acc[j], beta * crow[gn + j]);
                    crow[gn + j] = o;
                }
            }
        }
    } else {
        uint16_t *crow = static_cast<uint16_t *>(p.C) + (long long)gm * p.ldc;
        if (p.c_vec && gn + 32 <= p.N) {
            uint4 *dst = reinterpret_cast<uint4 *>(crow + gn);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = alpha * acc[8 * j + e];
                if (beta != 0.f) {
                    const uint4 c = dst[j];
                    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const uint32_t h = (e & 1) ? (cw[e >> 1] >> 16) : (cw[e >> 1] & 0xFFFFu);
                        o[e] = fmaf(alpha, acc[8 * j + e], beta * bf16_bits_to_float(h));
                    }
                }
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    __nv_bfloat162 pr = __floats2bfloat162_rn(o[2 * e], o[2 * e + 1]);
                    w[e] = *reinterpret_cast<uint32_t *>(&pr);
                }
                dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (gn + j < p.N) {
                    float o = alpha * acc[j];
                    if (beta != 0.f) o = fmaf(alpha, acc[j], beta * bf16_bits_to_float(crow[gn + j]));
                    __nv_bfloat16 h = __float2bfloat16_rn(o);
                    crow[gn + j] = *reinterpret_cast<uint16_t *>(&h);
                }
            }
        }
    }
}

template <int BN>
__global__ void __launch_bounds__(TC_THREADS, 1)
    bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const TcParams p) {
    using Cfg = TcCfg<BN>;
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzled tiles need 1024-byte aligned shared addresses.
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + Cfg::OFF_B;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
    uint64_t *full = bars;
    uint64_t *empty = bars + S;
    uint64_t *tfull = bars + 2 * S;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
    uint32_t *tmem_slot = misc;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    volatile int *last_flag = reinterpret_cast<volatile int *>(misc + 2);
    volatile int *epi_ok = reinterpret_cast<volatile int *>(misc + 3);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], TC_EPI_THREADS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *last_flag = 0;
        *epi_ok = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            int withheld = -1;
            bool ok = true;
            for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x) {
                int tile, mb, nb, kb0, kb1;
                decode_unit(p, u, tile, mb, nb, kb0, kb1);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1u;
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.timeout_ns)) {
                        record_fault(p, abort_flag, kRoleProducer, s, tile);
                        ok = false;
                        break;
                    }
                    if (p.fault_inject && blockIdx.x == 0 && it == 0) {
                        withheld = 0;  // test hook: this stage is never filled
                        continue;
                    }
                    mbar_arrive_expect_tx(&full[s], Cfg::STAGE_TX);
                    tma_load_2d(sA + s * Cfg::A_BYTES, &tmA, &full[s], kb * TC_BK, mb * TC_BM);
#pragma unroll
                    for (int j = 0; j < Cfg::B_BOXES; ++j)
                        tma_load_2d(sB + s * Cfg::B_BYTES + j * Cfg::B_BOX_BYTES, &tmB, &full[s],
                                    nb * BN + j * 64, kb * TC_BK);
                }
            }
            // Let every copy started here land before the CTA can exit.
            const uint32_t first = it > (uint32_t)S ? it - S : 0u;
            for (uint32_t i = first; i < it; ++i) {
                if ((int)i == withheld) continue;
                mbar_wait(&full[i % S], (i / S) & 1u, abort_flag, p.timeout_ns, true);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_bf16_f32<BN>();
            const uint32_t a_base = smem_addr(sA), b_base = smem_addr(sB);
            uint32_t it = 0, local = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < p.num_units && ok; u += gridDim.x, ++local) {
                int tile, mb, nb, kb0, kb1;
                decode_unit(p, u, tile, mb, nb, kb0, kb1);
                const uint32_t b = local & 1u, use = local >> 1;
                if (!mbar_wait(&tempty[b], (use & 1u) ^ 1u, abort_flag, p.timeout_ns)) {
                    record_fault(p, abort_flag, kRoleMma, 0xfe, tile);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * BN;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % S;
                    const uint32_t ph = (it / S) & 1u;
                    if (!mbar_wait(&full[s], ph, abort_flag, p.timeout_ns)) {
                        record_fault(p, abort_flag, kRoleMma, s, tile);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = a_base + s * Cfg::A_BYTES;
                    const uint32_t sb = b_base + s * Cfg::B_BYTES;
#pragma unroll
                    for (int k = 0; k < TC_BK / TC_UMMA_K; ++k) {
                        // A: K-major rows of 128 bytes, 8-row groups 1024 bytes
                        // apart; a K step of 16 moves 32 bytes along the row.
                        const uint64_t ad = smem_desc_sw128(sa + k * 32, 16, 1024);
                        // B: N-major; 64-column boxes Cfg::B_BOX_BYTES apart,
                        // 8 K-rows 1024 bytes apart; a K step of 16 is 16 rows.
                        const uint64_t bd =
                            smem_desc_sw128(sb + k * 16 * 128, Cfg::B_BOX_BYTES, 1024);
                        umma_f16(d_tmem, ad, bd, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
                    }
                    umma_commit(&empty[s]);  // frees the stage once these MMAs finish
                }
                if (!ok) break;
                umma_commit(&tfull[b]);  // accumulator b is complete
            }
            // All MMAs issued here must finish before TMEM is released.
            umma_commit(drain);
            mbar_wait(drain, 0, abort_flag, p.timeout_ns, true);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue warps 2-5
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        const int et = threadIdx.x - 64;
        uint32_t local = 0;
        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++local) {
            int tile, mb, nb, kb0, kb1;
            decode_unit(p, u, tile, mb, nb, kb0, kb1);
            const uint32_t b = local & 1u, use = local >> 1;
            // One thread waits (bounded) and the decision is shared, so the
            // epilogue warps always leave the loop together.
            if (et == 0) {
                const bool ok = mbar_wait(&tfull[b], use & 1u, abort_flag, p.timeout_ns);
                if (!ok) record_fault(p, abort_flag, kRoleEpilogue, 0xff, tile);
                *epi_ok = ok ? 1 : 0;
            }
            named_bar_sync(TC_EPI_BAR, TC_EPI_THREADS);
            if (!*epi_ok) break;
            mbar_wait(&tfull[b], use & 1u, abort_flag, p.timeout_ns, true);  // completed: no wait
            tc_fence_after_sync();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + b * BN;
            const int gm = mb * TC_BM + row;
            const int gn0 = nb * BN;
            if (p.splits == 1) {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, r);
                    tmem_ld_wait();
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    store_row_chunk(p, gm, gn0 + c * 32, v);
                }
                tc_fence_before_sync();
                mbar_arrive(&tempty[b]);
            } else {
                const int split = u - tile * p.splits;
                float *wrow = p.ws + (((size_t)tile * p.splits + split) * TC_BM + row) * BN;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, r);
                    tmem_ld_wait();
                    if (gm < p.M) {
                        float4 *dst = reinterpret_cast<float4 *>(wrow + c * 32);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            __stcg(dst + j, make_float4(__uint_as_float(r[4 * j]),
                                                        __uint_as_float(r[4 * j + 1]),
                                                        __uint_as_float(r[4 * j + 2]),
                                                        __uint_as_float(r[4 * j + 3])));
                    }
                }
                tc_fence_before_sync();
                mbar_arrive(&tempty[b]);
                __threadfence();
                named_bar_sync(TC_EPI_BAR, TC_EPI_THREADS);
                if (et == 0) {
                    const unsigned old = atomicAdd(&p.counters[tile], 1u);
                    *last_flag = (old == (unsigned)(p.splits - 1)) ? 1 : 0;
                }
                named_bar_sync(TC_EPI_BAR, TC_EPI_THREADS);
                if (*last_flag) {
                    // Last slice of this tile: sum slices 0..S-1 in order.
                    __threadfence();
                    if (gm < p.M) {
                        const float *base = p.ws + ((size_t)tile * p.splits * TC_BM + row) * BN;
#pragma unroll 1
                        for (int c = 0; c < BN / 32; ++c) {
                            float v[32];
#pragma unroll 1
                            for (int s = 0; s < p.splits; ++s) {
                                const float4 *src = reinterpret_cast<const float4 *>(
                                    base + (size_t)s * TC_BM * BN + c * 32);
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    const float4 x = __ldcg(src + j);
                                    if (s == 0) {
                                        v[4 * j] = x.x;
                                        v[4 * j + 1] = x.y;
                                        v[4 * j + 2] = x.z;
                                        v[4 * j + 3] = x.w;
                                    } else {
                                        v[4 * j] += x.x;
                                        v[4 * j + 1] += x.y;
                                        v[4 * j + 2] += x.z;
                                        v[4 * j + 3] += x.w;
                                    }
                                }
                            }
                            store_row_chunk(p, gm, gn0 + c * 32, v);
                        }
                    }
                    if (et == 0) p.counters[tile] = 0u;  // ready for the next launch
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 2-D bf16 tensor map over a row-major matrix: `inner` contiguous elements
// per row, `outer` rows, `pitch` elements between rows; box of
// box_inner x box_outer with 128-byte swizzle; out-of-range reads give 0.
bool make_map(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
              uint64_t pitch, uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Exactly one of st (library-owned workspace, grown on demand) and ext
// (caller-provided scratch, never allocated) supplies the split-K storage.
template <int BN>
int launch_tc(int device, int sm_count, DeviceState *st, const ExternalScratch *ext,
              TcParams &p, const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
              cudaStream_t stream) {
    using Cfg = TcCfg<BN>;
    static bool attr_done[kMaxDevices] = {};
    if (!attr_done[device]) {
        if (cudaFuncSetAttribute(bf16_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::SMEM_ALLOC) != cudaSuccess)
            return GEMM_ERR_CUDA;
        attr_done[device] = true;
    }
    alignas(64) CUtensorMap ta, tb;
    if (!make_map(&ta, A, (uint64_t)p.K, (uint64_t)p.M, (uint64_t)lda, TC_BK, TC_BM))
        return GEMM_ERR_CUDA;
    if (!make_map(&tb, B, (uint64_t)p.N, (uint64_t)p.K, (uint64_t)ldb, 64, TC_BK))
        return GEMM_ERR_CUDA;

    p.num_m_blk = (p.M + TC_BM - 1) / TC_BM;
    p.num_n_blk = (p.N + BN - 1) / BN;
    p.num_kb = (p.K + TC_BK - 1) / TC_BK;
    const long long tiles = (long long)p.num_m_blk * p.num_n_blk;
    int splits = 1;
    const RuntimeConfig cfg = runtime_config();
    if (cfg.split_k > 0) {
        splits = (int)cfg.split_k;
    } else if (tiles * 2 <= sm_count && p.num_kb >= 8) {
        splits = (int)(sm_count / tiles);
        if (splits > p.num_kb / 4) splits = p.num_kb / 4;
    }
    if (splits < 1) splits = 1;
    if (splits > p.num_kb) splits = p.num_kb;
    p.kb_per_split = (p.num_kb + splits - 1) / splits;
    p.splits = (p.num_kb + p.kb_per_split - 1) / p.kb_per_split;  // no empty slice
    const long long units = tiles * p.splits;
    if (units > 0x7fffffffLL) return GEMM_ERR_TOO_LARGE;
    p.num_units = (int)units;
    p.ws = nullptr;
    p.counters = nullptr;
    if (p.splits > 1) {
        const size_t ws_bytes = (size_t)units * TC_BM * BN * sizeof(float);
        if (ext) {
            if (ws_bytes > ext->ws_bytes || (size_t)tiles > ext->counters_n)
                return GEMM_ERR_SCRATCH_LIMIT;
            // The counters must start at zero; a call that gave up earlier
            // may have left some mid-count.
            if (cudaMemsetAsync(ext->counters, 0, (size_t)tiles * sizeof(unsigned), stream) !=
                cudaSuccess)
                return GEMM_ERR_CUDA;
            p.ws = ext->ws;
            p.counters = ext->counters;
        } else {
            const int rc = ensure_splitk_workspace(st, ws_bytes, (size_t)tiles);
            if (rc != GEMM_OK) return rc;
            p.ws = st->splitk_ws;
            p.counters = st->splitk_counters;
        }
    }
    const int grid = (int)(units < sm_count ? units : sm_count);
    bf16_tc_kernel<BN><<<grid, TC_THREADS, Cfg::SMEM_ALLOC, stream>>>(ta, tb, p);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

}  // namespace

namespace {

int launch_common(int device, int sm_count, DeviceState *st, const ExternalScratch *ext,
                  unsigned long long *fault_word, int M, int N, int K, float alpha,
                  const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb, float beta,
                  void *C, int64_t ldc, bool c_f32, cudaStream_t stream) {
    TcParams p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.C = C;
    p.ldc = ldc;
    p.c_f32 = c_f32 ? 1 : 0;
    const int esz = c_f32 ? 4 : 2;
    p.c_vec = ((reinterpret_cast<uintptr_t>(C) & 15) == 0) && ((ldc * esz) % 16 == 0);
    p.fault_word = fault_word;
    const RuntimeConfig cfg = runtime_config();
    p.timeout_ns = (unsigned long long)cfg.watchdog_ms * 1000000ull;
    p.fault_inject = cfg.fault_inject ? 1 : 0;
    if (p.fault_inject) consume_fault_inject();
    int bn = (int)cfg.bf16_tile_n;
    if (bn != 128 && bn != 256) bn = (N <= 128) ? 128 : 256;
    return bn == 256 ? launch_tc<256>(device, sm_count, st, ext, p, A, lda, B, ldb, stream)
                     : launch_tc<128>(device, sm_count, st, ext, p, A, lda, B, ldb, stream);
}

}  // namespace

int launch_bf16_tcgen05(DeviceState *st, int M, int N, int K, float alpha, const uint16_t *A,
                        int64_t lda, const uint16_t *B, int64_t ldb, float beta, void *C,
                        int64_t ldc, bool c_f32, cudaStream_t stream) {
    return launch_common(st->device, st->sm_count, st, nullptr, st->fault_word, M, N, K, alpha,
                         A, lda, B, ldb, beta, C, ldc, c_f32, stream);
}

int launch_bf16_tcgen05_external(int device, int sm_count, const ExternalScratch &ext, int M,
                                 int N, int K, float alpha, const uint16_t *A, int64_t lda,
                                 const uint16_t *B, int64_t ldb, float beta, void *C,
                                 int64_t ldc, bool c_f32, cudaStream_t stream) {
    return launch_common(device, sm_count, nullptr, &ext, ext.fault_word, M, N, K, alpha, A, lda,
                         B, ldb, beta, C, ldc, c_f32, stream);
}

}  // namespace gemm
