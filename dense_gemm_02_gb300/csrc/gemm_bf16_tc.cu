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
//     memory ring (A: the rows the launch needs, K-major, 128-byte swizzle;
//     B: BN/64 boxes of 64 x 64, N-major, 128-byte swizzle; the stages are
//     packed, so small-M launches get more of them); warp 1 allocates tensor
//     memory and runs the MMA loop as a whole warp, one elected lane issuing
//     each tcgen05.mma (M = 128, N = BN, K = 16) into one of two TMEM
//     accumulators; warps 2-5 drain the other accumulator with tcgen05.ld,
//     apply alpha/beta in fp32, convert and store, so a tile's epilogue
//     overlaps the next tile's main loop.
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

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "epilogue.cuh"
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
// Epilogue staging for TMA stores: each epilogue warp owns two 4 KiB
// buffers (a 32 x 32 fp32 or bf16 chunk of C, swizzled), 1024-byte aligned.
constexpr int kEpiChunkBytes = 4096;
constexpr int kEpiStagingBytes = 4 * 2 * kEpiChunkBytes;

// The operand ring of the single-CTA kernel is packed: a stage holds the A
// rows the launch loads (a_slot bytes: 16 KiB for 128 rows, less for a
// small M) followed by the B tile, so small-M launches fit more stages in
// the same bytes and keep more loads in flight (up to MAX_STAGES).
template <int BN>
struct TcCfg {
    static constexpr int STAGES = (BN == 256) ? 4 : 6;  // with 128 A rows
    static constexpr int MAX_STAGES = 12;
    static constexpr int A_BYTES = TC_BM * TC_BK * 2;  // 16 KiB
    static constexpr int B_BYTES = BN * TC_BK * 2;     // 32 KiB at BN = 256
    static constexpr int B_BOX_BYTES = 64 * TC_BK * 2; // one 64-column B box, 8 KiB
    static constexpr int RING_BYTES = STAGES * (A_BYTES + B_BYTES);
    static constexpr int OFF_STAGE = RING_BYTES;  // epilogue staging
    static constexpr int OFF_BAR = OFF_STAGE + kEpiStagingBytes;
    static constexpr int NUM_BARS = 2 * MAX_STAGES + 5;  // full, empty, tfull[2], tempty[2], drain
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
    // Stream-K (single-CTA kernel): the tiles' K iterations, tiles * num_kb
    // in tile-major order, are cut into gridDim.x contiguous ranges of equal
    // length, one per CTA; a tile shared by several CTAs is summed in a
    // workspace with up to max_parts slices per tile.
    int stream_k;
    int max_parts;
    int num_units;
    int group_m;     // M-blocks per raster band
    int tiles_main;  // tiles run at full width; the rest are split along N
    int tail_split;  // sub-tiles per tail tile (1, 2 or 4)
    // CTA-pair kernel: which units run their K blocks two at a time (one
    // barrier wait and eight MMAs per pair of stages): 0 every unit, 1 the
    // narrower tail sub-tiles only, 2 none.
    int stage_pairs;
    // CTA-pair kernel: the K-pair tensor maps are valid (see make_kpair_maps).
    int kpair;
    float alpha, beta;
    void *C;
    long long ldc;
    int c_f32;
    int c_vec;
    int c_tma;  // C is written by TMA stores through shared memory
    float *ws;
    unsigned *counters;
    int ws_tiles;  // tiles the split-K workspace and counters cover (checked in the debug build)
    unsigned long long *fault_word;
    unsigned long long timeout_ns;
    int fault_inject;
    EpiParams epi;  // bias / activation of the fused epilogue
    int a_mn;       // A stored K x M (op(A) = A^T): MN-major A tiles
    int b_kmaj;     // B stored N x K (op(B) = B^T): K-major B tiles
    // Strided batch: tile t is tile t % tiles_per_batch of matrix
    // t / tiles_per_batch; a_bmul / b_bmul are 0 for an operand shared by
    // the whole batch (its TMA batch coordinate stays 0); C matrix i starts
    // c_bstride elements after C.
    int tiles_per_batch, a_bmul, b_bmul;
    long long c_bstride;
    // Small M (one 128-row block, single-CTA kernel): A is loaded as
    // a_rows rows (a multiple of 8 covering M) instead of 128; the MMA still
    // reads 128 rows, the rest being stale shared memory whose products land
    // in accumulator rows past M, which are never stored.
    int a_rows;
    // Packed operand ring (single-CTA kernel): `stages` stages of
    // stage_bytes, each a_slot bytes of A followed by the B tile.
    int stages, stage_bytes, a_slot;
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

// The same descriptor with its start address moved by `bytes` (a multiple of
// 16).  Only the 14-bit start field changes; every address used here stays
// below 228 KiB, so the field (address >> 4 < 16384) cannot carry.
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) {
    return desc + (bytes >> 4);
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A bf16 (7-9 = 1), B bf16 (10-12 = 1), A major-ness in bit 15 (0: K-major,
// A row-major M x K; 1: MN-major, A stored K x M), B major-ness in bit 16
// (1: MN-major, B row-major K x N; 0: K-major, B stored N x K), N >> 3 in
// bits 17-22, M >> 4 in 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int n, int m, int a_mn, int b_kmaj) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(a_mn ? 1 : 0) << 15) |
           ((uint32_t)(b_kmaj ? 0 : 1) << 16) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

// Shared-memory operand tiles of one 64-deep K block, per layout (all with
// the 128-byte swizzle, rows of 128 bytes, 8-row groups 1024 bytes apart):
//   K-major   (A row-major, or B stored N x K): one row per M (or N) index
//             holding 64 K values; a K step of 16 moves 32 bytes along the
//             row.  Loaded as 64-wide K boxes of 128 (A) or 64 (B) rows.
//   MN-major  (A stored K x M, or B row-major): one row per K index holding
//             64 M (or N) values, 64-column boxes 8 KiB apart; a K step of 16
//             is 16 rows, 2048 bytes.
// Descriptors: K-major LBO 16 (unused with swizzling), SBO 1024; MN-major
// LBO = 8192 (the next 64 columns), SBO 1024.
struct OperandLayout {
    uint32_t lbo;   // leading-dimension byte offset of the descriptor
    uint32_t step;  // descriptor start-address step per K = 16, in 16-byte units
};
__device__ __forceinline__ OperandLayout operand_layout(int mn_major) {
    // K-major: TC_UMMA_K bf16 values along a row; MN-major: TC_UMMA_K rows.
    return mn_major ? OperandLayout{8192u, (TC_UMMA_K * 128u) >> 4}
                    : OperandLayout{16u, (TC_UMMA_K * 2u) >> 4};
}

// One unit of work: output rows m_blk*128.., columns n0..n0+width-1, K
// blocks kb0..kb1-1.  `tile` indexes the full-width tile (split-K counters);
// the tile's K range is shared by `nparts` units, this one being number
// `part` in K order (nparts == 1: the unit owns the whole tile).
struct Unit {
    int tile, m_blk, n0, width, kb0, kb1, part, nparts;
    int bidx;  // matrix of the batch
};

// C of matrix bidx of the batch.
__device__ __forceinline__ void *c_matrix(const TcParams &p, int bidx) {
    return static_cast<char *>(p.C) + (long long)bidx * p.c_bstride * (p.c_f32 ? 4 : 2);
}

// Unit order: split-K launches enumerate (tile, slice); otherwise the first
// tiles_main tiles run at full width BN and each remaining tile (the last,
// partial wave of the persistent grid) is cut into tail_split narrower
// sub-tiles so that the partial wave spreads over more SMs.
template <int BN>
__device__ __forceinline__ Unit decode_unit(const TcParams &p, int u) {
    Unit r;
    int sub = 0, nsub = 1;
    r.part = 0;
    r.nparts = p.splits;
    if (p.splits > 1) {
        r.tile = u / p.splits;
        r.part = u - r.tile * p.splits;
    } else if (u < p.tiles_main) {
        r.tile = u;
    } else {
        const int v = u - p.tiles_main;
        r.tile = p.tiles_main + v / p.tail_split;
        sub = v - (v / p.tail_split) * p.tail_split;
        nsub = p.tail_split;
    }
    int n_blk;
    r.bidx = r.tile / p.tiles_per_batch;
    grouped_tile_coords(r.tile - r.bidx * p.tiles_per_batch, p.num_m_blk, p.num_n_blk, p.group_m,
                        r.m_blk, n_blk);
    r.width = BN / nsub;
    r.n0 = n_blk * BN + sub * r.width;
    r.kb0 = r.part * p.kb_per_split;
    r.kb1 = min(r.kb0 + p.kb_per_split, p.num_kb);
    return r;
}

// Stream-K: the CTA that owns K iteration x of the tile-major sequence of
// T = tiles * num_kb iterations cut into P ranges [c*T/P, (c+1)*T/P).
__device__ __forceinline__ long long sk_owner(long long x, long long P, long long T) {
    return ((x + 1) * P - 1) / T;
}

// The i-th unit this CTA works on (false: none left).  Persistent mode:
// units blockIdx.x, blockIdx.x + gridDim.x, ...  Stream-K: the i-th piece
// of this CTA's iteration range, cut at tile boundaries.
template <int BN>
__device__ __forceinline__ bool cta_unit(const TcParams &p, int i, Unit &w) {
    if (!p.stream_k) {
        const long long u = (long long)blockIdx.x + (long long)i * gridDim.x;
        if (u >= p.num_units) return false;
        w = decode_unit<BN>(p, (int)u);
        return true;
    }
    const long long P = gridDim.x, nkb = p.num_kb;
    const long long T = (long long)p.num_units * nkb;  // num_units = tiles here
    const long long c = blockIdx.x;
    const long long s = c * T / P, e = (c + 1) * T / P;
    const long long t0 = s / nkb;
    const long long t = t0 + i;
    const long long pos = (i == 0) ? s : t * nkb;
    if (pos >= e) return false;
    w.tile = (int)t;
    w.kb0 = (int)(pos - t * nkb);
    w.kb1 = (int)min(nkb, e - t * nkb);
    const long long first = sk_owner(t * nkb, P, T), last = sk_owner(t * nkb + nkb - 1, P, T);
    w.part = (int)(c - first);
    w.nparts = (int)(last - first + 1);
    int n_blk;
    w.bidx = w.tile / p.tiles_per_batch;
    grouped_tile_coords(w.tile - w.bidx * p.tiles_per_batch, p.num_m_blk, p.num_n_blk, p.group_m,
                        w.m_blk, n_blk);
    w.width = BN;
    w.n0 = n_blk * BN;
    return true;
}

__device__ __forceinline__ void record_fault_word(unsigned long long *fault_word,
                                                  volatile int *abort_flag, unsigned role,
                                                  unsigned stage, unsigned tile) {
    *abort_flag = 1;
    atomicCAS(fault_word, 0ull, fault_code(role, stage, tile));
}

__device__ __forceinline__ void record_fault(const TcParams &p, volatile int *abort_flag,
                                             unsigned role, unsigned stage, unsigned tile) {
    record_fault_word(p.fault_word, abort_flag, role, stage, tile);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

// Stores 32 consecutive outputs of row gm starting at column gn:
// C = alpha * acc + beta * C, converted to C's type.  (With the fused
// epilogue, acc already holds act(alpha * acc + bias) and alpha is 1.)
__device__ __forceinline__ void store_row_chunk(const TcParams &p, float alpha, void *C, int gm,
                                                int gn,
                                                const float (&acc)[32]) {
    if (gm >= p.M) return;
    const float beta = p.beta;
    if (p.c_f32) {
        float *crow = static_cast<float *>(C) + (long long)gm * p.ldc;
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
        uint16_t *crow = static_cast<uint16_t *>(C) + (long long)gm * p.ldc;
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

// Writes columns gn..gn+31 of the warp's 32 rows (gm0..gm0+31; this thread's
// row is gm0 + lane) as C = alpha * acc + beta * C through the warp's
// staging buffers and a TMA store.  The staging layout is the one the C
// tensor map's swizzle expects: fp32 rows of 128 bytes with 16-byte chunk c
// at c ^ (row & 7); bf16 rows of 64 bytes with chunk c at c ^ ((row >> 1) & 3).
// Stores are asynchronous; a buffer is reused once the store issued two
// chunks earlier has finished reading it.
template <bool B3>
__device__ __forceinline__ void store_chunk_tma(const TcParams &p, float alpha, void *C, int bidx,
                                                const CUtensorMap *tmC,
                                                uint8_t *warp_stage, uint32_t &seq, int lane,
                                                int gm0, int gn, const float (&acc)[32]) {
    const int gm = gm0 + lane;
    const float beta = p.beta;
    float o[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) o[j] = alpha * acc[j];
    if (beta != 0.f && gm < p.M) {
        if (p.c_f32) {
            const float *crow = static_cast<const float *>(C) + (long long)gm * p.ldc + gn;
            if (gn + 32 <= p.N) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 c = reinterpret_cast<const float4 *>(crow)[j];
                    o[4 * j] = fmaf(alpha, acc[4 * j], beta * c.x);
                    o[4 * j + 1] = fmaf(alpha, acc[4 * j + 1], beta * c.y);
                    o[4 * j + 2] = fmaf(alpha, acc[4 * j + 2], beta * c.z);
                    o[4 * j + 3] = fmaf(alpha, acc[4 * j + 3], beta * c.w);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (gn + j < p.N) o[j] = fmaf(alpha, acc[j], beta * crow[j]);
            }
        } else {
            const uint16_t *crow = static_cast<const uint16_t *>(C) + (long long)gm * p.ldc + gn;
            if (gn + 32 <= p.N) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 c = reinterpret_cast<const uint4 *>(crow)[j];
                    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const uint32_t h = (e & 1) ? (cw[e >> 1] >> 16) : (cw[e >> 1] & 0xFFFFu);
                        o[8 * j + e] = fmaf(alpha, acc[8 * j + e], beta * bf16_bits_to_float(h));
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (gn + j < p.N)
                        o[j] = fmaf(alpha, acc[j], beta * bf16_bits_to_float(crow[j]));
            }
        }
    }
    uint8_t *buf = warp_stage + (seq & 1u) * kEpiChunkBytes;
    if (lane == 0) bulk_wait_group_read<1>();
    __syncwarp();
    if (p.c_f32) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4 *>(buf + lane * 128 + ((c ^ (lane & 7)) * 16)) =
                make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                __nv_bfloat162 pr = __floats2bfloat162_rn(o[8 * c + 2 * e], o[8 * c + 2 * e + 1]);
                w[e] = *reinterpret_cast<uint32_t *>(&pr);
            }
            *reinterpret_cast<uint4 *>(buf + lane * 64 + ((c ^ ((lane >> 1) & 3)) * 16)) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
        // A chunk wholly outside C stores nothing, but still closes a
        // (then empty) group so that the buffer-reuse wait above always
        // refers to the store issued two chunks earlier.
        if (gm0 < p.M && gn < p.N &&
            debug_check(p.fault_word, gn % (p.c_f32 ? 4 : 8) == 0, kSiteStoreC, 0)) {
            if constexpr (B3)
                tma_store_3d(tmC, buf, gn, gm0, bidx);
            else
                tma_store_2d(tmC, buf, gn, gm0);
        }
        bulk_commit_group();
    }
    ++seq;
}

// store_chunk_tma for beta != 0 (CTA-pair kernel): the warp's 32 x 32
// chunk of C is first copied into the staging buffer by a TMA load, in the
// layout the store uses, each lane reads its row's 32 values from there,
// and the result overwrites them in place before the TMA store.  A lane's
// row in global memory is 64 or 128 contiguous bytes, so loading C directly
// takes each warp load across 32 rows; through the TMA the shared-memory
// banks see 16 wavefronts per chunk instead of 128, which leaves them to the
// tensor cores' operand reads (measured on GB300, beta = 1 against beta =
// 0: 8192 x 14336 x 4096 cost 6.3%, 4096^3 8.5% with direct loads).
// cbar: the warp's two C-load barriers, one per staging buffer; each
// completes once per use of its buffer (every second chunk), also for a
// chunk outside C (a plain arrive then), so seq alone gives its phase.
template <bool B3>
__device__ __forceinline__ void store_chunk_tma_cload(const TcParams &p, float alpha, int bidx,
                                                      const CUtensorMap *tmC, uint8_t *warp_stage,
                                                      uint64_t *cbar, uint32_t &seq, int lane,
                                                      int gm0, int gn, const float (&acc)[32],
                                                      volatile int *abort_flag) {
    const float beta = p.beta;
    uint8_t *buf = warp_stage + (seq & 1u) * kEpiChunkBytes;
    uint64_t *bar = cbar + (seq & 1u);
    const uint32_t parity = (seq >> 1) & 1u;
    const bool in = gm0 < p.M && gn < p.N &&
                    debug_check(p.fault_word, gn % (p.c_f32 ? 4 : 8) == 0, kSiteStoreC, 0);
    if (lane == 0) {
        bulk_wait_group_read<1>();  // the store issued two chunks ago has read buf
        if (in) {
            mbar_arrive_expect_tx(bar, 32u * 32u * (p.c_f32 ? 4u : 2u));
            if constexpr (B3)
                tma_load_3d(buf, tmC, bar, gn, gm0, bidx);
            else
                tma_load_2d(buf, tmC, bar, gn, gm0);
        } else {
            mbar_arrive(bar);
        }
    }
    __syncwarp();
    // Waits even when another role has raised the abort flag (bounded by
    // the time limit), so that no load into buf is still in flight when the
    // buffer is rewritten or the CTA exits.
    if (!mbar_wait(bar, parity, abort_flag, p.timeout_ns, true) && lane == 0)
        record_fault(p, abort_flag, kRoleEpilogue, 0xfc, 0);
    if (p.c_f32) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float4 *slot = reinterpret_cast<float4 *>(buf + lane * 128 + ((c ^ (lane & 7)) * 16));
            const float4 v = *slot;
            *slot = make_float4(fmaf(alpha, acc[4 * c], beta * v.x),
                                fmaf(alpha, acc[4 * c + 1], beta * v.y),
                                fmaf(alpha, acc[4 * c + 2], beta * v.z),
                                fmaf(alpha, acc[4 * c + 3], beta * v.w));
        }
    } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint4 *slot = reinterpret_cast<uint4 *>(buf + lane * 64 + ((c ^ ((lane >> 1) & 3)) * 16));
            const uint4 v = *slot;
            const uint32_t cw[4] = {v.x, v.y, v.z, v.w};
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float lo = fmaf(alpha, acc[8 * c + 2 * e], beta * bf16_bits_to_float(cw[e] & 0xFFFFu));
                const float hi = fmaf(alpha, acc[8 * c + 2 * e + 1], beta * bf16_bits_to_float(cw[e] >> 16));
                __nv_bfloat162 pr = __floats2bfloat162_rn(lo, hi);
                wv[e] = *reinterpret_cast<uint32_t *>(&pr);
            }
            *slot = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
    }
    fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) {
        if (in) {
            if constexpr (B3)
                tma_store_3d(tmC, buf, gn, gm0, bidx);
            else
                tma_store_2d(tmC, buf, gn, gm0);
        }
        bulk_commit_group();
    }
    ++seq;
}

// One TMA box of an operand: 3-D maps (B3) take the batch coordinate.
template <bool B3>
__device__ __forceinline__ void load_box(void *dst, const CUtensorMap *map, uint64_t *bar, int c0,
                                         int c1, int c2) {
    if constexpr (B3)
        tma_load_3d(dst, map, bar, c0, c1, c2);
    else
        tma_load_2d(dst, map, bar, c0, c1);
}

template <bool B3>
__device__ __forceinline__ void load_box_pair(void *dst, const CUtensorMap *map, uint32_t bar_cl,
                                              int c0, int c1, int c2) {
    if constexpr (B3)
        tma_load_3d_pair(dst, map, bar_cl, c0, c1, c2);
    else
        tma_load_2d_pair(dst, map, bar_cl, c0, c1);
}

// Whether the single-CTA kernel takes its K blocks two at a time (see
// stage_pairs_for): only with a ring of six or more stages.  Measured on
// GB300: the packed small-M rings (8 to 12 stages) gain (decode 64 x 8192 x
// 8192 37.0 -> 36.1 us, a GEMV 36.8 -> 34.8 us), the four-stage ring of the
// 256-wide tiles loses (4096^3 on this kernel 104 -> 112 us).
__device__ __forceinline__ bool single_cta_pairs(const TcParams &p) {
    return p.stage_pairs != 2 && p.stages >= 6;
}

// TMA producer of the single-CTA kernel (lane 0 of warp 0) for one operand
// layout: A_MN, A stored K x M (two 64 (M) x 64 (K) boxes per stage); B_KM,
// B stored N x K (64 (K) x 64 (N) boxes); else row-major A (one 64 (K) x
// 128 (M) box) and B (64 (N) x 64 (K) boxes).  Every layout fills a stage
// with the same bytes.
template <int BN, bool A_MN, bool B_KM, bool B3>
__device__ __forceinline__ void tc_producer(const TcParams &p, const CUtensorMap *tmA,
                                            const CUtensorMap *tmB, uint8_t *ring,
                                            uint64_t *full, uint64_t *empty,
                                            volatile int *abort_flag) {
    using Cfg = TcCfg<BN>;
    const uint32_t S = (uint32_t)p.stages;
    uint32_t it = 0, s = 0, ph = 0;
    int withheld = 0;  // stages the fault-injection hook left unfilled
    bool ok = true;
    Unit w;
    for (int ui = 0; ok && cta_unit<BN>(p, ui, w); ++ui) {
        if (w.n0 >= p.N) continue;  // sub-tile wholly past the N edge
        const int boxes = w.width / 64;
        // A bytes per stage: a_rows rows of 64 K values (K-major), or the
        // one or two 64-row boxes of an MN-major A.
        const uint32_t a_tx =
            A_MN ? (p.a_rows > 64 ? 2u : 1u) * 8192u : (uint32_t)p.a_rows * 128u;
        const uint32_t tx = a_tx + boxes * Cfg::B_BOX_BYTES;
        const int m0 = w.m_blk * TC_BM;
        const int ab = w.bidx * p.a_bmul, bb = w.bidx * p.b_bmul;  // batch coordinates
        // Copies of K block kb into stage st, completing on `bar`.
        auto load_stage = [&](uint32_t st, int kb, uint64_t *bar) {
            uint8_t *a_dst = ring + st * (uint32_t)p.stage_bytes;
            uint8_t *b_dst = a_dst + p.a_slot;
            const int k0 = kb * TC_BK;
            // Debug build: innermost (x) coordinates a multiple of 8 bf16
            // elements (16 bytes); the copies inside stage st of the ring.
            if (!debug_check(p.fault_word, st < S && (A_MN ? m0 % 8 : k0 % 8) == 0 &&
                                               (int)a_tx <= p.a_slot,
                             kSiteLoadA, w.tile) ||
                !debug_check(p.fault_word, (B_KM ? k0 % 8 : w.n0 % 8) == 0 &&
                                               p.a_slot + boxes * Cfg::B_BOX_BYTES <= p.stage_bytes,
                             kSiteLoadB, w.tile))
                return;
            if constexpr (A_MN) {
                load_box<B3>(a_dst, tmA, bar, m0, k0, ab);
                if (p.a_rows > 64) load_box<B3>(a_dst + 8192, tmA, bar, m0 + 64, k0, ab);
            } else {
                load_box<B3>(a_dst, tmA, bar, k0, m0, ab);
            }
            for (int j = 0; j < boxes; ++j) {
                if constexpr (B_KM)
                    load_box<B3>(b_dst + j * Cfg::B_BOX_BYTES, tmB, bar, k0, w.n0 + j * 64, bb);
                else
                    load_box<B3>(b_dst + j * Cfg::B_BOX_BYTES, tmB, bar, w.n0 + j * 64, k0, bb);
            }
        };
        const bool paired = single_cta_pairs(p);
        for (int kb = w.kb0; kb < w.kb1 && ok;) {
            // Paired (as in the CTA-pair kernel): K blocks kb and kb + 1 go to
            // consecutive stages cur and nxt, both completing on full[cur];
            // full[nxt] is arrived at once to keep its phase in step.
            const bool two = paired && kb + 1 < w.kb1;
            const uint32_t cur = s, cur_ph = ph;
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
            uint32_t nxt = 0, nxt_ph = 0;
            if (two) {
                nxt = s;
                nxt_ph = ph;
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // For two stages wait on the second one's empty barrier alone: the
            // MMA thread commits stage nxt after stage cur, and a tcgen05
            // commit arrives only once every earlier MMA of that thread has
            // finished, so stage cur is free by then too.
            if ((!two && !mbar_wait(&empty[cur], cur_ph ^ 1u, abort_flag, p.timeout_ns)) ||
                (two && !mbar_wait(&empty[nxt], nxt_ph ^ 1u, abort_flag, p.timeout_ns))) {
                record_fault(p, abort_flag, kRoleProducer, cur, w.tile);
                ok = false;
                break;
            }
            const int step = two ? 2 : 1;
            if (p.fault_inject && blockIdx.x == 0 && it == 0) {
                withheld = step;  // test hook: these stages are never filled
                it += step;
                kb += step;
                continue;
            }
            mbar_arrive_expect_tx(&full[cur], (uint32_t)step * tx);
            if (two) mbar_arrive(&full[nxt]);
            load_stage(cur, kb, &full[cur]);
            if (two) load_stage(nxt, kb + 1, &full[cur]);
            it += step;
            kb += step;
        }
    }
    // Let every copy started here land before the CTA can exit.
    const uint32_t first = it > S ? it - S : 0u;
    for (uint32_t i = first; i < it; ++i) {
        if ((int)i < withheld) continue;  // withheld: the first 1 or 2 stages
        mbar_wait(&full[i % S], (i / S) & 1u, abort_flag, p.timeout_ns, true);
    }
}

// The producer loop for the launch's operand layouts, chosen once: per-stage
// branches in this single thread measurably slow the pipeline.
template <int BN, bool B3>
__device__ __forceinline__ void tc_produce_layout(const TcParams &p, const CUtensorMap *tmA,
                                                  const CUtensorMap *tmB, uint8_t *ring,
                                                  uint64_t *full, uint64_t *empty,
                                                  volatile int *abort_flag) {
    if (!p.a_mn && !p.b_kmaj)
        tc_producer<BN, false, false, B3>(p, tmA, tmB, ring, full, empty, abort_flag);
    else if (!p.a_mn)
        tc_producer<BN, false, true, B3>(p, tmA, tmB, ring, full, empty, abort_flag);
    else if (!p.b_kmaj)
        tc_producer<BN, true, false, B3>(p, tmA, tmB, ring, full, empty, abort_flag);
    else
        tc_producer<BN, true, true, B3>(p, tmA, tmB, ring, full, empty, abort_flag);
}

// Reads two consecutive 32-column chunks (64 floats) of this thread's
// accumulator row from tensor memory (columns taddr .. taddr + 63).
__device__ __forceinline__ void tmem_ld_chunk_pair(uint32_t taddr, float (&x)[2][32]) {
    uint32_t r0[32], r1[32];
    tmem_ld_32x32b_x32(taddr, r0);
    tmem_ld_32x32b_x32(taddr + 32, r1);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) x[0][j] = __uint_as_float(r0[j]), x[1][j] = __uint_as_float(r1[j]);
}

// Loads two consecutive 32-column chunks (64 floats) of this thread's row
// of a partial tile from the split-K workspace (float4 i of the pair at
// src + i * 32: the warp-coalesced workspace layout), all sixteen loads
// issued together.
__device__ __forceinline__ void load_partial_chunks(const float4 *src, float (&x)[2][32]) {
    float4 t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = __ldcg(src + i * 32);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float *d = &x[i >> 3][(i & 7) * 4];
        d[0] = t[i].x, d[1] = t[i].y, d[2] = t[i].z, d[3] = t[i].w;
    }
}

// Fused epilogue, first part: v[j] = act(alpha * v[j] + bias[gn + j]) for
// the 32 columns gn..gn+31 (columns past N use bias[N - 1]; they are never
// stored).  The store helpers then add beta * C with alpha = 1.  The bias
// chunk is read with 16-byte loads when it is aligned and inside N; the
// activation is chosen once per chunk, so each unrolled loop holds one form.
__device__ __forceinline__ void apply_pre(const TcParams &p, int gn, float (&v)[32]) {
    const float alpha = p.alpha;
    if (p.epi.bias) {
        float b[32];
        const uintptr_t addr = reinterpret_cast<uintptr_t>(p.epi.bias);
        if (gn + 32 <= p.N && p.epi.bias_f32 && (addr & 15) == 0) {
            const float4 *src = static_cast<const float4 *>(p.epi.bias) + (gn >> 2);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 x = __ldg(src + q);
                b[4 * q] = x.x, b[4 * q + 1] = x.y, b[4 * q + 2] = x.z, b[4 * q + 3] = x.w;
            }
        } else if (gn + 32 <= p.N && !p.epi.bias_f32 && (addr & 15) == 0) {
            const uint4 *src = static_cast<const uint4 *>(p.epi.bias) + (gn >> 3);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 x = __ldg(src + q);
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    b[8 * q + e] = __uint_as_float((e & 1) ? (w[e >> 1] & 0xFFFF0000u)
                                                           : (w[e >> 1] << 16));
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) b[j] = epi_bias(p.epi, min(gn + j, p.N - 1));
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = fmaf(alpha, v[j], b[j]);
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= alpha;
    }
    if (p.epi.act == 2) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = gelu_tanh(v[j]);
    } else if (p.epi.act == 1) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = relu(v[j]);
    }
}

// EPI: the fused bias / activation epilogue is compiled in (a separate
// instantiation, so the plain kernel's epilogue code stays as small as it
// can be: its size measurably affects the main loop's speed).
template <int BN, bool EPI, bool B3>
__global__ void __launch_bounds__(TC_THREADS, 1)
    bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams p) {
    using Cfg = TcCfg<BN>;
    constexpr int SMAX = Cfg::MAX_STAGES;
    const uint32_t S = (uint32_t)p.stages;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzled tiles need 1024-byte aligned shared addresses.
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
    uint64_t *full = bars;
    uint64_t *empty = bars + SMAX;
    uint64_t *tfull = bars + 2 * SMAX;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
    uint32_t *tmem_slot = misc;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    volatile int *last_flag = reinterpret_cast<volatile int *>(misc + 2);
    volatile int *epi_ok = reinterpret_cast<volatile int *>(misc + 3);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < S; ++s) {
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
            tc_produce_layout<BN, B3>(p, &tmA, &tmB, ring, full, empty, abort_flag);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // The whole warp runs the loop (every lane waits on the same
        // barriers and takes the same branches); one elected lane issues
        // each MMA and commit.
        {
            // Operand tiles as described at operand_layout.  The loop below
            // only adds offsets to these descriptors: the issuing warp must
            // spend as few instructions as possible between MMAs to keep the
            // tensor pipe fed.
            const OperandLayout la = operand_layout(p.a_mn), lb = operand_layout(!p.b_kmaj);
            const uint64_t a_desc0 = smem_desc_sw128(smem_addr(ring), la.lbo, 1024);
            const uint64_t b_desc0 = smem_desc_sw128(smem_addr(ring + p.a_slot), lb.lbo, 1024);
            const uint32_t stage_bytes = (uint32_t)p.stage_bytes;
            const uint32_t a1 = la.step, a2 = 2 * la.step, a3 = 3 * la.step;
            const uint32_t b1 = lb.step, b2 = 2 * lb.step, b3 = 3 * lb.step;
            uint32_t s = 0, ph = 0, local = 0;
            bool ok = true;
            Unit w;
            for (int ui = 0; ok && cta_unit<BN>(p, ui, w); ++ui) {
                if (w.n0 >= p.N) continue;
                const uint32_t idesc = idesc_bf16_f32(w.width, TC_BM, p.a_mn, p.b_kmaj);
                const uint32_t b = local & 1u, use = local >> 1;
                ++local;
                const bool got = mbar_wait(&tempty[b], (use & 1u) ^ 1u, abort_flag, p.timeout_ns);
                if (__any_sync(0xffffffffu, !got)) {
                    if (lane == 0) record_fault(p, abort_flag, kRoleMma, 0xfe, w.tile);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * BN;
                if (!debug_check(p.fault_word, b * BN + w.width <= Cfg::TMEM_COLS, kSiteTmem,
                                 w.tile)) {
                    ok = false;
                    break;
                }
                uint32_t acc = 0;
                const bool paired = single_cta_pairs(p);
                for (int kb = w.kb0; kb < w.kb1;) {
                    // Paired: stages s and s + 1 both completed on full[s].
                    const bool two = paired && kb + 1 < w.kb1;
                    const bool ready = mbar_wait(&full[s], ph, abort_flag, p.timeout_ns);
                    if (__any_sync(0xffffffffu, !ready)) {
                        if (lane == 0) record_fault(p, abort_flag, kRoleMma, s, w.tile);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t ad = desc_add(a_desc0, s * stage_bytes);
                    const uint64_t bd = desc_add(b_desc0, s * stage_bytes);
                    umma_f16_elect(d_tmem, ad, bd, idesc, acc);
                    umma_f16_elect(d_tmem, ad + a1, bd + b1, idesc, 1u);
                    umma_f16_elect(d_tmem, ad + a2, bd + b2, idesc, 1u);
                    umma_f16_elect(d_tmem, ad + a3, bd + b3, idesc, 1u);
                    umma_commit_elect(&empty[s]);  // frees the stage once these MMAs finish
                    acc = 1u;
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (two) {
                        const uint64_t ad2 = desc_add(a_desc0, s * stage_bytes);
                        const uint64_t bd2 = desc_add(b_desc0, s * stage_bytes);
                        umma_f16_elect(d_tmem, ad2, bd2, idesc, 1u);
                        umma_f16_elect(d_tmem, ad2 + a1, bd2 + b1, idesc, 1u);
                        umma_f16_elect(d_tmem, ad2 + a2, bd2 + b2, idesc, 1u);
                        umma_f16_elect(d_tmem, ad2 + a3, bd2 + b3, idesc, 1u);
                        umma_commit_elect(&empty[s]);
                        if (++s == S) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    kb += two ? 2 : 1;
                }
                if (!ok) break;
                umma_commit_elect(&tfull[b]);  // accumulator b is complete
            }
            // The elected lane's MMAs must finish before TMEM is released.
            umma_commit_elect(drain);
            mbar_wait(drain, 0, abort_flag, p.timeout_ns, true);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue warps 2-5
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        const int et = threadIdx.x - 64;
        uint8_t *warp_stage = smem + Cfg::OFF_STAGE + q * 2 * kEpiChunkBytes;
        uint32_t stage_seq = 0;
        uint32_t local = 0;
        Unit w;
        for (int ui = 0; cta_unit<BN>(p, ui, w); ++ui) {
            if (w.n0 >= p.N) continue;
            const int tile = w.tile;
            const uint32_t b = local & 1u, use = local >> 1;
            ++local;
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
            const int gm = w.m_blk * TC_BM + row;
            void *cmat = c_matrix(p, w.bidx);
            const int gn0 = w.n0;
            if (w.nparts == 1) {
#pragma unroll 1
                for (int c = 0; c < w.width / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, r);
                    tmem_ld_wait();
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    if constexpr (EPI) apply_pre(p, gn0 + c * 32, v);
                    const float alpha = EPI ? 1.f : p.alpha;
                    if (p.c_tma)
                        store_chunk_tma<B3>(p, alpha, cmat, w.bidx, &tmC, warp_stage, stage_seq, lane,
                                        gm - lane, gn0 + c * 32, v);
                    else
                        store_row_chunk(p, alpha, cmat, gm, gn0 + c * 32, v);
                }
                tc_fence_before_sync();
                mbar_arrive(&tempty[b]);
            } else {
                // Split tile: this slice's fp32 partial goes to the workspace
                // in a warp-coalesced layout (per slice: float4
                // ((q * BN/32 + chunk) * 8 + j) * 32 + lane holds columns
                // chunk * 32 + 4j .. +3 of row q * 32 + lane); warps whose 32
                // rows all lie past M skip it.
                const bool rows_in = w.m_blk * TC_BM + q * 32 < p.M &&
                                     debug_check(p.fault_word,
                                                 tile < p.ws_tiles && w.part < p.max_parts,
                                                 kSiteWorkspace, w.tile);
                const size_t slice4 = (size_t)TC_BM * BN / 4;
                float4 *wq = reinterpret_cast<float4 *>(p.ws) +
                             ((size_t)tile * p.max_parts + w.part) * slice4 +
                             (size_t)q * (BN / 32) * 8 * 32 + lane;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tbase + c * 32, r);
                    tmem_ld_wait();
                    if (rows_in) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            __stcg(wq + (c * 8 + j) * 32,
                                   make_float4(__uint_as_float(r[4 * j]),
                                               __uint_as_float(r[4 * j + 1]),
                                               __uint_as_float(r[4 * j + 2]),
                                               __uint_as_float(r[4 * j + 3])));
                    }
                }
                __threadfence();
                named_bar_sync(TC_EPI_BAR, TC_EPI_THREADS);
                if (et == 0) {
                    const unsigned old = atomicAdd(&p.counters[tile], 1u);
                    *last_flag = (old == (unsigned)(w.nparts - 1)) ? 1 : 0;
                }
                named_bar_sync(TC_EPI_BAR, TC_EPI_THREADS);
                if (!*last_flag) {
                    tc_fence_before_sync();
                    mbar_arrive(&tempty[b]);
                }
                if (*last_flag && rows_in) {
                    // Last slice of this tile: each thread sums its own row
                    // over slices 0..S-1 in order, two 32-column chunks at a
                    // time with a slice's sixteen loads in flight together,
                    // then stores the chunks as the plain epilogue does.  Its
                    // own slice it reads back from tensor memory (the same
                    // fp32 values it wrote), so the loads it waits for are
                    // only the other slices'.
                    __threadfence();
                    const float4 *rq = reinterpret_cast<const float4 *>(p.ws) +
                                       (size_t)tile * p.max_parts * slice4 +
                                       (size_t)q * (BN / 32) * 8 * 32 + lane;
#pragma unroll 1
                    for (int c = 0; c < BN / 32; c += 2) {
                        float v[2][32];
                        if (w.part == 0)
                            tmem_ld_chunk_pair(tbase + c * 32, v);
                        else
                            load_partial_chunks(rq + c * 8 * 32, v);
#pragma unroll 1
                        for (int sl = 1; sl < w.nparts; ++sl) {
                            float x[2][32];
                            if (sl == w.part)
                                tmem_ld_chunk_pair(tbase + c * 32, x);
                            else
                                load_partial_chunks(rq + sl * slice4 + c * 8 * 32, x);
#pragma unroll
                            for (int h = 0; h < 2; ++h)
#pragma unroll
                                for (int j = 0; j < 32; ++j) v[h][j] += x[h][j];
                        }
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int gn = gn0 + (c + h) * 32;
                            if constexpr (EPI) apply_pre(p, gn, v[h]);
                            const float alpha = EPI ? 1.f : p.alpha;
                            if (p.c_tma)
                                store_chunk_tma<B3>(p, alpha, cmat, w.bidx, &tmC, warp_stage,
                                                    stage_seq, lane, gm - lane, gn, v[h]);
                            else
                                store_row_chunk(p, alpha, cmat, gm, gn, v[h]);
                        }
                    }
                }
                if (*last_flag) {
                    tc_fence_before_sync();
                    mbar_arrive(&tempty[b]);
                    if (et == 0) p.counters[tile] = 0u;  // ready for the next launch
                }
            }
        }
    }

    if (warp >= 2 && lane == 0) bulk_wait_all();  // TMA stores of C have landed
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}


// ================================================================ CTA pairs
//
// The same GEMM with two CTAs (one per SM, a 2-CTA cluster) sharing each
// tcgen05 MMA (cta_group::2): a 256 x BN output tile per pair, CTA r owning
// rows r*128..r*128+127.  Each CTA loads its own 128 rows of A and its own
// half of the tile's B columns; the even CTA's lane issues MMA M = 256, N =
// BN that reads both CTAs' shared memory and writes both CTAs' TMEM.  Per
// CTA a stage is 32 KiB instead of 48 KiB (B is split between the pair), so
// six stages fit and L2 traffic per flop drops by a third.
//
//   full[s]   (even CTA only) 1 arrival (its producer, expect_tx = both CTAs'
//             bytes) + the TMA bytes of both CTAs (TMA .cta_group::2 signals
//             the even CTA's barrier)
//   empty[s]  (each CTA) arrived by the MMA commit, multicast to both CTAs
//   tfull[b]  (each CTA) arrived by the MMA commit, multicast
//   tempty[b] (even CTA) 8 arrivals: one per epilogue warp of both CTAs
struct Tc2Cfg {
    static constexpr int BN = 256;                     // pair tile width
    static constexpr int STAGES = 6;
    static constexpr int A_BYTES = TC_BM * TC_BK * 2;  // this CTA's 128 rows, 16 KiB
    static constexpr int B_BOX_BYTES = 64 * TC_BK * 2; // 8 KiB
    static constexpr int B_BYTES = 2 * B_BOX_BYTES;    // this CTA's half of 256 columns
    static constexpr int OFF_B = STAGES * A_BYTES;
    static constexpr int OFF_STAGE = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_STAGE + kEpiStagingBytes;
    // full, empty, tfull[2], tempty[2], drain, and two C-load barriers per
    // epilogue warp (one per staging buffer)
    static constexpr int NUM_BARS = 2 * STAGES + 5 + 8;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_ALLOC = SMEM_USED + 1024;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int EPI_WARPS_PER_PAIR = 8;
    static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

// Whether a unit of the CTA-pair kernel runs its K blocks two at a time:
// one barrier wait (with its warp vote and fence) per two 64-deep stages,
// then eight MMAs.  Measured on GB300 (per-stage clock stamps of the issuing
// warp): the wait costs about 67 ns even when the data is there and four
// MMA issues and a commit about 150-175 ns, so a 64-deep stage costs the
// issuer about 255-280 ns, as long as the four M = 256, N = 256 MMAs
// execute (262 ns) and twice as long as four N = 128 ones (131 ns, the
// tail's column halves).  Paired stages leave the tensor pipe the slack:
// 4096^3 90.2 -> 86.8 us pairing only the column halves, 80.1 us pairing
// every tile; the MLP shape 516 -> 470 us; 8192^3 576 -> 549 us.
__device__ __forceinline__ bool stage_pairs_for(const TcParams &p, const Unit &w) {
    return p.stage_pairs == 0 || (p.stage_pairs == 1 && w.width < Tc2Cfg::BN);
}

// TMA producer of the CTA-pair kernel (lane 0 of warp 0 in both CTAs), for
// one operand layout (as tc_producer).  Each CTA loads its own 128 rows of A
// and its half of the tile's B columns; all copies complete on the even
// CTA's full barrier.
template <bool A_MN, bool B_KM, bool B3>
__device__ __forceinline__ void tc2_producer(const TcParams &p, const CUtensorMap *tmA,
                                             const CUtensorMap *tmB, const CUtensorMap *tmA2,
                                             const CUtensorMap *tmB2, const CUtensorMap *tmBh,
                                             uint8_t *sA, uint8_t *sB,
                                             uint64_t *full, uint64_t *empty,
                                             volatile int *abort_flag, uint32_t rank, int pair,
                                             int npairs) {
    using Cfg = Tc2Cfg;
    constexpr int S = Cfg::STAGES;
    const bool leader = (rank == 0);
    uint32_t it = 0;
    int withheld = 0;  // stages the fault-injection hook left unfilled
    bool ok = true;
    for (int u = pair; u < p.num_units && ok; u += npairs) {
        const Unit w = decode_unit<Cfg::BN>(p, u);
        if (w.n0 >= p.N) continue;
        const int half = w.width / 2;  // this CTA's B columns
        const int boxes = half / 64;
        const uint32_t tx = 2u * (Cfg::A_BYTES + boxes * Cfg::B_BOX_BYTES);
        const int row0 = w.m_blk * 2 * TC_BM + (int)rank * TC_BM;
        const int col0 = w.n0 + (int)rank * half;
        const int ab = w.bidx * p.a_bmul, bb = w.bidx * p.b_bmul;  // batch coordinates
        // Copies of K block kb into stage st, completing on the even CTA's
        // barrier full_cl.
        auto load_stage = [&](int st, int kb, uint32_t full_cl) {
            uint8_t *a_dst = sA + st * Cfg::A_BYTES;
            const int k0 = kb * TC_BK;
            // Debug build: x coordinates a multiple of 8 bf16 elements, the
            // copies inside stage st's slots.
            if (!debug_check(p.fault_word, st >= 0 && st < S && (A_MN ? row0 % 8 : k0 % 8) == 0,
                             kSiteLoadA, w.tile) ||
                !debug_check(p.fault_word, (B_KM ? k0 % 8 : col0 % 8) == 0 &&
                                               boxes * Cfg::B_BOX_BYTES <= Cfg::B_BYTES,
                             kSiteLoadB, w.tile))
                return;
            if constexpr (A_MN) {
                load_box_pair<B3>(a_dst, tmA, full_cl, row0, k0, ab);
                load_box_pair<B3>(a_dst + 8192, tmA, full_cl, row0 + 64, k0, ab);
            } else {
                load_box_pair<B3>(a_dst, tmA, full_cl, k0, row0, ab);
            }
            uint8_t *b_dst = sB + st * Cfg::B_BYTES;
            for (int j = 0; j < boxes; ++j) {
                if constexpr (B_KM)
                    load_box_pair<B3>(b_dst + j * Cfg::B_BOX_BYTES, tmB, full_cl, k0,
                                      col0 + j * 64, bb);
                else
                    load_box_pair<B3>(b_dst + j * Cfg::B_BOX_BYTES, tmB, full_cl,
                                      col0 + j * 64, k0, bb);
            }
        };
        // K blocks kb and kb + 1 into stages st and st + 1 (back to back in
        // shared memory) through the K-pair maps: one copy for this CTA's A
        // rows and one for its B columns.  128 B columns fill both stages'
        // B slots; 64 (a column-half tail tile) land in stage st's B slot
        // alone, K block kb + 1 in its second 8 KiB, where the MMA warp
        // reads them (b_half_packed).
        auto load_two = [&](int st, int kb, uint32_t full_cl) {
            // Debug build: both stages inside the ring, the chunk coordinates
            // of the K-pair views whole 64-element chunks.
            if (!debug_check(p.fault_word, st >= 0 && st + 1 < S && (!A_MN || row0 % 64 == 0),
                             kSiteLoadA, w.tile) ||
                !debug_check(p.fault_word,
                             B_KM || col0 % ((boxes == 1 || boxes == 2) ? 64 : 8) == 0,
                             kSiteLoadB, w.tile))
                return;
            uint8_t *a_dst = sA + st * Cfg::A_BYTES;
            if constexpr (A_MN)
                tma_load_4d_pair(a_dst, tmA2, full_cl, 0, 0, row0 / 64, kb);
            else
                tma_load_3d_pair(a_dst, tmA2, full_cl, 0, row0, kb);
            uint8_t *b_dst = sB + st * Cfg::B_BYTES;
            if (boxes == 2) {
                if constexpr (B_KM)
                    tma_load_3d_pair(b_dst, tmB2, full_cl, 0, col0, kb);
                else
                    tma_load_4d_pair(b_dst, tmB2, full_cl, 0, 0, col0 / 64, kb);
                return;
            }
            if (boxes == 1) {
                if constexpr (B_KM)
                    tma_load_3d_pair(b_dst, tmBh, full_cl, 0, col0, kb);
                else
                    tma_load_4d_pair(b_dst, tmBh, full_cl, 0, 0, col0 / 64, kb);
                return;
            }
            for (int h = 0; h < 2; ++h) {
                const int k0 = (kb + h) * TC_BK;
                for (int j = 0; j < boxes; ++j) {
                    uint8_t *d = b_dst + h * Cfg::B_BYTES + j * Cfg::B_BOX_BYTES;
                    if constexpr (B_KM)
                        load_box_pair<B3>(d, tmB, full_cl, k0, col0 + j * 64, bb);
                    else
                        load_box_pair<B3>(d, tmB, full_cl, col0 + j * 64, k0, bb);
                }
            }
        };
        const bool paired = stage_pairs_for(p, w);
        for (int kb = w.kb0; kb < w.kb1 && ok;) {
            // Paired: K blocks kb and kb + 1 go to consecutive stages s and s2
            // and both complete on full[s]; full[s2] is arrived at once (no
            // bytes), which keeps its phase in step with the ring.
            const bool two = paired && kb + 1 < w.kb1;
            const int s = it % S;
            const uint32_t ph = (it / S) & 1u;
            const int s2 = (it + 1) % S;
            const uint32_t ph2 = ((it + 1) / S) & 1u;
            // For two stages wait on s2's empty barrier alone (its commit
            // follows stage s's; see tc_producer).  Measured on GB300: 4096^3
            // 82.9 -> 81.9 us.
            if ((!two && !mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.timeout_ns)) ||
                (two && !mbar_wait(&empty[s2], ph2 ^ 1u, abort_flag, p.timeout_ns))) {
                record_fault(p, abort_flag, kRoleProducer, s, w.tile);
                ok = false;
                break;
            }
            const int step = two ? 2 : 1;
            if (p.fault_inject && pair == 0 && leader && it == 0) {
                withheld = two ? 2 : 1;  // test hook: the stage's barrier never completes
                it += step;
                kb += step;
                continue;
            }
            const uint32_t full_cl = mapa_shared(smem_addr(&full[s]), 0);
            if (leader) {
                mbar_arrive_expect_tx(&full[s], (uint32_t)step * tx);
                if (two) mbar_arrive(&full[s2]);
            }
            if (!B3 && two && p.kpair && s2 == s + 1) {
                load_two(s, kb, full_cl);
            } else {
                load_stage(s, kb, full_cl);
                if (two) load_stage(s2, kb + 1, full_cl);
            }
            it += step;
            kb += step;
        }
    }
    // The even CTA's full barriers count both CTAs' copies: wait for the
    // ones still in flight before the pair may exit.
    if (leader) {
        const uint32_t first = it > (uint32_t)S ? it - S : 0u;
        for (uint32_t i = first; i < it; ++i) {
            if ((int)i < withheld) continue;  // withheld: the first 1 or 2 stages
            mbar_wait(&full[i % S], (i / S) & 1u, abort_flag, p.timeout_ns, true);
        }
    }
}

template <bool B3>
__device__ __forceinline__ void tc2_produce_layout(const TcParams &p, const CUtensorMap *tmA,
                                                   const CUtensorMap *tmB,
                                                   const CUtensorMap *tmA2,
                                                   const CUtensorMap *tmB2,
                                                   const CUtensorMap *tmBh, uint8_t *sA,
                                                   uint8_t *sB, uint64_t *full, uint64_t *empty,
                                                   volatile int *abort_flag, uint32_t rank,
                                                   int pair, int npairs) {
    if (!p.a_mn && !p.b_kmaj)
        tc2_producer<false, false, B3>(p, tmA, tmB, tmA2, tmB2, tmBh, sA, sB, full, empty,
                                       abort_flag, rank, pair, npairs);
    else if (!p.a_mn)
        tc2_producer<false, true, B3>(p, tmA, tmB, tmA2, tmB2, tmBh, sA, sB, full, empty,
                                      abort_flag, rank, pair, npairs);
    else if (!p.b_kmaj)
        tc2_producer<true, false, B3>(p, tmA, tmB, tmA2, tmB2, tmBh, sA, sB, full, empty,
                                      abort_flag, rank, pair, npairs);
    else
        tc2_producer<true, true, B3>(p, tmA, tmB, tmA2, tmB2, tmBh, sA, sB, full, empty,
                                     abort_flag, rank, pair, npairs);
}

template <bool EPI, bool B3>
__global__ void __launch_bounds__(TC_THREADS, 1)
    bf16_tc2_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC,
                    const __grid_constant__ CUtensorMap tmA2,
                    const __grid_constant__ CUtensorMap tmB2,
                    const __grid_constant__ CUtensorMap tmBh, const TcParams p) {
    using Cfg = Tc2Cfg;
    constexpr int S = Cfg::STAGES;
    constexpr int BN = Cfg::BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + Cfg::OFF_B;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
    uint64_t *full = bars;
    uint64_t *empty = bars + S;
    uint64_t *tfull = bars + 2 * S;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint64_t *cload = drain + 1;  // C-load barriers: two per epilogue warp
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
    uint32_t *tmem_slot = misc;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    volatile int *epi_ok = reinterpret_cast<volatile int *>(misc + 3);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = (rank == 0);
    const int pair = (int)cluster_id_x();
    const int npairs = (int)num_clusters_x();

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], Cfg::EPI_WARPS_PER_PAIR);
        }
        mbar_init(drain, 1);
        for (int i = 0; i < 8; ++i) mbar_init(&cload[i], 1);
        *abort_flag = 0;
        *epi_ok = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (p.kpair) {
            prefetch_tensormap(&tmA2);
            prefetch_tensormap(&tmB2);
            prefetch_tensormap(&tmBh);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // the peer's barriers are initialised before any remote signal
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            tc2_produce_layout<B3>(p, &tmA, &tmB, &tmA2, &tmB2, &tmBh, sA, sB, full, empty,
                                   abort_flag, rank, pair, npairs);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA)
        // The whole warp runs the loop (every lane waits on the same
        // barriers and takes the same branches); one elected lane issues
        // each MMA and commit.
        if (leader) {
            // Same descriptor scheme as the single-CTA kernel (offsets only).
            const OperandLayout la = operand_layout(p.a_mn), lb = operand_layout(!p.b_kmaj);
            const uint64_t a_desc0 = smem_desc_sw128(smem_addr(sA), la.lbo, 1024);
            const uint64_t b_desc0 = smem_desc_sw128(smem_addr(sB), lb.lbo, 1024);
            const uint32_t a1 = la.step, a2 = 2 * la.step, a3 = 3 * la.step;
            const uint32_t b1 = lb.step, b2 = 2 * lb.step, b3 = 3 * lb.step;
            uint32_t s = 0, ph = 0, local = 0;
            bool ok = true;
            for (int u = pair; u < p.num_units && ok; u += npairs) {
                const Unit w = decode_unit<BN>(p, u);
                if (w.n0 >= p.N) continue;
                const uint32_t idesc = idesc_bf16_f32(w.width, 2 * TC_BM, p.a_mn, p.b_kmaj);
                const uint32_t b = local & 1u, use = local >> 1;
                ++local;
                const bool got = mbar_wait(&tempty[b], (use & 1u) ^ 1u, abort_flag, p.timeout_ns);
                if (__any_sync(0xffffffffu, !got)) {
                    if (lane == 0) record_fault(p, abort_flag, kRoleMma, 0xfe, w.tile);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + b * BN;
                if (!debug_check(p.fault_word, b * BN + w.width <= Cfg::TMEM_COLS, kSiteTmem,
                                 w.tile)) {
                    ok = false;
                    break;
                }
                uint32_t acc = 0;
                const bool paired = stage_pairs_for(p, w);
                // Column-half tile whose paired K blocks were copied through
                // the K-pair maps: the second block's B sits in the first
                // stage's B slot, 8 KiB in (see tc2_producer).
                const bool b_half_packed = !B3 && p.kpair && w.width == BN / 2;
                for (int kb = w.kb0; kb < w.kb1;) {
                    // Paired: stages s and s + 1 both completed on full[s].
                    const bool two = paired && kb + 1 < w.kb1;
                    const uint32_t s_first = s;
                    const bool ready = mbar_wait(&full[s], ph, abort_flag, p.timeout_ns);
                    if (__any_sync(0xffffffffu, !ready)) {
                        if (lane == 0) record_fault(p, abort_flag, kRoleMma, s, w.tile);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t ad = desc_add(a_desc0, s * Cfg::A_BYTES);
                    const uint64_t bd = desc_add(b_desc0, s * Cfg::B_BYTES);
                    umma_f16_pair_elect(d_tmem, ad, bd, idesc, acc);
                    umma_f16_pair_elect(d_tmem, ad + a1, bd + b1, idesc, 1u);
                    umma_f16_pair_elect(d_tmem, ad + a2, bd + b2, idesc, 1u);
                    umma_f16_pair_elect(d_tmem, ad + a3, bd + b3, idesc, 1u);
                    umma_commit_pair_elect(&empty[s], 0x3);  // frees stage s in both CTAs
                    acc = 1u;
                    if (++s == (uint32_t)S) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (two) {
                        const uint64_t ad2 = desc_add(a_desc0, s * Cfg::A_BYTES);
                        const bool packed = b_half_packed && s_first + 1 < (uint32_t)S;
                        const uint64_t bd2 =
                            packed ? desc_add(b_desc0, s_first * Cfg::B_BYTES + Cfg::B_BOX_BYTES)
                                   : desc_add(b_desc0, s * Cfg::B_BYTES);
                        if (!debug_check(p.fault_word,
                                         s < (uint32_t)S && (!packed || s == s_first + 1),
                                         kSiteSmemDesc, w.tile)) {
                            ok = false;
                            break;
                        }
                        umma_f16_pair_elect(d_tmem, ad2, bd2, idesc, 1u);
                        umma_f16_pair_elect(d_tmem, ad2 + a1, bd2 + b1, idesc, 1u);
                        umma_f16_pair_elect(d_tmem, ad2 + a2, bd2 + b2, idesc, 1u);
                        umma_f16_pair_elect(d_tmem, ad2 + a3, bd2 + b3, idesc, 1u);
                        umma_commit_pair_elect(&empty[s], 0x3);
                        if (++s == (uint32_t)S) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    kb += two ? 2 : 1;
                }
                if (!ok) break;
                umma_commit_pair_elect(&tfull[b], 0x3);  // accumulator b complete in both CTAs
            }
            // The elected lane's MMAs must finish before TMEM is released.
            umma_commit_pair_elect(drain, 0x1);
            mbar_wait(drain, 0, abort_flag, p.timeout_ns, true);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue warps 2-5 (both CTAs)
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int et = threadIdx.x - 64;
        uint8_t *warp_stage = smem + Cfg::OFF_STAGE + q * 2 * kEpiChunkBytes;
        uint32_t stage_seq = 0;
        const uint32_t tempty_cl0 = mapa_shared(smem_addr(&tempty[0]), 0);
        const uint32_t tempty_cl1 = mapa_shared(smem_addr(&tempty[1]), 0);
        uint64_t *cbar = cload + 2 * q;
        // beta != 0 with TMA stores: C is loaded through the staging buffers
        // (store_chunk_tma_cload).  (Also asking L2 for each unit's C while
        // its MMAs ran measured no different.)
        const bool cload_path = p.beta != 0.f && p.c_tma;
        uint32_t local = 0;
        for (int u = pair; u < p.num_units; u += npairs) {
            const Unit w = decode_unit<BN>(p, u);
            if (w.n0 >= p.N) continue;
            const uint32_t b = local & 1u, use = local >> 1;
            ++local;
            if (et == 0) {
                const bool ok = mbar_wait(&tfull[b], use & 1u, abort_flag, p.timeout_ns);
                if (!ok) record_fault(p, abort_flag, kRoleEpilogue, 0xff, w.tile);
                *epi_ok = ok ? 1 : 0;
            }
            named_bar_sync(TC_EPI_BAR, TC_EPI_THREADS);
            if (!*epi_ok) break;
            mbar_wait(&tfull[b], use & 1u, abort_flag, p.timeout_ns, true);  // completed: no wait
            tc_fence_after_sync();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + b * BN;
            const int gm = w.m_blk * 2 * TC_BM + (int)rank * TC_BM + row;
            void *cmat = c_matrix(p, w.bidx);
#pragma unroll 1
            for (int c = 0; c < w.width / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + c * 32, r);
                tmem_ld_wait();
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                if constexpr (EPI) apply_pre(p, w.n0 + c * 32, v);
                const float alpha = EPI ? 1.f : p.alpha;
                if (cload_path)
                    store_chunk_tma_cload<B3>(p, alpha, w.bidx, &tmC, warp_stage, cbar, stage_seq,
                                              lane, gm - lane, w.n0 + c * 32, v, abort_flag);
                else if (p.c_tma)
                    store_chunk_tma<B3>(p, alpha, cmat, w.bidx, &tmC, warp_stage, stage_seq, lane,
                                    gm - lane, w.n0 + c * 32, v);
                else
                    store_row_chunk(p, alpha, cmat, gm, w.n0 + c * 32, v);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(b ? tempty_cl1 : tempty_cl0);
        }
    }

    if (warp >= 2 && lane == 0) bulk_wait_all();  // TMA stores of C have landed
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // no remote arrive or pair MMA can still touch this CTA
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

// ================================================================ grouped
//
// One persistent launch over the output tiles of up to kMaxGroupsPerLaunch
// problems of different shapes and operands (the grouped GEMM that
// "Blackwell BF16 GEMM ..." (lshu.cn), section 3.1, lists among a GEMM
// library's capabilities).  Tile u of the launch belongs to the last
// problem whose first tile is <= u; within a problem, 128 x 256 tiles in
// grouped raster order.  Warp roles, ring, TMEM double buffering and the
// epilogue are those of the single-CTA kernel (whole tiles only: no split
// and no narrower tail tiles); every problem's A, B and C tensor maps travel
// in the kernel parameters.
struct BgGroup {
    int M, N, num_m_blk, num_n_blk, num_kb, tile0;
    float alpha, beta;
    void *C;
    long long ldc;
    int c_vec, c_tma;
};
struct BgParams {
    CUtensorMap ma[kMaxGroupsPerLaunch];
    CUtensorMap mb[kMaxGroupsPerLaunch];
    CUtensorMap mc[kMaxGroupsPerLaunch];
    BgGroup g[kMaxGroupsPerLaunch];
    int groups, units, c_f32;
    int stages, stage_bytes;
    unsigned long long *fault_word;
    unsigned long long timeout_ns;
    int fault_inject;
};
constexpr int kGroupedBN = 256;

// Problem of launch tile u (problems have at least one tile each, so their
// first tiles increase strictly), and the tile's block coordinates in it.
__device__ __forceinline__ int group_tile(const BgParams &p, int u, int &m_blk, int &n_blk) {
    int g = 0;
    for (int i = 1; i < p.groups; ++i)
        if (p.g[i].tile0 <= u) g = i;
    const BgGroup &d = p.g[g];
    grouped_tile_coords(u - d.tile0, d.num_m_blk, d.num_n_blk, kRasterGroup, m_blk, n_blk);
    return g;
}

template <bool A_MN, bool B_KM>
__global__ void __launch_bounds__(TC_THREADS, 1)
    bf16_tc_grouped_kernel(const __grid_constant__ BgParams p) {
    constexpr int BN = kGroupedBN;
    using Cfg = TcCfg<BN>;
    constexpr int SMAX = Cfg::MAX_STAGES;
    const uint32_t S = (uint32_t)p.stages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *ring = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::OFF_BAR);
    uint64_t *full = bars;
    uint64_t *empty = bars + SMAX;
    uint64_t *tfull = bars + 2 * SMAX;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + Cfg::OFF_MISC);
    uint32_t *tmem_slot = misc;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    volatile int *epi_ok = reinterpret_cast<volatile int *>(misc + 3);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int a_slot = Cfg::A_BYTES;  // 128 rows of A per stage, in either layout

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], TC_EPI_THREADS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *epi_ok = 0;
        fence_barrier_init();
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
            const uint32_t tx = (uint32_t)a_slot + (BN / 64) * Cfg::B_BOX_BYTES;
            uint32_t it = 0, s = 0, ph = 0;
            int withheld = -1;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
                int m_blk, n_blk;
                const int g = group_tile(p, u, m_blk, n_blk);
                const int m0 = m_blk * TC_BM, n0 = n_blk * BN;
                const int nkb = p.g[g].num_kb;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t cur = s, cur_ph = ph;
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (!mbar_wait(&empty[cur], cur_ph ^ 1u, abort_flag, p.timeout_ns)) {
                        record_fault_word(p.fault_word, abort_flag, kRoleProducer, cur, u);
                        ok = false;
                        break;
                    }
                    if (p.fault_inject && blockIdx.x == 0 && it == 0) {
                        withheld = 0;  // test hook: this stage is never filled
                        continue;
                    }
                    mbar_arrive_expect_tx(&full[cur], tx);
                    uint8_t *a_dst = ring + cur * (uint32_t)p.stage_bytes;
                    uint8_t *b_dst = a_dst + a_slot;
                    const int k0 = kb * TC_BK;
                    // Debug build: x coordinates a multiple of 8 bf16 elements,
                    // the group index inside the launch's table.
                    if (!debug_check(p.fault_word, g >= 0 && g < p.groups && cur < S &&
                                                       (A_MN ? m0 % 8 : k0 % 8) == 0,
                                     kSiteLoadA, u) ||
                        !debug_check(p.fault_word, (B_KM ? k0 % 8 : n0 % 8) == 0, kSiteLoadB,
                                     u))
                        continue;
                    if constexpr (A_MN) {
                        tma_load_2d(a_dst, &p.ma[g], &full[cur], m0, k0);
                        tma_load_2d(a_dst + 8192, &p.ma[g], &full[cur], m0 + 64, k0);
                    } else {
                        tma_load_2d(a_dst, &p.ma[g], &full[cur], k0, m0);
                    }
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j) {
                        if constexpr (B_KM)
                            tma_load_2d(b_dst + j * Cfg::B_BOX_BYTES, &p.mb[g], &full[cur], k0,
                                        n0 + j * 64);
                        else
                            tma_load_2d(b_dst + j * Cfg::B_BOX_BYTES, &p.mb[g], &full[cur],
                                        n0 + j * 64, k0);
                    }
                }
            }
            // Let every copy started here land before the CTA can exit.
            const uint32_t first = it > S ? it - S : 0u;
            for (uint32_t i = first; i < it; ++i) {
                if ((int)i == withheld) continue;
                mbar_wait(&full[i % S], (i / S) & 1u, abort_flag, p.timeout_ns, true);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (whole warp)
        const OperandLayout la = operand_layout(A_MN), lb = operand_layout(!B_KM);
        const uint64_t a_desc0 = smem_desc_sw128(smem_addr(ring), la.lbo, 1024);
        const uint64_t b_desc0 = smem_desc_sw128(smem_addr(ring + a_slot), lb.lbo, 1024);
        const uint32_t stage_bytes = (uint32_t)p.stage_bytes;
        const uint32_t a1 = la.step, a2 = 2 * la.step, a3 = 3 * la.step;
        const uint32_t b1 = lb.step, b2 = 2 * lb.step, b3 = 3 * lb.step;
        const uint32_t idesc = idesc_bf16_f32(BN, TC_BM, A_MN, B_KM);
        uint32_t s = 0, ph = 0, local = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < p.units; u += gridDim.x) {
            int m_blk, n_blk;
            const int g = group_tile(p, u, m_blk, n_blk);
            const int nkb = p.g[g].num_kb;
            const uint32_t b = local & 1u, use = local >> 1;
            ++local;
            const bool got = mbar_wait(&tempty[b], (use & 1u) ^ 1u, abort_flag, p.timeout_ns);
            if (__any_sync(0xffffffffu, !got)) {
                if (lane == 0) record_fault_word(p.fault_word, abort_flag, kRoleMma, 0xfe, u);
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + b * BN;
            if (!debug_check(p.fault_word, b * BN + BN <= Cfg::TMEM_COLS, kSiteTmem, u)) {
                ok = false;
                break;
            }
            uint32_t acc = 0;
            for (int kb = 0; kb < nkb; ++kb) {
                const bool ready = mbar_wait(&full[s], ph, abort_flag, p.timeout_ns);
                if (__any_sync(0xffffffffu, !ready)) {
                    if (lane == 0) record_fault_word(p.fault_word, abort_flag, kRoleMma, s, u);
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint64_t ad = desc_add(a_desc0, s * stage_bytes);
                const uint64_t bd = desc_add(b_desc0, s * stage_bytes);
                umma_f16_elect(d_tmem, ad, bd, idesc, acc);
                umma_f16_elect(d_tmem, ad + a1, bd + b1, idesc, 1u);
                umma_f16_elect(d_tmem, ad + a2, bd + b2, idesc, 1u);
                umma_f16_elect(d_tmem, ad + a3, bd + b3, idesc, 1u);
                umma_commit_elect(&empty[s]);  // frees the stage once these MMAs finish
                acc = 1u;
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            umma_commit_elect(&tfull[b]);  // accumulator b is complete
        }
        // The elected lane's MMAs must finish before TMEM is released.
        umma_commit_elect(drain);
        mbar_wait(drain, 0, abort_flag, p.timeout_ns, true);
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue warps 2-5
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        const int et = threadIdx.x - 64;
        uint8_t *warp_stage = smem + Cfg::OFF_STAGE + q * 2 * kEpiChunkBytes;
        uint32_t stage_seq = 0;
        uint32_t local = 0;
        for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
            int m_blk, n_blk;
            const int g = group_tile(p, u, m_blk, n_blk);
            const BgGroup &d = p.g[g];
            const uint32_t b = local & 1u, use = local >> 1;
            ++local;
            if (et == 0) {
                const bool ok = mbar_wait(&tfull[b], use & 1u, abort_flag, p.timeout_ns);
                if (!ok) record_fault_word(p.fault_word, abort_flag, kRoleEpilogue, 0xff, u);
                *epi_ok = ok ? 1 : 0;
            }
            named_bar_sync(TC_EPI_BAR, TC_EPI_THREADS);
            if (!*epi_ok) break;
            mbar_wait(&tfull[b], use & 1u, abort_flag, p.timeout_ns, true);  // completed: no wait
            tc_fence_after_sync();
            // The store helpers read these fields of a parameter block.
            TcParams tp{};
            tp.M = d.M;
            tp.N = d.N;
            tp.ldc = d.ldc;
            tp.beta = d.beta;
            tp.c_f32 = p.c_f32;
            tp.c_vec = d.c_vec;
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + b * BN;
            const int gm = m_blk * TC_BM + row;
            const int gn0 = n_blk * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + c * 32, r);
                tmem_ld_wait();
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                if (d.c_tma)
                    store_chunk_tma<false>(tp, d.alpha, d.C, 0, &p.mc[g], warp_stage, stage_seq,
                                           lane, gm - lane, gn0 + c * 32, v);
                else
                    store_row_chunk(tp, d.alpha, d.C, gm, gn0 + c * 32, v);
            }
            tc_fence_before_sync();
            mbar_arrive(&tempty[b]);
        }
    }

    if (warp >= 2 && lane == 0) bulk_wait_all();  // TMA stores of C have landed
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

// Tensor maps encoded on this thread, most recent first in no particular
// order: a map is plain data fixed by its arguments (base address, shape,
// strides, box, swizzle), so a call that repeats them reuses the encoded
// map instead of encoding it again (about a microsecond each).
struct MapEntry {
    bool used;
    CUtensorMapDataType dtype;
    cuuint32_t rank;
    const void *base;
    cuuint64_t dims[4];
    cuuint64_t strides[3];
    cuuint32_t box[4];
    CUtensorMapSwizzle swizzle;
    CUtensorMapL2promotion l2;
    CUtensorMap map;
};
constexpr int kMapCacheSize = 32;
thread_local MapEntry t_maps[kMapCacheSize];
thread_local int t_next_map = 0;

bool encode_cached(CUtensorMap *map, CUtensorMapDataType dtype, cuuint32_t rank, const void *base,
                   const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box,
                   CUtensorMapSwizzle swizzle, CUtensorMapL2promotion l2) {
    for (MapEntry &e : t_maps) {
        if (!e.used || e.base != base || e.dtype != dtype || e.rank != rank ||
            e.swizzle != swizzle || e.l2 != l2)
            continue;
        bool same = true;
        for (cuuint32_t i = 0; i < rank; ++i)
            same = same && e.dims[i] == dims[i] && e.box[i] == box[i] &&
                   (i + 1 == rank || e.strides[i] == strides[i]);
        if (same) {
            *map = e.map;
            return true;
        }
    }
    auto fn = encode_fn();
    if (!fn || rank > 4) return false;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (fn(map, dtype, rank, const_cast<void *>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
        return false;
    MapEntry &e = t_maps[t_next_map];
    t_next_map = (t_next_map + 1) % kMapCacheSize;
    e.used = true;
    e.dtype = dtype;
    e.rank = rank;
    e.base = base;
    e.swizzle = swizzle;
    e.l2 = l2;
    for (cuuint32_t i = 0; i < 4; ++i) {
        e.dims[i] = i < rank ? dims[i] : 0;
        e.box[i] = i < rank ? box[i] : 0;
    }
    for (cuuint32_t i = 0; i < 3; ++i) e.strides[i] = i + 1 < rank ? strides[i] : 0;
    e.map = *map;
    return true;
}

// 2-D bf16 tensor map over a row-major matrix: `inner` contiguous elements
// per row, `outer` rows, `pitch` elements between rows; box of
// box_inner x box_outer with 128-byte swizzle; out-of-range reads give 0.
bool make_map(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
              uint64_t pitch, uint32_t box_inner, uint32_t box_outer, uint64_t depth,
              uint64_t depth_stride) {
    return encode_tensor_map_3d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, inner, outer, depth,
                                pitch * 2, depth_stride * 2, box_inner, box_outer,
                                CU_TENSOR_MAP_SWIZZLE_128B);
}

// Tensor maps of the A and B operands in the layouts p.a_mn / p.b_kmaj
// select (see operand_layout): row-major A as 64 (K) x 128 (M) boxes,
// A stored K x M as 64 (M) x 64 (K) boxes; row-major B as 64 (N) x 64 (K)
// boxes, B stored N x K as 64 (K) x 64 (N) boxes.  Every box's x coordinate
// is a multiple of 64 elements (128 bytes).
bool make_ab_maps(CUtensorMap *ta, CUtensorMap *tb, const TcParams &p, const uint16_t *A,
                  int64_t lda, const uint16_t *B, int64_t ldb, const GemmOpts &o) {
    const uint64_t M = (uint64_t)p.M, N = (uint64_t)p.N, K = (uint64_t)p.K;
    // 2-D maps (depth 0) for one product; for a batch both are 3-D, an
    // operand shared by the whole batch with depth 1.
    const bool b3 = o.batch > 1;
    const uint64_t da = b3 ? (p.a_bmul ? (uint64_t)o.batch : 1) : 0;
    const uint64_t db = b3 ? (p.b_bmul ? (uint64_t)o.batch : 1) : 0;
    const uint64_t sa = (uint64_t)o.stride_a, sb = (uint64_t)o.stride_b;
    const bool ok_a = p.a_mn ? make_map(ta, A, M, K, (uint64_t)lda, 64, TC_BK, da, sa)
                             : make_map(ta, A, K, M, (uint64_t)lda, TC_BK, (uint32_t)p.a_rows,
                                        da, sa);
    const bool ok_b = p.b_kmaj ? make_map(tb, B, K, N, (uint64_t)ldb, TC_BK, 64, db, sb)
                               : make_map(tb, B, N, K, (uint64_t)ldb, 64, TC_BK, db, sb);
    return ok_a && ok_b;
}

// Exactly one of st (library-owned workspace, grown on demand) and ext
// (caller-provided scratch, never allocated) supplies the split-K storage.
// Tensor map for TMA stores of C (rows of N elements, pitch ldc): boxes of
// 32 x 32, swizzled as store_chunk_tma lays out its staging buffers.  Also
// decides p.c_tma: TMA stores need a 16-byte aligned C with a pitch that is
// a multiple of 16 bytes; otherwise the epilogue stores directly.
bool make_c_map(CUtensorMap *map, TcParams &p, int64_t batch) {
    const int esz = p.c_f32 ? 4 : 2;
    p.c_tma = ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0) && ((p.ldc * esz) % 16 == 0) &&
              ((p.c_bstride * esz) % 16 == 0);
    if (!p.c_tma) {
        memset(map, 0, sizeof(*map));
        return true;
    }
    const uint64_t depth = batch > 1 ? (uint64_t)batch : 1;
    const uint64_t dstride = (uint64_t)p.c_bstride * esz;
    const cuuint64_t dims[3] = {(cuuint64_t)p.N, (cuuint64_t)p.M, depth};
    const cuuint64_t strides[2] = {(cuuint64_t)p.ldc * esz, dstride};
    const cuuint32_t box[3] = {32, 32, 1};
    return encode_cached(map,
                         p.c_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         batch > 1 ? 3 : 2, p.C, dims, strides, box,
                         p.c_f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE);
}

// K-pair tensor maps of the CTA-pair kernel: boxes that span two
// consecutive 64-deep K blocks, so that one TMA copy fills an operand's part
// of two ring stages (stages s and s + 1 lie back to back in shared memory,
// and the box's outermost dimension walks the K blocks).  The K blocks
// become a dimension of their own, 128 bytes apart: a K-major operand (K
// contiguous) is viewed as 64 (k within the block) x rows x K/64 blocks, an
// MN-major one as 64 (m or n within a 64-wide chunk) x 64 (k) x chunks x
// K/64 blocks.  Such a view reads only inside the matrix when K is a
// multiple of 64 and, for an MN-major operand, M or N is too (a K-major
// view's rows past M or N are its own dimension's out-of-range rows, read as
// zeros like the 2-D maps' ones).  One product only (no batch).  Sets
// p.kpair when all three maps (A, B for whole tiles, B for column-half
// tiles) are encoded; otherwise the kernel copies one K block per box.  A whole tile's pair of stages then takes two copies per
// CTA instead of six, which shortens the producer's turn between a stage
// being freed and its refill (measured on GB300, N(0,1) data, L2 flushed:
// 4096^3 85.5 -> 82.7 us, 8192 x 14336 x 4096 508.6 -> 489.8 us, 8192^3
// 593.9 -> 579.7 us).
void make_kpair_maps(CUtensorMap *ta, CUtensorMap *tb, CUtensorMap *tbh, TcParams &p,
                     const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb) {
    p.kpair = 0;
    memset(ta, 0, sizeof(*ta));
    memset(tb, 0, sizeof(*tb));
    memset(tbh, 0, sizeof(*tbh));
    const uint64_t M = (uint64_t)p.M, N = (uint64_t)p.N, K = (uint64_t)p.K;
    if (K % 64 != 0 || (p.a_mn && M % 64 != 0) || (!p.b_kmaj && N % 64 != 0)) return;
    const uint64_t kb = K / 64, pa = (uint64_t)lda * 2, pb = (uint64_t)ldb * 2;
    const auto bf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
    const auto l2 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
    bool ok;
    if (p.a_mn) {  // A stored K x M: element (m, k) at k * lda + m
        const cuuint64_t dims[4] = {64, 64, M / 64, kb};
        const cuuint64_t str[3] = {pa, 128, 64 * pa};
        const cuuint32_t box[4] = {64, TC_BK, TC_BM / 64, 2};
        ok = encode_cached(ta, bf16, 4, A, dims, str, box, sw, l2);
    } else {  // row-major A: element (m, k) at m * lda + k
        const cuuint64_t dims[3] = {64, M, kb};
        const cuuint64_t str[2] = {pa, 128};
        const cuuint32_t box[3] = {TC_BK, TC_BM, 2};
        ok = encode_cached(ta, bf16, 3, A, dims, str, box, sw, l2);
    }
    // tb: this CTA's 128 B columns of a whole tile; tbh: its 64 columns of
    // a column-half tail tile.
    if (ok && p.b_kmaj) {  // B stored N x K: element (k, n) at n * ldb + k
        const cuuint64_t dims[3] = {64, N, kb};
        const cuuint64_t str[2] = {pb, 128};
        const cuuint32_t box[3] = {TC_BK, 128, 2};
        const cuuint32_t box_h[3] = {TC_BK, 64, 2};
        ok = encode_cached(tb, bf16, 3, B, dims, str, box, sw, l2) &&
             encode_cached(tbh, bf16, 3, B, dims, str, box_h, sw, l2);
    } else if (ok) {  // row-major B: element (k, n) at k * ldb + n
        const cuuint64_t dims[4] = {64, 64, N / 64, kb};
        const cuuint64_t str[3] = {pb, 128, 64 * pb};
        const cuuint32_t box[4] = {64, TC_BK, 2, 2};
        const cuuint32_t box_h[4] = {64, TC_BK, 1, 2};
        ok = encode_cached(tb, bf16, 4, B, dims, str, box, sw, l2) &&
             encode_cached(tbh, bf16, 4, B, dims, str, box_h, sw, l2);
    }
    if (ok) {
        p.kpair = 1;
    } else {
        memset(ta, 0, sizeof(*ta));
        memset(tb, 0, sizeof(*tb));
        memset(tbh, 0, sizeof(*tbh));
    }
}

template <int BN>
int launch_tc(int device, int sm_count, DeviceState *st, const ExternalScratch *ext,
              TcParams &p, const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
              const GemmOpts &o, cudaStream_t stream) {
    using Cfg = TcCfg<BN>;
    static PerDeviceOnce attrs;
    if (attrs.run(device, [] {
            const void *fns[4] = {(const void *)bf16_tc_kernel<BN, false, false>,
                                  (const void *)bf16_tc_kernel<BN, true, false>,
                                  (const void *)bf16_tc_kernel<BN, false, true>,
                                  (const void *)bf16_tc_kernel<BN, true, true>};
            for (const void *fn : fns)
                if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::SMEM_ALLOC) != cudaSuccess)
                    return 1;
            return 0;
        }) != 0)
        return GEMM_ERR_CUDA;
    alignas(64) CUtensorMap ta, tb, tc;
    if (!make_ab_maps(&ta, &tb, p, A, lda, B, ldb, o)) return GEMM_ERR_CUDA;
    if (!make_c_map(&tc, p, o.batch)) return GEMM_ERR_CUDA;

    p.num_m_blk = (p.M + TC_BM - 1) / TC_BM;
    p.num_n_blk = (p.N + BN - 1) / BN;
    p.num_kb = (p.K + TC_BK - 1) / TC_BK;
    const long long tiles_per_batch = (long long)p.num_m_blk * p.num_n_blk;
    const long long tiles = tiles_per_batch * o.batch;  // over the whole batch
    if (tiles > 0x7fffffffLL) return GEMM_ERR_TOO_LARGE;
    p.tiles_per_batch = (int)tiles_per_batch;
    int splits = 1;
    const RuntimeConfig cfg = runtime_config();
    p.stage_pairs = (int)cfg.stage_pairs;
    // Few tiles (at most half the SMs) and a long K: split K.  By default
    // into equal slices per tile (as many as keep the SMs busy); with
    // `stream_k` set, stream-K instead: all tiles * num_kb K iterations are
    // dealt out to P CTAs in equal contiguous ranges (P = SMs, at least 4
    // iterations each), so every SM streams the same number of operand
    // bytes whatever the tile count.  (Measured on GB300, 64 x 8192 x 8192:
    // equal slices 42 us, stream-K 46 us; its tiles are shared by up to
    // four CTAs and the extra partial tiles cost more than the balance
    // gains.)
    const bool small = tiles * 2 <= sm_count && p.num_kb >= 8;
    long long sk_ctas = 0;
    if (cfg.split_k > 0) {
        splits = (int)cfg.split_k;
    } else if (small && cfg.stream_k) {
        sk_ctas = std::min<long long>(sm_count, tiles * p.num_kb / 4);
    } else if (small) {
        splits = (int)(sm_count / tiles);
        if (splits > p.num_kb / 4) splits = p.num_kb / 4;
    }
    if (splits < 1) splits = 1;
    if (splits > p.num_kb) splits = p.num_kb;
    p.kb_per_split = (p.num_kb + splits - 1) / splits;
    p.splits = (p.num_kb + p.kb_per_split - 1) / p.kb_per_split;  // no empty slice
    if (tiles > 0x7fffffffLL) return GEMM_ERR_TOO_LARGE;
    // Raster band: 8 M-blocks when A and B fit in L2 together (concurrent
    // CTAs then share A and B blocks best); otherwise as many M-blocks as
    // keep the band's A panel (128 rows x K bf16 each) within about 32 MiB
    // of L2, so A is fetched from DRAM about once.  (Measured on GB300:
    // 4096^3 is fastest with 8; 8192 x 14336 x 4096 with 32.)
    {
        const long long panel = (long long)TC_BM * p.K * 2;
        const long long ab_bytes = 2ll * ((long long)p.M * p.K + (long long)p.K * p.N);
        long long g = (ab_bytes <= (80ll << 20)) ? 8 : (32ll << 20) / (panel > 0 ? panel : 1);
        if (g < 8) g = 8;
        if (cfg.raster_group > 0) g = cfg.raster_group;
        if (g > p.num_m_blk) g = p.num_m_blk;
        p.group_m = (int)g;
    }
    // Wave quantisation: with P persistent CTAs, tiles beyond the last full
    // wave are cut into 2 or 4 narrower sub-tiles when the partial wave
    // leaves at least that many SMs per tile idle.
    p.tiles_main = (int)tiles;
    p.tail_split = 1;
    if (p.splits == 1) {
        const long long P = sm_count;
        const long long rem = tiles % P;
        long long f = rem ? P / rem : 1;
        if (f > BN / 64) f = BN / 64;
        if (f >= 4) f = 4;
        else if (f >= 2) f = 2;
        else f = 1;
        if (cfg.tail_split_off) f = 1;
        if (f > 1) {
            p.tiles_main = (int)(tiles - rem);
            p.tail_split = (int)f;
        }
    }
    long long units = (p.splits > 1) ? tiles * p.splits
                                     : p.tiles_main + (tiles - p.tiles_main) * p.tail_split;
    p.stream_k = 0;
    p.max_parts = p.splits;
    if (sk_ctas > 1) {
        // Largest number of CTAs sharing one tile (each tile's first and
        // last iterations' owners, as the kernel computes them).
        const long long T = tiles * p.num_kb;
        long long mp = 1;
        for (long long t = 0; t < tiles; ++t) {
            const long long first = ((t * p.num_kb + 1) * sk_ctas - 1) / T;
            const long long last = ((t * p.num_kb + p.num_kb) * sk_ctas - 1) / T;
            mp = std::max(mp, last - first + 1);
        }
        p.stream_k = 1;
        p.max_parts = (int)mp;
        p.tiles_main = (int)tiles;
        p.tail_split = 1;
        units = tiles;  // the kernel deals out num_units * num_kb iterations
    }
    if (units > 0x7fffffffLL) return GEMM_ERR_TOO_LARGE;
    p.num_units = (int)units;
    p.ws = nullptr;
    p.counters = nullptr;
    p.ws_tiles = 0;
    if (p.splits > 1 || p.stream_k) {
        p.ws_tiles = (int)tiles;
        const size_t ws_bytes = (size_t)tiles * p.max_parts * TC_BM * BN * sizeof(float);
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
            Workspace *w = nullptr;
            const int rc = stream_workspace(st, stream, ws_bytes, (size_t)tiles, &w);
            if (rc != GEMM_OK) return rc;
            p.ws = w->ws;
            p.counters = w->counters;
        }
    }
    // Packed ring: the A rows this launch loads, then the B tile, per stage.
    p.a_slot = p.a_mn ? (p.a_rows > 64 ? 16384 : 8192) : p.a_rows * 128;
    p.stage_bytes = p.a_slot + Cfg::B_BYTES;
    p.stages = std::min(Cfg::MAX_STAGES, Cfg::RING_BYTES / p.stage_bytes);
    const int grid = p.stream_k ? (int)sk_ctas : (int)(units < sm_count ? units : sm_count);
    const int smem = Cfg::SMEM_ALLOC;
    if (o.batch > 1) {
        if (p.epi.on)
            bf16_tc_kernel<BN, true, true><<<grid, TC_THREADS, smem, stream>>>(ta, tb, tc, p);
        else
            bf16_tc_kernel<BN, false, true><<<grid, TC_THREADS, smem, stream>>>(ta, tb, tc, p);
    } else {
        if (p.epi.on)
            bf16_tc_kernel<BN, true, false><<<grid, TC_THREADS, smem, stream>>>(ta, tb, tc, p);
        else
            bf16_tc_kernel<BN, false, false><<<grid, TC_THREADS, smem, stream>>>(ta, tb, tc, p);
    }
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

cudaError_t query_resident_pairs(int *n);

// Largest number of CTA pairs that can be resident at once.  A pair must sit
// in one GPC, so this can be below sm_count / 2.
int max_resident_pairs(int device) {
    static PerDeviceOnce once;
    static int cache[kMaxDevices] = {};
    if (once.run(device, [device] {
            int n = 0;
            if (query_resident_pairs(&n) != cudaSuccess || n <= 0) return 1;
            cache[device] = n;
            return 0;
        }) != 0)
        return 0;
    return cache[device];
}

// Cluster occupancy of the CTA-pair kernel on the current device.
cudaError_t query_resident_pairs(int *n) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(2048, 1, 1);
    lc.blockDim = dim3(TC_THREADS, 1, 1);
    lc.dynamicSmemBytes = Tc2Cfg::SMEM_ALLOC;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(n, bf16_tc2_kernel<false, false>, &lc);
}

int launch_tc2(int device, TcParams &p, const uint16_t *A, int64_t lda, const uint16_t *B,
               int64_t ldb, const GemmOpts &o, cudaStream_t stream) {
    using Cfg = Tc2Cfg;
    static PerDeviceOnce attrs;
    if (attrs.run(device, [] {
            const void *fns[4] = {(const void *)bf16_tc2_kernel<false, false>,
                                  (const void *)bf16_tc2_kernel<true, false>,
                                  (const void *)bf16_tc2_kernel<false, true>,
                                  (const void *)bf16_tc2_kernel<true, true>};
            for (const void *fn : fns)
                if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::SMEM_ALLOC) != cudaSuccess)
                    return 1;
            return 0;
        }) != 0)
        return GEMM_ERR_CUDA;
    const RuntimeConfig cfg = runtime_config();
    p.stage_pairs = (int)cfg.stage_pairs;
    int pairs_max = max_resident_pairs(device);
    if (pairs_max <= 0) return GEMM_ERR_CUDA;
    if (cfg.pair_limit > 0 && cfg.pair_limit < pairs_max) pairs_max = (int)cfg.pair_limit;
    alignas(64) CUtensorMap ta, tb, tc, ta2, tb2, tbh;
    if (!make_ab_maps(&ta, &tb, p, A, lda, B, ldb, o)) return GEMM_ERR_CUDA;
    if (!make_c_map(&tc, p, o.batch)) return GEMM_ERR_CUDA;
    if (o.batch > 1 || cfg.kpair_maps_off || cfg.stage_pairs == 2) {
        p.kpair = 0;
        memset(&ta2, 0, sizeof(ta2));
        memset(&tb2, 0, sizeof(tb2));
        memset(&tbh, 0, sizeof(tbh));
    } else {
        make_kpair_maps(&ta2, &tb2, &tbh, p, A, lda, B, ldb);
    }
    p.num_m_blk = (p.M + 2 * TC_BM - 1) / (2 * TC_BM);  // 256-row pair tiles
    p.num_n_blk = (p.N + Cfg::BN - 1) / Cfg::BN;
    p.num_kb = (p.K + TC_BK - 1) / TC_BK;
    p.splits = 1;
    p.kb_per_split = p.num_kb;
    p.ws = nullptr;
    p.counters = nullptr;
    const long long tiles_per_batch = (long long)p.num_m_blk * p.num_n_blk;
    const long long tiles = tiles_per_batch * o.batch;  // over the whole batch
    if (tiles > 0x7fffffffLL) return GEMM_ERR_TOO_LARGE;
    p.tiles_per_batch = (int)tiles_per_batch;
    // Raster band in 256-row blocks: 1024 rows when A and B fit in L2
    // together, else a band whose A panel takes about 32 MiB of L2.
    {
        const long long ab_bytes = 2ll * ((long long)p.M * p.K + (long long)p.K * p.N);
        long long rows = (ab_bytes <= (80ll << 20)) ? 1024 : (32ll << 20) / ((long long)p.K * 2);
        long long g = rows / (2 * TC_BM);
        if (g < 4) g = 4;
        if (cfg.raster_group > 0) g = cfg.raster_group;
        if (g > p.num_m_blk) g = p.num_m_blk;
        p.group_m = (int)g;
    }
    // Partial last wave: cut its tiles into two 128-column halves when that
    // still leaves every half a pair of its own.  (Dealing the tail tiles'
    // K iterations out to all pairs instead, stream-K style, was measured
    // slower on GB300: 4096^3 94 us against 83 us.  The pieces' MMAs take
    // 8-12 us, but the last piece of each tile to arrive must read three
    // or four 128 KiB fp32 partials per CTA, and with the loads one SM keeps
    // in flight that takes 7-10 us.)
    p.tiles_main = (int)tiles;
    p.tail_split = 1;
    {
        const long long rem = tiles % pairs_max;
        if (rem && !cfg.tail_split_off && pairs_max / rem >= 2) {
            p.tiles_main = (int)(tiles - rem);
            p.tail_split = 2;
        }
    }
    const long long units = p.tiles_main + (tiles - p.tiles_main) * p.tail_split;
    if (units > 0x7fffffffLL) return GEMM_ERR_TOO_LARGE;
    p.num_units = (int)units;
    const int pairs = (int)(units < pairs_max ? units : pairs_max);

    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(2 * pairs, 1, 1);
    lc.blockDim = dim3(TC_THREADS, 1, 1);
    lc.dynamicSmemBytes = Cfg::SMEM_ALLOC;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    cudaError_t e;
    if (o.batch > 1)
        e = p.epi.on
                ? cudaLaunchKernelEx(&lc, bf16_tc2_kernel<true, true>, ta, tb, tc, ta2, tb2, tbh, p)
                : cudaLaunchKernelEx(&lc, bf16_tc2_kernel<false, true>, ta, tb, tc, ta2, tb2, tbh, p);
    else
        e = p.epi.on
                ? cudaLaunchKernelEx(&lc, bf16_tc2_kernel<true, false>, ta, tb, tc, ta2, tb2, tbh, p)
                : cudaLaunchKernelEx(&lc, bf16_tc2_kernel<false, false>, ta, tb, tc, ta2, tb2, tbh, p);
    if (e != cudaSuccess) return GEMM_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

// Grouped launch: the A, B and C tensor maps of each problem as the
// single-CTA kernel would encode them (128-row A boxes, 256-column tiles).
template <bool A_MN, bool B_KM>
int launch_grouped_layout(int device, int sm_count, BgParams &gp, cudaStream_t stream) {
    using Cfg = TcCfg<kGroupedBN>;
    static PerDeviceOnce attrs;
    if (attrs.run(device, [] {
            return cudaFuncSetAttribute(bf16_tc_grouped_kernel<A_MN, B_KM>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        Cfg::SMEM_ALLOC) == cudaSuccess
                       ? 0
                       : 1;
        }) != 0)
        return GEMM_ERR_CUDA;
    const int grid = gp.units < sm_count ? gp.units : sm_count;
    bf16_tc_grouped_kernel<A_MN, B_KM><<<grid, TC_THREADS, Cfg::SMEM_ALLOC, stream>>>(gp);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

int launch_grouped(int device, int sm_count, unsigned long long *fault_word, int count,
                   const GroupProblem *g, bool c_f32, int trans_a, int trans_b,
                   cudaStream_t stream) {
    using Cfg = TcCfg<kGroupedBN>;
    if (count < 1 || count > kMaxGroupsPerLaunch) return GEMM_ERR_INVALID_ARG;
    static_assert(sizeof(BgParams) <= 32000, "kernel parameter space");
    thread_local BgParams gp;  // about 28 KiB: kept off the stack
    long long tiles = 0;
    GemmOpts o{};
    o.trans_a = trans_a;
    o.trans_b = trans_b;
    for (int i = 0; i < count; ++i) {
        const GroupProblem &x = g[i];
        TcParams tp{};
        tp.M = (int)x.M;
        tp.N = (int)x.N;
        tp.K = (int)x.K;
        tp.a_mn = trans_a ? 1 : 0;
        tp.b_kmaj = trans_b ? 1 : 0;
        tp.a_rows = TC_BM;
        tp.C = x.C;
        tp.ldc = x.ldc;
        tp.c_f32 = c_f32 ? 1 : 0;
        if (!make_ab_maps(&gp.ma[i], &gp.mb[i], tp, static_cast<const uint16_t *>(x.A), x.lda,
                          static_cast<const uint16_t *>(x.B), x.ldb, o) ||
            !make_c_map(&gp.mc[i], tp, 1))
            return GEMM_ERR_CUDA;
        BgGroup &d = gp.g[i];
        d.M = tp.M;
        d.N = tp.N;
        d.num_m_blk = (tp.M + TC_BM - 1) / TC_BM;
        d.num_n_blk = (tp.N + kGroupedBN - 1) / kGroupedBN;
        d.num_kb = (tp.K + TC_BK - 1) / TC_BK;
        d.tile0 = (int)tiles;
        d.alpha = x.alpha;
        d.beta = x.beta;
        d.C = x.C;
        d.ldc = x.ldc;
        const int esz = c_f32 ? 4 : 2;
        d.c_vec = ((reinterpret_cast<uintptr_t>(x.C) & 15) == 0) && ((x.ldc * esz) % 16 == 0);
        d.c_tma = tp.c_tma;
        tiles += (long long)d.num_m_blk * d.num_n_blk;
        if (tiles > 0x7fffffffLL) return GEMM_ERR_TOO_LARGE;
    }
    gp.groups = count;
    gp.units = (int)tiles;
    gp.c_f32 = c_f32 ? 1 : 0;
    gp.stage_bytes = Cfg::A_BYTES + Cfg::B_BYTES;
    gp.stages = std::min(Cfg::MAX_STAGES, Cfg::RING_BYTES / gp.stage_bytes);
    gp.fault_word = fault_word;
    const RuntimeConfig cfg = runtime_config();
    gp.timeout_ns = (unsigned long long)cfg.watchdog_ms * 1000000ull;
    gp.fault_inject = cfg.fault_inject ? 1 : 0;
    if (gp.fault_inject) consume_fault_inject();
    if (!trans_a && !trans_b) return launch_grouped_layout<false, false>(device, sm_count, gp, stream);
    if (!trans_a) return launch_grouped_layout<false, true>(device, sm_count, gp, stream);
    if (!trans_b) return launch_grouped_layout<true, false>(device, sm_count, gp, stream);
    return launch_grouped_layout<true, true>(device, sm_count, gp, stream);
}

}  // namespace

namespace {

int launch_common(int device, int sm_count, DeviceState *st, const ExternalScratch *ext,
                  unsigned long long *fault_word, int M, int N, int K, float alpha,
                  const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb, float beta,
                  void *C, int64_t ldc, bool c_f32, const GemmOpts *opts, cudaStream_t stream) {
    TcParams p{};
    GemmOpts o = opts ? *opts : GemmOpts{};
    if (o.batch < 1) o.batch = 1;
    p.a_mn = o.trans_a ? 1 : 0;
    p.b_kmaj = o.trans_b ? 1 : 0;
    p.epi.bias = o.bias;
    p.epi.bias_f32 = o.bias_f32 ? 1 : 0;
    p.epi.act = o.act;
    p.epi.on = (o.bias != nullptr || o.act != 0) ? 1 : 0;
    p.a_bmul = (o.batch > 1 && o.stride_a != 0) ? 1 : 0;
    p.b_bmul = (o.batch > 1 && o.stride_b != 0) ? 1 : 0;
    p.c_bstride = o.batch > 1 ? o.stride_c : 0;
    p.M = M;
    p.N = N;
    p.K = K;
    p.alpha = alpha;
    p.beta = beta;
    p.C = C;
    p.ldc = ldc;
    p.c_f32 = c_f32 ? 1 : 0;
    const int esz = c_f32 ? 4 : 2;
    p.c_vec = ((reinterpret_cast<uintptr_t>(C) & 15) == 0) && ((ldc * esz) % 16 == 0) &&
              ((p.c_bstride * esz) % 16 == 0);
    p.fault_word = fault_word;
    const RuntimeConfig cfg = runtime_config();
    p.timeout_ns = (unsigned long long)cfg.watchdog_ms * 1000000ull;
    p.fault_inject = cfg.fault_inject ? 1 : 0;
    if (p.fault_inject) consume_fault_inject();
    int bn = (int)cfg.bf16_tile_n;
    if (bn != 128 && bn != 256) {
        bn = (N <= 128) ? 128 : 256;
        // When 256-wide tiles are too few for the SMs (the split-K regime),
        // 128-wide tiles need half as many K slices for the same parallelism:
        // less partial-sum traffic and a shorter reduction (measured on
        // GB300, 64 x 8192 x 8192 -> fp32, L2 flushed: 35.0 us against 38.8
        // us; 64 x 4096 x 14336: 33.2 against 43.1 us).
        const long long tiles256 =
            (long long)((M + TC_BM - 1) / TC_BM) * ((N + 255) / 256) * o.batch;
        if (bn == 256 && tiles256 * 2 <= sm_count && (K + TC_BK - 1) / TC_BK >= 8 &&
            cfg.split_k == 0)
            bn = 128;
    }
    // CTA pairs for problems with more than one 128-row block that give every
    // SM whole tiles; the single-CTA kernel (with split-K) for small or
    // short-and-deep problems.
    bool pair = false;
    if (cfg.cta_pair == 2) {
        pair = true;
    } else if (cfg.cta_pair == 0 && cfg.split_k == 0 && cfg.bf16_tile_n == 0 && M > TC_BM) {
        const long long tiles1 =
            (long long)((M + TC_BM - 1) / TC_BM) * ((N + 255) / 256) * o.batch;
        const int num_kb = (K + TC_BK - 1) / TC_BK;
        pair = !(tiles1 * 2 <= sm_count && num_kb >= 8);
    }
    p.a_rows = TC_BM;
    if (!pair && M <= TC_BM) p.a_rows = std::max(8, (M + 7) / 8 * 8);
    if (pair) return launch_tc2(device, p, A, lda, B, ldb, o, stream);
    return bn == 256 ? launch_tc<256>(device, sm_count, st, ext, p, A, lda, B, ldb, o, stream)
                     : launch_tc<128>(device, sm_count, st, ext, p, A, lda, B, ldb, o, stream);
}

}  // namespace

bool encode_tensor_map_3d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base,
                          uint64_t inner, uint64_t outer, uint64_t depth, uint64_t pitch_bytes,
                          uint64_t depth_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                          CUtensorMapSwizzle swizzle) {
    const cuuint32_t rank = depth == 0 ? 2 : 3;
    if (depth == 1)  // any valid stride: the third coordinate is always 0
        depth_stride_bytes = (pitch_bytes * (outer > 0 ? outer : 1) + 15) / 16 * 16;
    const cuuint64_t dims[3] = {inner, outer, depth};
    const cuuint64_t strides[2] = {pitch_bytes, depth_stride_bytes};
    const cuuint32_t box[3] = {box_inner, box_outer, 1};
    return encode_cached(map, dtype, rank, base, dims, strides, box, swizzle,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
}

int launch_bf16_tcgen05(DeviceState *st, int M, int N, int K, float alpha, const uint16_t *A,
                        int64_t lda, const uint16_t *B, int64_t ldb, float beta, void *C,
                        int64_t ldc, bool c_f32, const GemmOpts *opts, cudaStream_t stream) {
    return launch_common(st->device, st->sm_count, st, nullptr, st->fault_word, M, N, K, alpha,
                         A, lda, B, ldb, beta, C, ldc, c_f32, opts, stream);
}

int launch_bf16_tcgen05_external(int device, int sm_count, const ExternalScratch &ext, int M,
                                 int N, int K, float alpha, const uint16_t *A, int64_t lda,
                                 const uint16_t *B, int64_t ldb, float beta, void *C,
                                 int64_t ldc, bool c_f32, const GemmOpts *opts,
                                 cudaStream_t stream) {
    return launch_common(device, sm_count, nullptr, &ext, ext.fault_word, M, N, K, alpha, A, lda,
                         B, ldb, beta, C, ldc, c_f32, opts, stream);
}

int launch_bf16_tcgen05_grouped(DeviceState *st, int count, const GroupProblem *g, bool c_f32,
                                int trans_a, int trans_b, cudaStream_t stream) {
    return launch_grouped(st->device, st->sm_count, st->fault_word, count, g, c_f32, trans_a,
                          trans_b, stream);
}

}  // namespace gemm
