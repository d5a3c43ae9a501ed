// gemm_bf16.cuh -- persistent weight-streaming tcgen05 GEMM for the
// projections around the attention: W^UK^T q (mla_absorb_q), W^UV o and W^O v
// (mla_out_proj), the prologue's W^DKV h, W^KR h and W^Q h, the prefill
// expansion and output, and the merged-weight variants.
//
//     D_z[m, n] = sum_k A_z[m, k] * X_z[n, k]        (z = head, or 0)
//
// In decode the activations are a few dozen rows (B*T) while the weights are
// megabytes, so the weight's output dimension sits on the UMMA M axis (128
// TMEM lanes) and the activation rows on N ("swap AB").  A is read by TMA in
// 128 x 64 tiles, K-major or MN-major (W^UK, whose stored rows run along
// d_c); X is K-major, BN rows x 64 per stage.
//
// Work is cut into items (head z, N tile, K split, M unit of MT = 1 or 2
// M tiles), M unit fastest.  With MT = 2 the two A tiles of a stage share
// one X tile: the TMA unit issues about one 128-byte row per 3 cycles per
// SM (measured), so halving the X rows per A byte raises what one SM can
// stream.  One CTA per SM walks a contiguous range of items with one
// continuous TMA ring, so the copies of the next item start while the
// current one is still being multiplied, and the accumulator is
// double-buffered in TMEM so the epilogue of item i runs while the products
// of item i+1 are issued; the epilogue hands its TMEM buffer back as soon as
// the columns are in registers, before its stores.
//
// Roles (192 threads): warp 0 (one lane) issues TMA; warp 1 owns TMEM and
// issues UMMA from an elected lane; warps 2..5 run the epilogue, warp w
// reading TMEM lanes 32 (w % 4) .. +31.  The epilogue stages 64 accumulator
// columns at a time through shared memory, so that every global store is a
// 16-byte piece of a contiguous output row.
//
// Output modes: OUT_BF16 (no split: bf16 rows of D), OUT_REDUCE (split-K:
// each split's fp32 partial goes to the workspace, and the last CTA to finish
// a tile adds the splits in split order and writes bf16), OUT_PARTS (every
// split's fp32 partial to the workspace, added up by the caller's next
// kernel, which also applies its own epilogue), OUT_QROPE (no split: D is
// the stacked per-head query W^Q h; each row goes to its head's q^C or q^R,
// and the q^R pairs are rotated at their token's position before the one
// rounding to bf16).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "pdl.cuh"
#include "ptx.cuh"
#include "rope.cuh"
#include "status.cuh"
#include "tmem_batch.cuh"

namespace mla {
namespace gemm {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int MAX_STAGES = 8;
constexpr int THREADS = 192;
constexpr int EPI_WARP0 = 2;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB per stage
constexpr int EPI_COLS = 64;                    // accumulator columns staged per round
constexpr int STG_BYTES = EPI_COLS * BM * 4;    // 32 KB (fp32 rows of 128)
constexpr int CTL_BYTES = 256;                  // barriers, TMEM address, reducer flag
constexpr int FREQ_BYTES = rope::MAX_PAIRS * 8; // OUT_QROPE: the RoPE frequencies
constexpr int POS_BYTES = 256 * 4;              // OUT_QROPE: positions of an N tile's tokens
constexpr int ROPE_TABLE_MAX = 16 * 1024;       // OUT_QROPE: largest sin/cos table kept in shared memory
// shared memory besides the ring: 1 KB alignment slack, staging, control,
// frequencies, positions
constexpr int FIXED_SMEM = 1024 + STG_BYTES + CTL_BYTES + FREQ_BYTES + POS_BYTES;
static_assert((2 * MAX_STAGES + 5) * 8 + 8 <= CTL_BYTES, "barriers, TMEM address and flag fit");
constexpr uint32_t SMEM_CAP = 227 * 1024;

enum : int { OUT_BF16 = 0, OUT_REDUCE = 1, OUT_PARTS = 2, OUT_QROPE = 3 };

struct Params {
    int M;                // rows of D that exist (a multiple of 8; the last M tile may be partial)
    int N, K;             // columns of D; reduction length (a multiple of BK)
    int m_tiles;          // ceil(M / BM)
    int MT;               // M tiles per item (1, or 2 sharing each X tile)
    int m_units;          // m_tiles / MT
    int m_split;          // M tiles >= m_split load A from the second map, at row (mt - m_split) * BM
    int BN, n_tiles;      // N tile (multiple of 16, <= 256) and ceil(N / BN)
    int a_mn;             // A stored MN-major
    int x_batched;        // X has a head coordinate (z); else z = 0 for X
    int splits;           // K splits
    int chunks_per_split; // K chunks (of BK) per split; the last split may be shorter
    int items;            // Z * n_tiles * splits * m_units
    int stages;           // TMA ring depth, 1..MAX_STAGES
    int mode;             // OUT_BF16 / OUT_REDUCE / OUT_PARTS / OUT_QROPE
    int a_evict_first;    // A is read once (one N tile): let it leave L2 first
    int vec_out;          // out, ldo and out_z allow 16-byte stores
    __nv_bfloat16* out;   // out[(n0+n) * ldo + z * out_z + m]
    int64_t ldo, out_z;
    float* ws_part;       // [splits][Z][N][M] fp32 partials (OUT_REDUCE, OUT_PARTS)
    int* ws_count;        // [Z * n_tiles * m_tiles] arrival counters (OUT_REDUCE), zero between calls
    // OUT_QROPE: row m of D is row f = m % (d_h + d_r) of query head
    // i = m / (d_h + d_r); f < d_h goes to q_nope[n][i][f], the rest, pair
    // (f - d_h, f - d_h + 1) rotated at positions[n] with frequency
    // freq[(f - d_h) / 2] (rope.cuh), to q_pe[n][i][f - d_h].  d_h and d_r
    // are multiples of 8, so an 8-row piece of a tile lies in one part.
    __nv_bfloat16* q_nope;
    __nv_bfloat16* q_pe;
    const int32_t* positions;
    int q_heads, d_h, d_r;
    int rope_table;       // sin, cos of every (token, pair) of the N tile precomputed in shared memory
                          // (BN x d_r/2 float2 after the fixed area; the planner adds its bytes)
    uint64_t freq[rope::MAX_PAIRS];
};

struct Item {
    int z, nt, split, mt, kc0, kc1;  // mt: the item's first M tile
};

__device__ __forceinline__ Item decode_item(const Params& p, int item) {
    Item w;
    w.mt = (item % p.m_units) * p.MT;
    int r = item / p.m_units;
    w.split = r % p.splits;
    r /= p.splits;
    w.nt = r % p.n_tiles;
    w.z = r / p.n_tiles;
    w.kc0 = w.split * p.chunks_per_split;
    w.kc1 = min(p.K / BK, w.kc0 + p.chunks_per_split);
    return w;
}

// Named barrier of the four epilogue warps (barrier 0 is __syncthreads).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// The same barrier, returning whether v held in every epilogue thread.
__device__ __forceinline__ bool epi_sync_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// One M tile of an item's accumulator (TMEM columns 0..BN of `tacc`, this
// thread's lane quarter already added) to global memory: bf16 rows of `out`,
// this split's fp32 rows of the partials (fp32), or the query heads
// (OUT_QROPE, staged in fp32 so that the rotation precedes the rounding).
// Runs in the 128 epilogue
// threads (t = 0..127, row = t in the tile); 64 columns per round through
// `stg`.  When release != 0 the TMEM buffer is handed back (one arrival per
// warp on that barrier) as soon as the last round's columns are in
// registers.
template <bool QR>
__device__ __forceinline__ void store_tile(const Params& p, const Item& w, int mt, int Z, uint32_t tacc,
                                           uint8_t* stg, const uint64_t* freq, const int32_t* pos_s,
                                           const float2* tab, int t, bool fp32, uint32_t release) {
    const int m0 = mt * BM, n0 = w.nt * p.BN;
    const int n_valid = min(p.BN, p.N - n0);
    const int mv = min(BM, p.M - m0);
    float* stg_f = reinterpret_cast<float*>(stg);
    uint16_t* stg_h = reinterpret_cast<uint16_t*>(stg);
    constexpr bool qrope = QR;  // p.mode == OUT_QROPE
    const bool stage32 = fp32 || qrope;
    for (int c0 = 0; c0 < n_valid; c0 += EPI_COLS) {
        uint32_t r[64];
        const bool two = c0 + 32 < n_valid;
        tmem_ld32_nowait(tacc + (uint32_t)c0, r);
        if (two) tmem_ld32_nowait(tacc + (uint32_t)c0 + 32, r + 32);
        tmem_wait_ld();
        tmem_reg_fence(r, 64);
        if (release != 0 && c0 + EPI_COLS >= n_valid) {
            tc_fence_before();
            __syncwarp();
            if ((t & 31) == 0) mbar_arrive(release);
        }
        const int nj = two ? 64 : 32;
        if (stage32) {
#pragma unroll
            for (int j = 0; j < 64; ++j)
                if (j < nj) stg_f[j * BM + t] = __uint_as_float(r[j]);
        } else {
#pragma unroll
            for (int j = 0; j < 64; ++j)
                if (j < nj) {
                    const __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(r[j]));
                    stg_h[j * BM + t] = *reinterpret_cast<const uint16_t*>(&h);
                }
        }
        epi_sync();
        const int ncols = min(EPI_COLS, n_valid - c0);
        // Thread t always takes the same rows of the tile (a 16-byte piece
        // of 4 fp32 or 8 bf16 rows) and every 4th / 8th token column.  Each
        // batch of pieces is read from the staging rows first and then
        // stored, so that the stores issue back to back (one load, one
        // store per step ran ~3x slower).
        if (fp32) {
            constexpr int PIECES = EPI_COLS * 32 / BM;  // float4 pieces per thread and round
            const int m = (t & 31) * 4;
            float* base = p.ws_part + (((int64_t)w.split * Z + w.z) * p.N + n0 + c0) * p.M + m0 + m;
#pragma unroll
            for (int h = 0; h < PIECES; h += 8) {
                float4 v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int j = (t >> 5) + (h + k) * (BM / 32);
                    v[k] = j < ncols ? *reinterpret_cast<const float4*>(stg_f + j * BM + m)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                if (m < mv) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int j = (t >> 5) + (h + k) * (BM / 32);
                        if (j < ncols) *reinterpret_cast<float4*>(base + (int64_t)j * p.M) = v[k];
                    }
                }
            }
        } else if (qrope) {
            // The head, part and frequencies of the thread's 8 rows are fixed
            // for the tile; only the token changes.
            const int m = (t & 15) * 8;
            const int qw = p.d_h + p.d_r, row = m0 + m;
            const int i = row / qw, f = row - i * qw;
            const bool rot = f >= p.d_h;
            uint64_t fr[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) fr[k] = rot ? freq[(f - p.d_h) / 2 + k] : 0;
            __nv_bfloat16* dst0 = rot ? p.q_pe + (int64_t)i * p.d_r + (f - p.d_h) : p.q_nope + (int64_t)i * p.d_h + f;
            const int64_t tok_stride = (int64_t)p.q_heads * (rot ? p.d_r : p.d_h);
            if (p.rope_table) {
                // sin and cos from the N tile's table: the pieces are read,
                // rotated and packed first, then stored back to back
                constexpr int PIECES = EPI_COLS * 16 / BM;  // 8
                const int pairs = p.d_r / 2, k0 = rot ? (f - p.d_h) / 2 : 0;
                if (m < mv) {
                    uint4 packed[PIECES];
#pragma unroll
                    for (int k = 0; k < PIECES; ++k) {
                        const int j = (t >> 4) + k * (BM / 16);
                        if (j >= ncols) continue;
                        const float4 lo = *reinterpret_cast<const float4*>(stg_f + j * BM + m);
                        const float4 hi = *reinterpret_cast<const float4*>(stg_f + j * BM + m + 4);
                        float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                        if (rot) {
                            // (sn, cs) of pairs k0 .. k0+3: 32 bytes, 16-byte aligned (k0 % 4 == 0)
                            const float4* sc = reinterpret_cast<const float4*>(tab + (c0 + j) * pairs + k0);
                            const float4 a = sc[0], b = sc[1];
                            rope::rotate(v[0], v[1], a.x, a.y, v[0], v[1]);
                            rope::rotate(v[2], v[3], a.z, a.w, v[2], v[3]);
                            rope::rotate(v[4], v[5], b.x, b.y, v[4], v[5]);
                            rope::rotate(v[6], v[7], b.z, b.w, v[6], v[7]);
                        }
                        packed[k] = make_uint4(pack2_bf16(v[0], v[1]), pack2_bf16(v[2], v[3]),
                                               pack2_bf16(v[4], v[5]), pack2_bf16(v[6], v[7]));
                    }
#pragma unroll
                    for (int k = 0; k < PIECES; ++k) {
                        const int j = (t >> 4) + k * (BM / 16);
                        if (j < ncols)
                            *reinterpret_cast<uint4*>(dst0 + (int64_t)(n0 + c0 + j) * tok_stride) = packed[k];
                    }
                }
            } else if (m < mv) {
                // no table (large N tiles): one piece at a time, its angles
                // computed here (unrolled, that code slowed the whole kernel)
                for (int j = t >> 4; j < ncols; j += BM / 16) {
                    const float4 lo = *reinterpret_cast<const float4*>(stg_f + j * BM + m);
                    const float4 hi = *reinterpret_cast<const float4*>(stg_f + j * BM + m + 4);
                    float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                    if (rot) {
                        const int64_t pos = pos_s[c0 + j];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            float sn, cs;
                            rope::rope_sincos(pos, fr[q], sn, cs);
                            rope::rotate(v[2 * q], v[2 * q + 1], sn, cs, v[2 * q], v[2 * q + 1]);
                        }
                    }
                    *reinterpret_cast<uint4*>(dst0 + (int64_t)(n0 + c0 + j) * tok_stride) =
                        make_uint4(pack2_bf16(v[0], v[1]), pack2_bf16(v[2], v[3]), pack2_bf16(v[4], v[5]),
                                   pack2_bf16(v[6], v[7]));
                }
            }
        } else {
            constexpr int PIECES = EPI_COLS * 16 / BM;  // 8
            const int m = (t & 15) * 8;
            __nv_bfloat16* base = p.out + (int64_t)(n0 + c0) * p.ldo + (int64_t)w.z * p.out_z + m0 + m;
            uint4 v[PIECES];
#pragma unroll
            for (int k = 0; k < PIECES; ++k) {
                const int j = (t >> 4) + k * (BM / 16);
                v[k] = j < ncols ? *reinterpret_cast<const uint4*>(stg_h + j * BM + m) : make_uint4(0u, 0u, 0u, 0u);
            }
            if (m < mv) {
#pragma unroll
                for (int k = 0; k < PIECES; ++k) {
                    const int j = (t >> 4) + k * (BM / 16);
                    if (j >= ncols) continue;
                    __nv_bfloat16* dst = base + (int64_t)j * p.ldo;
                    if (p.vec_out) {
                        *reinterpret_cast<uint4*>(dst) = v[k];
                    } else {
                        const uint16_t* e = reinterpret_cast<const uint16_t*>(&v[k]);
#pragma unroll
                        for (int q = 0; q < 8; ++q) reinterpret_cast<uint16_t*>(dst)[q] = e[q];
                    }
                }
            }
        }
        epi_sync();  // the staging buffer is rewritten by the next round
    }
}

// The last CTA to finish a split tile adds every split's fp32 partial in
// split order and writes the bf16 tile (128 epilogue threads).
__device__ __forceinline__ void reduce_tile(const Params& p, const Item& w, int mt, int Z, int t) {
    const int m0 = mt * BM, n0 = w.nt * p.BN;
    const int n_valid = min(p.BN, p.N - n0);
    const int mv = min(BM, p.M - m0);
    const int64_t split_stride = (int64_t)Z * p.N * p.M;
    const float* src0 = p.ws_part + ((int64_t)w.z * p.N + n0) * p.M + m0;
    __nv_bfloat16* out0 = p.out + (int64_t)n0 * p.ldo + (int64_t)w.z * p.out_z + m0;
    const int total = n_valid * 32;  // float4 pieces of the tile
    for (int base = t; base < total; base += 4 * BM) {
        float4 acc[4];
        int64_t off[4];
        bool on[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = base + u * BM;
            const int j = idx >> 5, m = (idx & 31) * 4;
            on[u] = idx < total && m < mv;
            off[u] = (int64_t)j * p.M + m;
            acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll 2
        for (int s = 0; s < p.splits; ++s) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                v[u] = on[u] ? __ldcg(reinterpret_cast<const float4*>(src0 + s * split_stride + off[u]))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                acc[u].x += v[u].x;
                acc[u].y += v[u].y;
                acc[u].z += v[u].z;
                acc[u].w += v[u].w;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (!on[u]) continue;
            const int idx = base + u * BM;
            const int j = idx >> 5, m = (idx & 31) * 4;
            __nv_bfloat16* dst = out0 + (int64_t)j * p.ldo + m;
            const uint32_t lo = pack2_bf16(acc[u].x, acc[u].y), hi = pack2_bf16(acc[u].z, acc[u].w);
            if (p.vec_out) {
                *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
            } else {
                reinterpret_cast<uint16_t*>(dst)[0] = (uint16_t)lo;
                reinterpret_cast<uint16_t*>(dst)[1] = (uint16_t)(lo >> 16);
                reinterpret_cast<uint16_t*>(dst)[2] = (uint16_t)hi;
                reinterpret_cast<uint16_t*>(dst)[3] = (uint16_t)(hi >> 16);
            }
        }
    }
}

// MT (M tiles per item, 1 or 2) is a template parameter: with it known at
// compile time the product and copy issue loops unroll.  QR (the query
// output mode, OUT_QROPE) is one too, so that the other modes' kernels
// carry none of its code.
template <int MT, bool QR>
__global__ void __launch_bounds__(THREADS, 1)
wgemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_a2,
             const __grid_constant__ CUtensorMap tm_x, const Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t xb = (uint32_t)p.BN * BK * 2;
    const uint32_t a_all = (uint32_t)MT * A_BYTES;
    const uint32_t stage_bytes = a_all + xb;  // multiple of 1024 (BN % 16 == 0)
    const int S = p.stages;
    uint8_t* stg = smem + S * stage_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(stg + STG_BYTES);
    // bars: [0, S) full, [S, 2S) empty, 2S + b acc_full, 2S + 2 + b acc_empty, 2S + 4 final
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
    int* flag = reinterpret_cast<int*>(tmem_slot + 1);  // [0] this tile's reducer
    uint64_t* freq_s = reinterpret_cast<uint64_t*>(stg + STG_BYTES + CTL_BYTES);
    int32_t* pos_s = reinterpret_cast<int32_t*>(stg + STG_BYTES + CTL_BYTES + FREQ_BYTES);
    float2* tab_s = reinterpret_cast<float2*>(stg + STG_BYTES + CTL_BYTES + FREQ_BYTES + POS_BYTES);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int i0 = (int)((int64_t)p.items * blockIdx.x / gridDim.x);
    const int i1 = (int)((int64_t)p.items * (blockIdx.x + 1) / gridDim.x);
    const int Z = p.items / (p.n_tiles * p.splits * p.m_units);
    uint32_t acc_cols = 32;
    while (acc_cols < (uint32_t)(MT * p.BN)) acc_cols <<= 1;
    const uint32_t tmem_cols = 2 * acc_cols;

    poison_smem(smem, (uint32_t)S * stage_bytes + STG_BYTES);  // debug build: ring and staging
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const uint32_t accf0 = smem_u32(bars + 2 * S), acce0 = smem_u32(bars + 2 * S + 2);
    const uint32_t fin = smem_u32(bars + 2 * S + 4);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, 4);  // one arrival per epilogue warp
        }
        mbar_init(fin, 1);
        flag[0] = 0;
        // the frequencies in shared memory: the epilogue's threads index
        // them by row, which the constant bank would serialise
        if (QR)
            for (int k = 0; k < rope::MAX_PAIRS; ++k) freq_s[k] = p.freq[k];
        fence_mbar_init_cluster();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_a2);
        tma_prefetch_desc(&tm_x);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The kernel may have been launched before the one ahead of it on the
    // stream finished (pdl.cuh): the set-up above touched no global memory;
    // from here on every thread may.  The next kernel may launch now: it
    // waits the same way before it reads what this one writes.
    grid_dep_wait();
    if (threadIdx.x == 0) grid_dep_launch();
    // No read of the device status word here (a cold global load on every
    // CTA's critical path): when another kernel has raised it, the first
    // wait below that is not met at once gives up and the CTA winds down.

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol_a = p.a_evict_first ? l2_policy_evict_first() : l2_policy_evict_last();
            const uint64_t pol_x = l2_policy_evict_last();
            // the copies of one chunk into stage s: A (MT tiles), then X
            auto load_a = [&](const Item& w, int kc, int s) {
                const uint32_t sa = smem_u32(smem + s * stage_bytes);
#pragma unroll
                for (int j = 0; j < MT; ++j) {
                    const int mt = w.mt + j;
                    const bool second = mt >= p.m_split;
                    const CUtensorMap* am = second ? &tm_a2 : &tm_a;
                    const int m0 = (second ? mt - p.m_split : mt) * BM;
                    const uint32_t da = sa + j * A_BYTES;
                    if (p.a_mn) {
                        tma_load_3d(da, am, full0 + 8 * s, m0, kc * BK, w.z, pol_a);
                        tma_load_3d(da + A_BYTES / 2, am, full0 + 8 * s, m0 + 64, kc * BK, w.z, pol_a);
                    } else {
                        tma_load_3d(da, am, full0 + 8 * s, kc * BK, m0, w.z, pol_a);
                    }
                }
            };
            auto load_x = [&](const Item& w, int kc, int s) {
                const uint32_t sx = smem_u32(smem + s * stage_bytes) + a_all;
                tma_load_3d(sx, &tm_x, full0 + 8 * s, kc * BK, p.x_batched ? w.z : 0, w.nt * p.BN, pol_x);
            };
            // The chunks of the CTA's items in order, as (item, kc).
            int item = i0, kc = 0;
            Item w{};
            if (item < i1) {
                w = decode_item(p, item);
                kc = w.kc0;
            }
            auto next = [&]() {
                if (++kc >= w.kc1 && ++item < i1) {
                    w = decode_item(p, item);
                    kc = w.kc0;
                }
            };
            // debug build: every item of this CTA lies in the problem
            for (int i = i0; i < i1; ++i) {
                const Item c = decode_item(p, i);
                check_split(c.z < Z && c.nt < p.n_tiles && c.mt + MT <= p.m_tiles && c.kc0 < c.kc1 &&
                                c.kc1 <= p.K / BK && c.split < p.splits,
                            0x72);
            }
            int it = 0;
            for (; item < i1; ++it, next()) {
                const int s = it % S;
                if (!mbar_wait(empty0 + 8 * s, ((it / S) & 1) ^ 1, 0x101)) break;
                mbar_arrive_expect_tx(full0 + 8 * s, stage_bytes);
                load_a(w, kc, s);
                load_x(w, kc, s);
            }
            // every issued copy lands before the CTA can exit (on the normal
            // path these phases have completed; after an abort they may not)
            for (int i = max(0, it - S); i < it; ++i)
                mbar_wait_teardown(full0 + 8 * (i % S), (i / S) & 1, MLA_WAIT_LIMIT_NS);
        }
    } else if (warp == 1) {
        // --------------------------------------------------------------- MMA
        const uint32_t idesc = idesc_bf16(BM, p.BN, p.a_mn != 0, false);
        int it = 0, acc = 0;
        bool ok = true;
        for (int item = i0; item < i1 && ok; ++item, ++acc) {
            const Item w = decode_item(p, item);
            const uint32_t b = acc & 1, use = acc >> 1;
            ok = __all_sync(0xffffffffu, mbar_wait(acce0 + 8 * b, (use & 1) ^ 1, 0x102));
            if (!ok) break;
            tc_fence_after();
            const uint32_t d = tmem + b * acc_cols;
            for (int kc = w.kc0; kc < w.kc1; ++kc, ++it) {
                const int s = it % S;
                ok = __all_sync(0xffffffffu, mbar_wait(full0 + 8 * s, (it / S) & 1, 0x103));
                if (!ok) break;
                tc_fence_after();
                if (elect_one_sync()) {
                    const uint32_t sa = smem_u32(smem + s * stage_bytes);
                    const uint32_t sx = sa + a_all;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t dx = smem_desc(sx + kk * 32, 16, 1024, SWZ_128B);
#pragma unroll
                        for (int j = 0; j < MT; ++j) {
                            // A: K-major 128B-swizzled rows of 64 k, +32 B per 16-k step;
                            //    MN-major: two 64-m boxes 8 KB apart, 16 k-rows = 2 KB.
                            const uint32_t aj = sa + j * A_BYTES;
                            const uint64_t da = p.a_mn ? smem_desc(aj + kk * 2048, 8192, 1024, SWZ_128B)
                                                       : smem_desc(aj + kk * 32, 16, 1024, SWZ_128B);
                            mma_ss(d + j * p.BN, da, dx, idesc, (kc > w.kc0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    tc_commit(empty0 + 8 * s);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (elect_one_sync()) tc_commit(accf0 + 8 * b);
            __syncwarp();
        }
        // tracks every product issued, also on the abort path
        if (elect_one_sync()) tc_commit(fin);
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int t = q * 32 + lane;  // row of the tile this thread reads from TMEM
        bool ok = true;
        int acc = 0, pos_nt = -1;
        for (int item = i0; item < i1; ++item, ++acc) {
            const Item w = decode_item(p, item);
            const uint32_t b = acc & 1, use = acc >> 1;
            if (QR && w.nt != pos_nt) {
                // the N tile's token positions, read while the products run
                // (the previous item's stores, which read them, are done)
                pos_nt = w.nt;
                for (int j = t; j < p.BN; j += BM)
                    pos_s[j] = w.nt * p.BN + j < p.N ? __ldg(p.positions + w.nt * p.BN + j) : 0;
                if (p.rope_table) {
                    const int pairs = p.d_r / 2;
                    for (int e = t; e < p.BN * pairs; e += BM) {
                        const int j = e / pairs, n = w.nt * p.BN + j;
                        float sn = 0.f, cs = 1.f;
                        if (n < p.N) rope::rope_sincos(__ldg(p.positions + n), freq_s[e - j * pairs], sn, cs);
                        tab_s[e] = make_float2(sn, cs);
                    }
                }
            }
            bool good = ok && __all_sync(0xffffffffu, mbar_wait(accf0 + 8 * b, use & 1, 0x104));
            good = epi_sync_and(good);
            ok = good;
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < MT; ++j) {
                const int mt = w.mt + j;
                // the last tile's final TMEM read hands the buffer back
                if (good)
                    store_tile<QR>(p, w, mt, Z, tmem + b * acc_cols + (uint32_t)(j * p.BN) + ((uint32_t)(q * 32) << 16),
                               stg, freq_s, pos_s, tab_s, t, p.mode == OUT_REDUCE || p.mode == OUT_PARTS,
                               j == MT - 1 ? acce0 + 8 * b : 0u);
                if (p.mode == OUT_REDUCE) {
                    // Every CTA of a split tile arrives on its counter -- also
                    // one that gave up -- and the last arrival resets it, so
                    // the counters are back at zero for the next call whatever
                    // happened in this one.  Only a last arrival that sees no
                    // error anywhere reduces.
                    __threadfence();
                    epi_sync();
                    if (t == 0) {
                        const int tile = (w.z * p.n_tiles + w.nt) * p.m_tiles + mt;
                        const int prev = atomicAdd(p.ws_count + tile, 1);
                        const bool last = prev == p.splits - 1;
                        if (last) p.ws_count[tile] = 0;
                        flag[0] = last && good && !device_status_raised() ? 1 : 0;
                    }
                    epi_sync();
                    if (flag[0]) {
                        __threadfence();
                        reduce_tile(p, w, mt, Z, t);
                    }
                }
            }
        }
    }

    // the products (and their commits) are done before TMEM goes away, even
    // when the epilogue gave up waiting for them
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        mbar_wait_teardown(fin, 0, MLA_WAIT_LIMIT_NS);
        __syncwarp();
        tmem_dealloc(tmem, tmem_cols);
    }
}

}  // namespace gemm
}  // namespace mla
