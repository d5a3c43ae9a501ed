// prologue.cuh -- the two steps that precede the absorbed decode of a new
// token h (one row of the model's hidden state):
//
//   cache write  c = W^DKV h,  k^R = RoPE(W^KR h, pos);  the row [c ; k^R]
//                is stored at the token's position in the paged latent pool
//   query        q = W^Q h, per head i the slice [q^C_i ; q^R_i], with q^R_i
//                rotated at the token's position
//
// ([Mishra] "Step 1: a low-rank latent": only c = W^DKV h is cached;
// "Step 4: decoupled RoPE": the positional part of a head comes from a
// separate small projection of h, is rotated, and for the key is one vector
// k^R shared by all heads; [llms] "Low-Rank Key-Value Joint Compression" and
// "The Positional Problem and Decoupled RoPE".)
//
// RoPE: pair (x_2k, x_2k+1) rotated by pos * base^(-2k/d_r), the angle
// taken in fixed-point turns without fp64 (rope.cuh).
//
// In bf16 mode the products W^DKV h, W^KR h and W^Q h run on the tensor-core
// GEMM (gemm_bf16.cuh).  For the cache write, and for a query projection with
// too few output tiles to fill the GPU, it leaves each K split's fp32 partial
// in the workspace, and the finishing kernels here add the splits, rotate,
// round once and scatter; a query projection whose tiles fill the GPU is
// written by the GEMM's own epilogue (OUT_QROPE).  In fp32 mode the kernels
// here compute every row on CUDA cores.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "pdl.cuh"
#include "rope.cuh"
#include "status.cuh"

namespace mla {
namespace pro {

constexpr int THREADS = 256;  // 8 warps
constexpr int TOK = 8;        // tokens per block (fp32 kernels)
constexpr int ROWS = 8;       // weight rows (outputs) per block (fp32 kernels)
constexpr int MAX_PAIRS = rope::MAX_PAIRS;  // d_r <= 128
constexpr int Q_HEADS = 4;    // heads per block of the bf16 query finish

// sum over the K splits, in split order, of the fp32 pair at src in each
// split's partials (split_stride floats apart).  The loads of up to
// SUM_BATCH splits are issued together: a split count in the tens would
// otherwise make this a chain of dependent L2 round trips.
constexpr int SUM_BATCH = 16;
__device__ __forceinline__ float2 sum_splits(const float* src, int64_t split_stride, int splits) {
    float a = 0.f, b = 0.f;
    for (int s0 = 0; s0 < splits; s0 += SUM_BATCH) {
        float2 v[SUM_BATCH];
#pragma unroll
        for (int k = 0; k < SUM_BATCH; ++k)
            v[k] = s0 + k < splits ? __ldcg(reinterpret_cast<const float2*>(src + (s0 + k) * split_stride))
                                   : make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < SUM_BATCH; ++k) {
            a += v[k].x;
            b += v[k].y;
        }
    }
    return make_float2(a, b);
}

using rope::rope_sincos;
using rope::rotate;

// 16 bytes of T widened to fp32 (bf16 -> fp32 is exact: the bits move up).
__device__ __forceinline__ void widen(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}

// tile[t][r] = sum_k W_r[k] * h_t[k] for the block's tokens t < nt and rows
// r < ROWS (wrow[r] == nullptr: row absent), fp32.  Thread j of the block
// takes the 16-byte chunks j, j + 256, ... of k for every token and row, so
// each weight chunk is read once and used for all eight tokens; the
// per-thread sums are reduced over the warp by shuffles and over the eight
// warps in shared memory.  Ends with the tile visible to the whole block.
__device__ void dot_tile(const float* const (&wrow)[ROWS], const float* __restrict__ h0, int nt, int d,
                         float (*part)[ROWS * TOK], float (*tile)[ROWS]) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    float acc[ROWS][TOK];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int t = 0; t < TOK; ++t) acc[r][t] = 0.f;
    const int nv = d / 4;
    for (int kv = threadIdx.x; kv < nv; kv += THREADS) {
        float hv[TOK][4];
#pragma unroll
        for (int t = 0; t < TOK; ++t) {
            const uint4 x = t < nt ? __ldg(reinterpret_cast<const uint4*>(h0 + (int64_t)t * d) + kv)
                                   : make_uint4(0u, 0u, 0u, 0u);
            widen(x, hv[t]);
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            if (wrow[r] == nullptr) continue;
            float wv[4];
            widen(__ldg(reinterpret_cast<const uint4*>(wrow[r]) + kv), wv);
#pragma unroll
            for (int t = 0; t < TOK; ++t)
#pragma unroll
                for (int v = 0; v < 4; ++v) acc[r][t] = fmaf(wv[v], hv[t][v], acc[r][t]);
        }
    }
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int t = 0; t < TOK; ++t) {
            float s = acc[r][t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) part[warp][r * TOK + t] = s;
        }
    __syncthreads();
    if (threadIdx.x < ROWS * TOK) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < THREADS / 32; ++w) s += part[w][threadIdx.x];  // fixed order
        tile[threadIdx.x % TOK][threadIdx.x / TOK] = s;
    }
    __syncthreads();
}

// ------------------------------------------------------------ cache write

struct KvParams {
    const void* h;            // [N, d]                  (fp32 path)
    const void* w_dkv;        // [d_c, d]                (fp32 path)
    const void* w_kr;         // [d_r, d]                (fp32 path)
    const float* parts;       // bf16 path: [splits][N][d_c + d_r] fp32 partials of [W^DKV ; W^KR] h
    int splits;
    const int32_t* seq_ids;   // [N]
    const int32_t* positions; // [N]
    const int32_t* page_table;  // [B, max_pages]
    void* pool;               // [num_pages, page, d_c + d_r]
    int N, d, d_c, d_r, B, page, max_pages;
    int64_t num_pages;
    uint64_t freq[MAX_PAIRS]; // RoPE frequencies as 0.64 fixed-point turns
};

// Pool row of token n, or null (and the status word raised) when its
// sequence, position or page id is out of range.
template <typename T>
__device__ __forceinline__ T* kv_row(const KvParams& p, int n) {
    const int s = p.seq_ids[n];
    const int64_t pos = p.positions[n];
    if (s < 0 || s >= p.B || pos < 0 || pos >= (int64_t)p.max_pages * p.page) {
        raise_device_status(MLA_DEV_BOUNDS, 0x30);
        return nullptr;
    }
    const int64_t pg = p.page_table[(int64_t)s * p.max_pages + pos / p.page];
    if (pg < 0 || pg >= p.num_pages) {
        raise_device_status(MLA_DEV_BOUNDS, 0x31);
        return nullptr;
    }
    return static_cast<T*>(p.pool) + (pg * p.page + pos % p.page) * (int64_t)(p.d_c + p.d_r);
}

// fp32: block (x, y) computes rows 8y .. 8y+7 of [W^DKV ; W^KR] h for
// tokens 8x .. 8x+7 and stores them, k^R rotated pair by pair (pairs never
// straddle a tile: d_c and the tile start are even).
__global__ void __launch_bounds__(THREADS) kv_rows_fp32_kernel(const KvParams p) {
    __shared__ float part[THREADS / 32][ROWS * TOK];
    __shared__ float tile[TOK][ROWS];
    __shared__ float* rowp[TOK];
    __shared__ int stop;
    if (threadIdx.x == 0) stop = device_status_raised() ? 1 : 0;  // one decision for the block
    __syncthreads();
    if (stop) return;
    const int n0 = blockIdx.x * TOK, nt = min(TOK, p.N - n0);
    const int E = p.d_c + p.d_r;
    const int e0 = blockIdx.y * ROWS;
    if (threadIdx.x < TOK) rowp[threadIdx.x] = threadIdx.x < nt ? kv_row<float>(p, n0 + threadIdx.x) : nullptr;
    const float* wrow[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const int e = e0 + r;
        wrow[r] = e >= E ? nullptr
                         : (e < p.d_c ? static_cast<const float*>(p.w_dkv) + (int64_t)e * p.d
                                      : static_cast<const float*>(p.w_kr) + (int64_t)(e - p.d_c) * p.d);
    }
    dot_tile(wrow, static_cast<const float*>(p.h) + (int64_t)n0 * p.d, nt, p.d, part, tile);
    if (threadIdx.x < ROWS * TOK) {
        const int t = threadIdx.x / ROWS, r = threadIdx.x % ROWS, e = e0 + r;
        float* row = t < nt ? rowp[t] : nullptr;
        if (row != nullptr && e < E) {
            if (e < p.d_c) {
                row[e] = tile[t][r];
            } else if (((e - p.d_c) & 1) == 0) {
                float sn, cs, ya, yb;
                rope_sincos(p.positions[n0 + t], p.freq[(e - p.d_c) / 2], sn, cs);
                rotate(tile[t][r], tile[t][r + 1], sn, cs, ya, yb);
                row[e] = ya;
                row[e + 1] = yb;
            }
        }
    }
}

// bf16: block n finishes token n's row: thread j takes the pair of columns
// (2j, 2j+1) of [c ; k^R], adds the K splits' partials in split order,
// rotates the pair when it belongs to k^R, rounds once to bf16 and stores
// it, so that the block writes the whole pool row in one pass.
__global__ void kv_finish_bf16_kernel(const KvParams p) {
    __shared__ __nv_bfloat16* row;
    const int n = blockIdx.x;
    const int E = p.d_c + p.d_r;
    const int e = 2 * (int)threadIdx.x;
    // The pool row and the rotation depend only on the call's inputs, which
    // are complete before the GEMM ahead lets this kernel launch (pdl.cuh):
    // look them up while the GEMM finishes, then wait for its partials.
    if (threadIdx.x == 0) row = kv_row<__nv_bfloat16>(p, n);
    float sn = 0.f, cs = 1.f;
    if (e >= p.d_c && e < E) rope_sincos(p.positions[n], p.freq[(e - p.d_c) / 2], sn, cs);
    grid_dep_wait();
    if (threadIdx.x == 0 && device_status_raised()) row = nullptr;
    __syncthreads();
    if (row == nullptr || e >= E) return;
    const float2 ab = sum_splits(p.parts + (int64_t)n * E + e, (int64_t)p.N * E, p.splits);
    float a = ab.x, b = ab.y;
    if (e >= p.d_c) rotate(a, b, sn, cs, a, b);
    *reinterpret_cast<__nv_bfloat162*>(row + e) = __floats2bfloat162_rn(a, b);
}

// ----------------------------------------------------------------- query

struct QParams {
    const void* h;            // [N, d]                      (fp32 path)
    const void* w_q;          // [H * (d_h + d_r), d]        (fp32 path)
    const float* parts;       // bf16 path: [splits][N][H * (d_h + d_r)] fp32 partials of W^Q h
    int splits;
    const int32_t* positions; // [N]
    void* q_nope;             // [N, H, d_h]
    void* q_pe;               // [N, H, d_r]
    int N, d, H, d_h, d_r;
    uint64_t freq[MAX_PAIRS];
};

// fp32: block (x, y) computes rows 8y .. 8y+7 of W^Q h for tokens 8x .. 8x+7;
// row e goes to head e / (d_h + d_r): content part as is, RoPE part rotated
// (pairs never straddle a tile: d_h, d_r and the tile start are even).
__global__ void __launch_bounds__(THREADS) q_rows_fp32_kernel(const QParams p) {
    __shared__ float part[THREADS / 32][ROWS * TOK];
    __shared__ float tile[TOK][ROWS];
    __shared__ int stop;
    if (threadIdx.x == 0) stop = device_status_raised() ? 1 : 0;  // one decision for the block
    __syncthreads();
    if (stop) return;
    const int n0 = blockIdx.x * TOK, nt = min(TOK, p.N - n0);
    const int qw = p.d_h + p.d_r;
    const int M = p.H * qw;
    const int e0 = blockIdx.y * ROWS;
    const float* wrow[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
        wrow[r] = e0 + r < M ? static_cast<const float*>(p.w_q) + (int64_t)(e0 + r) * p.d : nullptr;
    dot_tile(wrow, static_cast<const float*>(p.h) + (int64_t)n0 * p.d, nt, p.d, part, tile);
    if (threadIdx.x < ROWS * TOK) {
        const int t = threadIdx.x / ROWS, r = threadIdx.x % ROWS, e = e0 + r;
        if (t < nt && e < M) {
            const int n = n0 + t, i = e / qw, f = e % qw;
            const int64_t ni = (int64_t)n * p.H + i;
            if (f < p.d_h) {
                static_cast<float*>(p.q_nope)[ni * p.d_h + f] = tile[t][r];
            } else if (((f - p.d_h) & 1) == 0) {
                float sn, cs, ya, yb;
                rope_sincos(p.positions[n], p.freq[(f - p.d_h) / 2], sn, cs);
                rotate(tile[t][r], tile[t][r + 1], sn, cs, ya, yb);
                float* dst = static_cast<float*>(p.q_pe) + ni * p.d_r + (f - p.d_h);
                dst[0] = ya;
                dst[1] = yb;
            }
        }
    }
}

// bf16: block (n, y) finishes heads Q_HEADS*y .. +Q_HEADS-1 of token n:
// thread j takes one pair of a head's columns, adds the K splits' partials
// in split order, rotates the pair when it belongs to q^R, rounds once to
// bf16 and stores it to q_nope or q_pe.
__global__ void q_finish_bf16_kernel(const QParams p) {
    __shared__ int stop;
    grid_dep_wait();  // the GEMM's partials (launched as its dependent, pdl.cuh)
    if (threadIdx.x == 0) stop = device_status_raised() ? 1 : 0;
    __syncthreads();
    if (stop) return;
    const int qw = p.d_h + p.d_r, pairs = qw / 2;
    const int i = blockIdx.y * Q_HEADS + (int)threadIdx.x / pairs;
    const int f = 2 * ((int)threadIdx.x % pairs);
    if (i >= p.H) return;
    const int n = blockIdx.x;
    const int M = p.H * qw;
    const float2 ab = sum_splits(p.parts + (int64_t)n * M + (int64_t)i * qw + f, (int64_t)p.N * M, p.splits);
    float a = ab.x, b = ab.y;
    const int64_t ni = (int64_t)n * p.H + i;
    if (f < p.d_h) {
        *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.q_nope) + ni * p.d_h + f) =
            __floats2bfloat162_rn(a, b);
    } else {
        float sn, cs;
        rope_sincos(p.positions[n], p.freq[(f - p.d_h) / 2], sn, cs);
        rotate(a, b, sn, cs, a, b);
        *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(p.q_pe) + ni * p.d_r + (f - p.d_h)) =
            __floats2bfloat162_rn(a, b);
    }
}

}  // namespace pro
}  // namespace mla
