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
// RoPE rotates pair (x_2k, x_2k+1) of a d_r-vector by pos * base^(-2k/d_r)
// (the pages fix only that the angle grows with the position; pairing and
// frequencies are the common reading).  The angle and its sine and cosine
// are taken in fp64, so positions in the hundreds of thousands keep their
// phase.
//
// In bf16 mode the large weight-streaming products (W^DKV h, W^Q h) run on
// the tensor-core GEMM (gemm_bf16.cuh) into a scratch buffer; the kernels here
// add the d_r rows of W^KR, rotate, and scatter.  In fp32 mode the kernels
// here compute every row on CUDA cores.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "status.cuh"

namespace mla {
namespace pro {

constexpr int THREADS = 256;  // 8 warps
constexpr int TOK = 8;        // tokens per block
constexpr int ROWS = 8;       // weight rows (outputs) per block

// 16 bytes of T widened to fp32 (bf16 -> fp32 is exact: the bits move up).
__device__ __forceinline__ void widen(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void widen(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

template <typename T> struct Lanes;  // elements of T in 16 bytes
template <> struct Lanes<float> { static constexpr int N = 4; };
template <> struct Lanes<__nv_bfloat16> { static constexpr int N = 8; };

__device__ __forceinline__ void put(float* p, double v) { *p = (float)v; }
__device__ __forceinline__ void put(__nv_bfloat16* p, double v) { *p = __double2bfloat16(v); }

// Pair k of a d_r-vector (a, b) rotated at position pos, in fp64.
__device__ __forceinline__ void rope_pair(float a, float b, int k, int d_r, int64_t pos,
                                          double base, double& ya, double& yb) {
    const double theta = pow(base, -2.0 * k / (double)d_r);
    double sn, cs;
    sincos((double)pos * theta, &sn, &cs);
    ya = (double)a * cs - (double)b * sn;
    yb = (double)a * sn + (double)b * cs;
}

// tile[t][r] = sum_k W_r[k] * h_t[k] for the block's tokens t < nt and rows
// r < ROWS (wrow[r] == nullptr: row absent).  Thread j of the block takes the
// 16-byte chunks j, j + 256, ... of k for every token and row, so each
// weight chunk is read once and used for all eight tokens; the per-thread
// sums are reduced over the warp by shuffles and over the eight warps in
// shared memory.  Ends with the tile visible to the whole block.
template <typename T>
__device__ void dot_tile(const T* const (&wrow)[ROWS], const T* __restrict__ h0, int nt, int d,
                         float (*part)[ROWS * TOK], float (*tile)[ROWS]) {
    constexpr int V = Lanes<T>::N;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    float acc[ROWS][TOK];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
#pragma unroll
        for (int t = 0; t < TOK; ++t) acc[r][t] = 0.f;
    const int nv = d / V;
    for (int kv = threadIdx.x; kv < nv; kv += THREADS) {
        float hv[TOK][V];
#pragma unroll
        for (int t = 0; t < TOK; ++t) {
            const uint4 x = t < nt ? __ldg(reinterpret_cast<const uint4*>(h0 + (int64_t)t * d) + kv)
                                   : make_uint4(0u, 0u, 0u, 0u);
            widen(x, hv[t]);
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            if (wrow[r] == nullptr) continue;
            float wv[V];
            widen(__ldg(reinterpret_cast<const uint4*>(wrow[r]) + kv), wv);
#pragma unroll
            for (int t = 0; t < TOK; ++t)
#pragma unroll
                for (int v = 0; v < V; ++v) acc[r][t] = fmaf(wv[v], hv[t][v], acc[r][t]);
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
    const void* h;            // [N, d]
    const void* w_dkv;        // [d_c, d]
    const void* w_kr;         // [d_r, d]
    const void* c_tmp;        // bf16 mode: c = W^DKV h from the GEMM, [N, d_c]; else null
    const int32_t* seq_ids;   // [N]
    const int32_t* positions; // [N]
    const int32_t* page_table;  // [B, max_pages]
    void* pool;               // [num_pages, page, d_c + d_r]
    int N, d, d_c, d_r, B, page, max_pages;
    int64_t num_pages;
    int e_first;              // first row computed here: 0 (fp32) or d_c (bf16)
    double rope_base;
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

// Block (x, y): tokens 8x .. 8x+7, rows e_first + 8y .. +7 of [W^DKV ; W^KR].
// In bf16 mode the block also copies its share of the GEMM's c columns into
// the pool rows of its tokens.
template <typename T>
__global__ void __launch_bounds__(THREADS) kv_rows_kernel(const KvParams p) {
    __shared__ float part[THREADS / 32][ROWS * TOK];
    __shared__ float tile[TOK][ROWS];
    __shared__ T* rowp[TOK];
    __shared__ int stop;
    if (threadIdx.x == 0) stop = device_status_raised() ? 1 : 0;  // one decision for the block
    __syncthreads();
    if (stop) return;
    const int n0 = blockIdx.x * TOK, nt = min(TOK, p.N - n0);
    const int E = p.d_c + p.d_r;
    const int e0 = p.e_first + blockIdx.y * ROWS;
    if (threadIdx.x < TOK) rowp[threadIdx.x] = threadIdx.x < nt ? kv_row<T>(p, n0 + threadIdx.x) : nullptr;
    const T* wrow[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r) {
        const int e = e0 + r;
        wrow[r] = e >= E ? nullptr
                         : (e < p.d_c ? static_cast<const T*>(p.w_dkv) + (int64_t)e * p.d
                                      : static_cast<const T*>(p.w_kr) + (int64_t)(e - p.d_c) * p.d);
    }
    dot_tile<T>(wrow, static_cast<const T*>(p.h) + (int64_t)n0 * p.d, nt, p.d, part, tile);
    // rows of the tile: c as is, k^R rotated pair by pair (pairs never
    // straddle a tile: d_c and the tile start are even)
    if (threadIdx.x < ROWS * TOK) {
        const int t = threadIdx.x / ROWS, r = threadIdx.x % ROWS, e = e0 + r;
        T* row = t < nt ? rowp[t] : nullptr;
        if (row != nullptr && e < E) {
            if (e < p.d_c) {
                put(row + e, (double)tile[t][r]);
            } else if (((e - p.d_c) & 1) == 0) {
                double ya, yb;
                rope_pair(tile[t][r], tile[t][r + 1], (e - p.d_c) / 2, p.d_r,
                          p.positions[n0 + t], p.rope_base, ya, yb);
                put(row + e, ya);
                put(row + e + 1, yb);
            }
        }
    }
    if (p.c_tmp != nullptr) {  // bf16: this block's share of the 16-byte chunks of c
        const int per_row = p.d_c / Lanes<T>::N;
        const int share = (per_row + gridDim.y - 1) / gridDim.y;
        const int j0 = blockIdx.y * share, j1 = min(per_row, j0 + share);
        for (int idx = threadIdx.x; idx < nt * (j1 - j0); idx += THREADS) {
            const int t = idx / (j1 - j0), j = j0 + idx % (j1 - j0);
            T* row = rowp[t];
            if (row == nullptr) continue;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.c_tmp) +
                                                                (int64_t)(n0 + t) * p.d_c) + j);
            reinterpret_cast<uint4*>(row)[j] = v;
        }
    }
}

// ----------------------------------------------------------------- query

struct QParams {
    const void* h;            // [N, d]                      (fp32 path)
    const void* w_q;          // [H * (d_h + d_r), d]        (fp32 path)
    const void* q_tmp;        // [N, H * (d_h + d_r)] = W^Q h (bf16 path)
    const int32_t* positions; // [N]
    void* q_nope;             // [N, H, d_h]
    void* q_pe;               // [N, H, d_r]
    int N, d, H, d_h, d_r;
    double rope_base;
};

// Row e of W^Q h for token n goes to head e / (d_h + d_r): content part as
// is, RoPE part rotated (called for the even column of each pair).
template <typename T>
__device__ __forceinline__ void q_store(const QParams& p, int n, int e, float x, float x_next) {
    const int qw = p.d_h + p.d_r;
    const int i = e / qw, f = e % qw;
    const int64_t ni = (int64_t)n * p.H + i;
    if (f < p.d_h) {
        put(static_cast<T*>(p.q_nope) + ni * p.d_h + f, (double)x);
    } else if (((f - p.d_h) & 1) == 0) {
        double ya, yb;
        rope_pair(x, x_next, (f - p.d_h) / 2, p.d_r, p.positions[n], p.rope_base, ya, yb);
        T* dst = static_cast<T*>(p.q_pe) + ni * p.d_r + (f - p.d_h);
        put(dst, ya);
        put(dst + 1, yb);
    }
}

// fp32: block (x, y) computes rows 8y .. 8y+7 of W^Q h for tokens 8x .. 8x+7.
__global__ void __launch_bounds__(THREADS) q_rows_fp32_kernel(const QParams p) {
    __shared__ float part[THREADS / 32][ROWS * TOK];
    __shared__ float tile[TOK][ROWS];
    __shared__ int stop;
    if (threadIdx.x == 0) stop = device_status_raised() ? 1 : 0;  // one decision for the block
    __syncthreads();
    if (stop) return;
    const int n0 = blockIdx.x * TOK, nt = min(TOK, p.N - n0);
    const int M = p.H * (p.d_h + p.d_r);
    const int e0 = blockIdx.y * ROWS;
    const float* wrow[ROWS];
#pragma unroll
    for (int r = 0; r < ROWS; ++r)
        wrow[r] = e0 + r < M ? static_cast<const float*>(p.w_q) + (int64_t)(e0 + r) * p.d : nullptr;
    dot_tile<float>(wrow, static_cast<const float*>(p.h) + (int64_t)n0 * p.d, nt, p.d, part, tile);
    if (threadIdx.x < ROWS * TOK) {
        const int t = threadIdx.x / ROWS, r = threadIdx.x % ROWS;
        if (t < nt && e0 + r < M)
            q_store<float>(p, n0 + t, e0 + r, tile[t][r], r + 1 < ROWS ? tile[t][r + 1] : 0.f);
    }
}

// bf16: block n splits token n's row of W^Q h per head and rotates the RoPE
// parts.  The angle of pair k depends on the token's position only, so its
// sine and cosine are taken once per token (angle, sine and cosine in fp64,
// kept as fp32) and the rotations of all heads use them, in fp32.
__global__ void __launch_bounds__(THREADS) q_split_bf16_kernel(const QParams p) {
    extern __shared__ float rot[];  // [d_r / 2][cos, sin]
    __shared__ int stop;
    if (threadIdx.x == 0) stop = device_status_raised() ? 1 : 0;  // one decision for the block
    __syncthreads();
    if (stop) return;
    const int n = blockIdx.x;
    const int half = p.d_r / 2, qw = p.d_h + p.d_r;
    const int64_t pos = p.positions[n];
    for (int k = threadIdx.x; k < half; k += THREADS) {
        const double theta = pow(p.rope_base, -2.0 * k / (double)p.d_r);
        double sn, cs;
        sincos((double)pos * theta, &sn, &cs);
        rot[2 * k] = (float)cs;
        rot[2 * k + 1] = (float)sn;
    }
    __syncthreads();
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(p.q_tmp) + (int64_t)n * p.H * qw;
    const int nv = p.d_h / 8;  // 16-byte chunks of a head's content part
    uint4* nope = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.q_nope) + (int64_t)n * p.H * p.d_h);
    for (int idx = threadIdx.x; idx < p.H * nv; idx += THREADS) {
        const int i = idx / nv, v = idx % nv;
        nope[idx] = __ldg(reinterpret_cast<const uint4*>(src + (int64_t)i * qw) + v);
    }
    __nv_bfloat16* pe = static_cast<__nv_bfloat16*>(p.q_pe) + (int64_t)n * p.H * p.d_r;
    for (int idx = threadIdx.x; idx < p.H * half; idx += THREADS) {
        const int i = idx / half, k = idx % half;
        const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(src + (int64_t)i * qw + p.d_h + 2 * k);
        const float a = __low2float(x), b = __high2float(x);
        const float cs = rot[2 * k], sn = rot[2 * k + 1];
        *reinterpret_cast<__nv_bfloat162*>(pe + (int64_t)i * p.d_r + 2 * k) =
            __floats2bfloat162_rn(fmaf(a, cs, -b * sn), fmaf(a, sn, b * cs));
    }
}

}  // namespace pro
}  // namespace mla
