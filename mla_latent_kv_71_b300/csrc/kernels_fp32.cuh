// kernels_fp32.cuh -- fp32 kernels on CUDA cores (dtype MLA_FP32) and the
// log-sum-exp combine used by both dtypes.
//
// The fp32 mode computes the same decode step in fp32 arithmetic: absorbed
// query (W^UK^T q), scores of the absorbed query against the cached latent
// plus the decoupled RoPE term, softmax over the cached positions, the
// latent-weighted sum, then W^UV and W^O.  (Pages: [llms] "Query Key
// Absorption", "Value Output Absorption"; [Zhang] "Decoupled RoPE",
// "Value absorption".)  It serves small models whose widths the bf16
// tensor-core kernels do not cover and runs at CUDA-core speed.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "status.cuh"

namespace mla {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Visible cached positions of query t (of T) in a sequence of length len.
__device__ __forceinline__ int64_t visible_len(int64_t len, int T, int t, int causal) {
    int64_t n = causal ? len - (T - 1 - t) : len;
    return n < 0 ? 0 : n;
}

// ------------------------------------------------------------ fp32 absorb

// q_lat[r,i,c] = sum_e q_nope[r,i,e] * w_uk[i,e,c]; one thread per (r,i,c).
__global__ void absorb_q_fp32_kernel(const float* __restrict__ q_nope,
                                     const float* __restrict__ w_uk, float* __restrict__ q_lat,
                                     int rows, int H, int d_h, int d_c) {
    if (device_status_raised()) return;
    const int ri = blockIdx.x;  // r * H + i
    const int i = ri % H;
    const int c = blockIdx.y * blockDim.x + threadIdx.x;
    if (c >= d_c) return;
    const float* q = q_nope + (int64_t)ri * d_h;
    const float* w = w_uk + (int64_t)i * d_h * d_c + c;
    float acc = 0.f;
    for (int e = 0; e < d_h; ++e) acc = fmaf(q[e], w[(int64_t)e * d_c], acc);
    q_lat[(int64_t)ri * d_c + c] = acc;
}

// -------------------------------------------------------- fp32 out_proj

// v[r, i*d_h + e] = sum_c w_uv[i,e,c] * o[r,i,c]; one warp per (r,i,e).
__global__ void out_proj_v_fp32_kernel(const float* __restrict__ o, const float* __restrict__ w_uv,
                                       float* __restrict__ v, int rows, int H, int d_h,
                                       int d_c) {
    if (device_status_raised()) return;
    const int64_t gw = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (gw >= (int64_t)rows * H * d_h) return;
    const int e = (int)(gw % d_h);
    const int64_t ri = gw / d_h;  // r * H + i
    const int i = (int)(ri % H);
    const float* orow = o + ri * d_c;
    const float* wrow = w_uv + ((int64_t)i * d_h + e) * d_c;
    float acc = 0.f;
    for (int c = lane; c < d_c; c += 32) acc = fmaf(wrow[c], orow[c], acc);
    acc = warp_sum(acc);
    if (lane == 0) v[gw] = acc;
}

// out[r, n] = sum_k w_o[n, k] * v[r, k]; one warp per (r, n).
__global__ void out_proj_o_fp32_kernel(const float* __restrict__ v, const float* __restrict__ w_o,
                                       float* __restrict__ out, int rows, int K, int d) {
    if (device_status_raised()) return;
    const int64_t gw = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (gw >= (int64_t)rows * d) return;
    const int n = (int)(gw % d);
    const int64_t r = gw / d;
    const float* vrow = v + r * K;
    const float* wrow = w_o + (int64_t)n * K;
    float acc = 0.f;
    for (int k = lane; k < K; k += 32) acc = fmaf(wrow[k], vrow[k], acc);
    acc = warp_sum(acc);
    if (lane == 0) out[r * d + n] = acc;
}

// ---------------------------------------------------------- fp32 decode

constexpr int FP32_MAX_DC = 512;
constexpr int FP32_MAX_DR = 64;
constexpr int FP32_WARPS = 4;

// One block per (b*T + t, head).  Each warp walks every 4th visible position
// with an online softmax (running maximum and sum); the four warp states are
// merged at the end.  Scores: lanes split the d_c + d_r features, then a
// warp reduction.
__global__ void __launch_bounds__(FP32_WARPS * 32)
decode_fp32_kernel(const float* __restrict__ q_lat, const float* __restrict__ q_pe,
                   const float* __restrict__ pool, const int32_t* __restrict__ page_table,
                   const int32_t* __restrict__ seq_lens, int T, int H, int d_c, int d_r,
                   int page, int max_pages, int64_t num_pages, float scale, int causal,
                   float* __restrict__ o, float* __restrict__ lse) {
    __shared__ float q[FP32_MAX_DC + FP32_MAX_DR];
    __shared__ float wm[FP32_WARPS], wl[FP32_WARPS];
    __shared__ float wo[FP32_WARPS][FP32_MAX_DC];
    if (device_status_raised()) return;
    const int bt = blockIdx.x;
    const int i = blockIdx.y;
    const int b = bt / T, t = bt % T;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int width = d_c + d_r;
    const int64_t qrow = (int64_t)bt * H + i;
    for (int f = threadIdx.x; f < width; f += blockDim.x)
        q[f] = f < d_c ? q_lat[qrow * d_c + f] : q_pe[qrow * d_r + (f - d_c)];
    int64_t len = seq_lens[b];
    if (len < 0 || len > (int64_t)max_pages * page) {
        raise_device_status(MLA_DEV_BOUNDS, 1);
        len = len < 0 ? 0 : (int64_t)max_pages * page;
    }
    const int64_t n = visible_len(len, T, t, causal);
    __syncthreads();

    constexpr int PER_LANE = FP32_MAX_DC / 32;
    float acc[PER_LANE];
#pragma unroll
    for (int k = 0; k < PER_LANE; ++k) acc[k] = 0.f;
    float m = -INFINITY, l = 0.f;
    for (int64_t j = warp; j < n; j += FP32_WARPS) {
        int64_t pg = page_table[(int64_t)b * max_pages + j / page];
        if (pg < 0 || pg >= num_pages) {
            raise_device_status(MLA_DEV_BOUNDS, 2);
            continue;
        }
        const float* row = pool + (pg * page + j % page) * width;
        float part = 0.f;
        for (int f = lane; f < width; f += 32) part = fmaf(q[f], row[f], part);
        const float s = warp_sum(part) * scale;
        const float m_new = fmaxf(m, s);
        const float alpha = expf(m - m_new);
        const float p = expf(s - m_new);
        l = l * alpha + p;
#pragma unroll
        for (int k = 0; k < PER_LANE; ++k) {
            const int c = lane + 32 * k;
            const float cv = c < d_c ? row[c] : 0.f;
            acc[k] = fmaf(acc[k], alpha, p * cv);
        }
        m = m_new;
    }
    if (lane == 0) {
        wm[warp] = m;
        wl[warp] = l;
    }
#pragma unroll
    for (int k = 0; k < PER_LANE; ++k) {
        const int c = lane + 32 * k;
        if (c < d_c) wo[warp][c] = acc[k];
    }
    __syncthreads();
    float M = -INFINITY;
    for (int w = 0; w < FP32_WARPS; ++w) M = fmaxf(M, wm[w]);
    float L = 0.f;
    if (M != -INFINITY)
        for (int w = 0; w < FP32_WARPS; ++w) L += wl[w] * expf(wm[w] - M);
    for (int c = threadIdx.x; c < d_c; c += blockDim.x) {
        float v = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < FP32_WARPS; ++w) v += wo[w][c] * expf(wm[w] - M);
            v /= L;
        }
        o[qrow * d_c + c] = v;
    }
    if (threadIdx.x == 0) lse[qrow] = (M == -INFINITY) ? -INFINITY : M + logf(L);
}

// --------------------------------------------------------------- combine

// Merge S pieces of softmax rows: o_part [S, rows, d_c], lse_part [S, rows].
// One warp per row; lanes take float4 chunks of the row.
template <typename OutT>
__global__ void combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                               int S, int64_t rows, int d_c, OutT* __restrict__ o,
                               float* __restrict__ lse) {
    if (device_status_raised()) return;
    const int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (r >= rows) return;
    float m = -INFINITY;
    for (int s = 0; s < S; ++s) m = fmaxf(m, lse_part[(int64_t)s * rows + r]);
    float L = -INFINITY;
    if (m != -INFINITY) {
        float sum = 0.f;
        for (int s = 0; s < S; ++s) sum += expf(lse_part[(int64_t)s * rows + r] - m);
        L = m + logf(sum);
    }
    for (int c = 4 * lane; c < d_c; c += 128) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (L != -INFINITY) {
            for (int s = 0; s < S; ++s) {
                const float w = expf(lse_part[(int64_t)s * rows + r] - L);
                if (w == 0.f) continue;
                const float4 v =
                    *reinterpret_cast<const float4*>(o_part + ((int64_t)s * rows + r) * d_c + c);
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
            }
        }
        OutT* dst = o + r * d_c + c;
        if constexpr (sizeof(OutT) == 4) {
            *reinterpret_cast<float4*>(dst) = acc;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(dst) = pk;
        }
    }
    if (lane == 0) lse[r] = L;
}

}  // namespace mla
