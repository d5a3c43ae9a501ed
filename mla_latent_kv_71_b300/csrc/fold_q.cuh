// fold_q.cuh -- helpers of the query-side weight merge: W^UK_i^T W^UQ_i
// folded ahead of time into one weight per head ([Mishra] "Multi-head
// Latent Attention": the up-projections can be folded once, offline;
// [Zhang] "Matrix absorption: compression that also saves compute").
//
//   uq_transpose_kernel   W^UQ_i (the content rows of each head's block of
//                         W^Q) -> [d_q, H, d_h], so that the fold is the query
//                         absorption with the rows of W^UQ^T in the place of
//                         q^C
//   q_merged_fp32_kernel  q_lat[r, m] = sum_k W_merged[k, m] c^Q[r, k] on CUDA
//                         cores (the fp32 mode of the merged projection; the
//                         bf16 mode is a tensor-core GEMM)
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "status.cuh"

namespace mla {
namespace foldq {

constexpr int TT = 32;  // transpose tile

// out[k][i][e] = w_q[(i * (d_h + d_r) + e) * d_q + k] for e < d_h: 32 x 32
// tiles through shared memory (coalesced on both sides).  grid (ceil(d_q /
// 32), ceil(H * d_h / 32)), 32 x 8 threads.
template <typename T>
__global__ void uq_transpose_kernel(const T* __restrict__ w_q, T* __restrict__ out, int H, int d_h,
                                    int d_r, int d_q) {
    if (device_status_raised()) return;
    __shared__ T tile[TT][TT + 1];
    const int k0 = blockIdx.x * TT, r0 = blockIdx.y * TT;  // r = i * d_h + e (content rows only)
    for (int y = threadIdx.y; y < TT; y += blockDim.y) {
        const int r = r0 + y, k = k0 + threadIdx.x;
        if (r < H * d_h && k < d_q) {
            const int i = r / d_h, e = r % d_h;
            tile[y][threadIdx.x] = w_q[((int64_t)i * (d_h + d_r) + e) * d_q + k];
        }
    }
    __syncthreads();
    for (int y = threadIdx.y; y < TT; y += blockDim.y) {
        const int k = k0 + y, r = r0 + threadIdx.x;
        if (r < H * d_h && k < d_q) out[(int64_t)k * H * d_h + r] = tile[threadIdx.x][y];
    }
}

// One thread per output element, consecutive threads on consecutive m (the
// weight rows are read coalesced, c^Q broadcast).  grid (ceil(M / 128), rows).
__global__ void q_merged_fp32_kernel(const float* __restrict__ cq, const float* __restrict__ w,
                                     float* __restrict__ q_lat, int M, int d_q) {
    if (device_status_raised()) return;
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    const int r = blockIdx.y;
    if (m >= M) return;
    const float* x = cq + (int64_t)r * d_q;
    float acc = 0.f;
    for (int k = 0; k < d_q; ++k) acc = fmaf(w[(int64_t)k * M + m], x[k], acc);
    q_lat[(int64_t)r * M + m] = acc;
}

}  // namespace foldq
}  // namespace mla
