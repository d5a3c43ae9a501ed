// gemm_bf16.cuh -- weight-streaming tcgen05 GEMM for the projections around
// the absorbed decode: W^UK^T q (mla_absorb_q), W^UV o and W^O v
// (mla_out_proj).
//
// In decode the activations are a few dozen rows (B*T) while the weights are
// megabytes, so the weight's output dimension is placed on the UMMA M axis
// (128 lanes of TMEM) and the activation rows on N ("swap AB"):
//
//     D[m, n] = sum_k A_z[m, k] * X_z[n, k]        (z = head, or 0)
//
// A (weight) is read once from HBM by TMA in 128 x 64 tiles, either K-major
// (rows of A contiguous along k) or MN-major (contiguous along m, as for
// W^UK whose stored rows run along d_c); X is K-major.  The accumulator
// tile [128 x BN] lives in TMEM.  A split-K grid dimension spreads long
// reductions (W^O: K = H*d_h) over more SMs; the last CTA of a tile to finish
// adds the fp32 partials in a fixed order and writes the bf16 result.
//
// Roles: warp 0 lane 0 issues TMA, warp 1 lane 0 issues UMMA (warp 1 also
// owns the TMEM allocation), then all four warps run the epilogue (warp w
// reads TMEM lanes 32w..32w+31).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "status.cuh"

namespace mla {
namespace gemm {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int STAGES = 4;  // pipeline depth (fewer when a CTA has fewer K chunks)
constexpr int THREADS = 128;
constexpr int A_BYTES = BM * BK * 2;  // 16 KB per stage

struct Params {
    int M, N, K;          // D is M x N, reduction length K (multiples of BM / BK)
    int BN;               // N tile (multiple of 16, <= 256)
    int n_tiles;          // ceil(N / BN)
    int a_mn;             // A stored MN-major
    int x_batched;        // X has a head coordinate (z); else z = 0 for X
    int splits;           // split-K factor (grid.z)
    int chunks_per_split; // K chunks (of BK) per split
    int stages;           // pipeline stages in shared memory, 1..STAGES
    __nv_bfloat16* out;   // out[(n0+n) * ldo + z * out_z + m0 + m]
    int64_t ldo, out_z;
    float* ws_part;       // [splits][Z][N][M] fp32 partials (split-K only)
    int* ws_count;        // [Z * n_tiles * (M / BM)] arrival counters (split-K only)
};

__device__ __forceinline__ uint32_t x_bytes(int BN) { return (uint32_t)BN * BK * 2; }

// At most 128 registers, so that up to four CTAs fit an SM when the
// pipeline is short (a short K leaves each CTA little to load: more CTAs in
// flight hide the TMA round trip).
__global__ void __launch_bounds__(THREADS, 4)
wgemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_x,
             const Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t xb = x_bytes(p.BN);
    const uint32_t stage_bytes = A_BYTES + xb;  // multiple of 1024 (BN % 8 == 0)
    const int S = p.stages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * stage_bytes);
    // bars[0..S): full, bars[S..2S): empty, bars[2S]: accumulator ready
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 1);
    int* flag = reinterpret_cast<int*>(tmem_slot + 1);  // [0] abort, [1] skip, [2] reduce

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int m_tile = blockIdx.x;
    const int z = blockIdx.y / p.n_tiles;
    const int n_tile = blockIdx.y % p.n_tiles;
    const int split = blockIdx.z;
    const int m0 = m_tile * BM, n0 = n_tile * p.BN;
    const int kc0 = split * p.chunks_per_split;
    const int kc1 = min(p.K / BK, kc0 + p.chunks_per_split);
    uint32_t tmem_cols = 32;
    while (tmem_cols < (uint32_t)p.BN) tmem_cols <<= 1;

    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S);
    const uint32_t acc_bar = smem_u32(bars + 2 * S);
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(acc_bar, 1);
        flag[0] = 0;
        flag[1] = device_status_raised() ? 1 : 0;  // one decision for the whole CTA
        fence_mbar_init_cluster();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool skip = flag[1] != 0 || kc1 <= kc0;

    bool ok = true;
    if (!skip && warp == 0 && lane == 0) {
        // ---------------------------------------------------------- producer
        const uint64_t pol = l2_policy_evict_first();
        int it = 0;
        for (int kc = kc0; kc < kc1; ++kc, ++it) {
            const int s = it % S;
            if (!mbar_wait(empty0 + 8 * s, ((it / S) & 1) ^ 1, 0x101)) { ok = false; break; }
            const uint32_t sa = smem_u32(smem + s * stage_bytes);
            const uint32_t sx = sa + A_BYTES;
            mbar_arrive_expect_tx(full0 + 8 * s, stage_bytes);
            if (p.a_mn) {
                tma_load_3d(sa, &tm_a, full0 + 8 * s, m0, kc * BK, z, pol);
                tma_load_3d(sa + A_BYTES / 2, &tm_a, full0 + 8 * s, m0 + 64, kc * BK, z, pol);
            } else {
                tma_load_3d(sa, &tm_a, full0 + 8 * s, kc * BK, m0, z, pol);
            }
            tma_load_3d(sx, &tm_x, full0 + 8 * s, kc * BK, p.x_batched ? z : 0, n0, pol);
        }
        // every issued copy lands before the CTA can exit (on the normal path
        // these phases have completed; after an abort they may not have)
        for (int i = max(0, it - S); i < it; ++i)
            mbar_wait_teardown(full0 + 8 * (i % S), (i / S) & 1, MLA_WAIT_LIMIT_NS);
    } else if (!skip && warp == 1 && lane == 0) {
        // --------------------------------------------------------------- MMA
        const uint32_t idesc = idesc_bf16(BM, p.BN, p.a_mn != 0, false);
        int it = 0;
        for (int kc = kc0; kc < kc1; ++kc, ++it) {
            const int s = it % S;
            if (!mbar_wait(full0 + 8 * s, (it / S) & 1, 0x103)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * stage_bytes);
            const uint32_t sx = sa + A_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                // A: K-major 128B-swizzled rows of 64 k, +32 B per 16-k step;
                //    MN-major: two 64-m boxes 8 KB apart, 16 k-rows = 2 KB.
                const uint64_t da = p.a_mn ? smem_desc(sa + kk * 2048, 8192, 1024, SWZ_128B)
                                           : smem_desc(sa + kk * 32, 16, 1024, SWZ_128B);
                const uint64_t dx = smem_desc(sx + kk * 32, 16, 1024, SWZ_128B);
                mma_ss(tmem, da, dx, idesc, (it > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(empty0 + 8 * s);
        }
        tc_commit(acc_bar);  // also on the abort path: tracks every issued MMA
    }
    if (!ok) atomicExch(flag, 1);

    // ------------------------------------------------------------- epilogue
    // good: this CTA's accumulator is complete and no error is known
    bool good = false;
    if (!skip) {
        good = __syncthreads_and(mbar_wait(acc_bar, 0, 0x104) ? 1 : 0) != 0;
        tc_fence_after();
        good = good && *flag == 0;
    }
    const int m = m0 + warp * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const int n_valid = min(p.BN, p.N - n0);
    if (p.splits == 1) {
        if (good) {
            __nv_bfloat16* dst = p.out + (int64_t)z * p.out_z + m;
            for (int c0 = 0; c0 < p.BN; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(trow + c0, r);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (c0 + j < n_valid)
                        dst[(int64_t)(n0 + c0 + j) * p.ldo] = __float2bfloat16_rn(__uint_as_float(r[j]));
            }
        }
    } else {
        const int Z = gridDim.y / p.n_tiles;
        if (good) {
            float* part = p.ws_part + (((int64_t)split * Z + z) * p.N) * p.M + m;
            for (int c0 = 0; c0 < p.BN; c0 += 16) {
                uint32_t r[16];
                tmem_ld16(trow + c0, r);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (c0 + j < n_valid) part[(int64_t)(n0 + c0 + j) * p.M] = __uint_as_float(r[j]);
            }
            __threadfence();
        }
        // Every CTA of the tile arrives on its counter -- also one that
        // skipped or gave up -- and the last arrival resets it, so the
        // counters are back at zero for the next call whatever happened in
        // this one.  Only a last arrival that sees no error anywhere reduces.
        __syncthreads();
        const int tile = (z * p.n_tiles + n_tile) * (p.M / BM) + m_tile;
        if (threadIdx.x == 0) {
            const int prev = atomicAdd(p.ws_count + tile, 1);
            const bool last = prev == p.splits - 1;
            if (last) p.ws_count[tile] = 0;
            flag[2] = last && good && !device_status_raised() ? 2 : 0;
        }
        __syncthreads();
        if (flag[2] == 2) {  // last split of this tile: reduce in split order
            __threadfence();
            __nv_bfloat16* dst = p.out + (int64_t)z * p.out_z + m;
            // 8 columns at a time, each split's 8 loads issued together (the
            // sum still runs over the splits in order)
            for (int nb = 0; nb < n_valid; nb += 8) {
                float acc[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll 4
                for (int s = 0; s < p.splits; ++s) {
                    const float* src = p.ws_part + (((int64_t)s * Z + z) * p.N + n0 + nb) * p.M + m;
                    float v[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = nb + j < n_valid ? __ldcg(src + (int64_t)j * p.M) : 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[j] += v[j];
                }
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (nb + j < n_valid) dst[(int64_t)(n0 + nb + j) * p.ldo] = __float2bfloat16_rn(acc[j]);
            }
        }
    }
    // the products (and their commits) are done before TMEM goes away, even
    // when the epilogue gave up waiting for them
    if (!skip && threadIdx.x == 32) mbar_wait_teardown(acc_bar, 0, MLA_WAIT_LIMIT_NS);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, tmem_cols);
}

}  // namespace gemm
}  // namespace mla
