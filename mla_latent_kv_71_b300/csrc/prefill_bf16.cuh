// prefill_bf16.cuh -- training-form (unabsorbed) MLA attention on tcgen05
// tensor cores, for prefill: every token of a sequence is a query.
//
// What it computes (per sequence b, query position t, head i):
//     k_{j,i} = [K_nope[j,i,:] ; k^R_j],   v_{j,i} = V[j,i,:]
//     s_j     = q_{t,i} . k_{j,i} * scale,      j <= t (causal) or all j < L
//     u_{t,i} = sum_j softmax_j(s) v_{j,i},     lse_{t,i} = ln sum_j e^{s_j}
// with K_nope = W^UK c and V = W^UV c expanded per head beforehand (a GEMM)
// and the decoupled RoPE key k^R_j shared by all heads ([Mishra] "Multi-head
// Latent Attention": the unabsorbed form is the one used in training; [llms]
// "Low-Rank Key-Value Joint Compression", "The Positional Problem and
// Decoupled RoPE").  For many queries this route needs 2(d_h + d_r) + 2 d_h
// = 640 FLOPs per (query, key, head) against 2176 for the absorbed one, so
// prefill runs it; it is bound by the tensor cores, not by memory.
//
// One CTA takes 128 queries of one head of one sequence and walks the key
// blocks of 128 (up to the diagonal when causal):
//     S [128 x 128] = Q [128 x 192] . K^T      (Q in TMEM, K in shared memory)
//     O [128 x 128] += P [128 x 128] . V       (P in TMEM, V in shared memory)
// TMEM (512 columns): S double-buffered at [0,128) and [128,256), O at
// [256,384), Q at [384,480).  Block j's P (bf16 pairs) overwrites the first
// 64 columns of its own S buffer once the softmax has its scores in
// registers.  Keys and values stream through separate TMA rings: a key
// block is released once its score product is done (three stages, so keys
// run well ahead), a value block once its P . V product is (two stages);
// the query rows are loaded by the softmax threads (one row each) into
// TMEM.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: K (content part per head, RoPE part shared)
//               and V tiles into the ring,
//   warp 1      TMEM owner; an elected lane issues S(j+1) while the softmax
//               works on S(j), then O += P(j) . V(j) once P(j) is in TMEM,
//   warps 2..5  one query row per thread (TMEM lane quarter = warp % 4):
//               online softmax with lazy rescaling, P into TMEM, the final
//               u = O / l and lse.
// Every wait is bounded (ptx.cuh); on a wait that gives up the CTA waits for
// its own copies and products before it frees TMEM and exits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "status.cuh"

namespace mla {
namespace pre {

constexpr int BQ = 128;        // queries per CTA (UMMA M)
constexpr int BK = 128;        // keys per block (UMMA N of S, K of O)
constexpr int DH = 128;        // content dims of q and k; dims of v
constexpr int DR = 64;         // RoPE dims
constexpr int NK = 3;           // key stages
constexpr int NV = 2;           // value stages
constexpr int THREADS = 192;
constexpr int SM_WARP0 = 2;    // softmax warps 2..5

constexpr uint32_t BOX_BYTES = BK * 128;                 // 128 rows x 64 bf16 (128-byte swizzle)
constexpr uint32_t K_BYTES = 3 * BOX_BYTES;              // content 0..63, 64..127, RoPE 0..63
constexpr uint32_t V_BYTES = 2 * BOX_BYTES;              // dims 0..63, 64..127
constexpr uint32_t OFF_V = NK * K_BYTES;                 // 144 KB of keys, then 64 KB of values
constexpr uint32_t OFF_BAR = OFF_V + NV * V_BYTES;
constexpr uint32_t NUM_BARS = 2 * NK + 2 * NV + 2 + 2 + 1 + 1 + 1;
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * NUM_BARS;
constexpr uint32_t SMEM_ALLOC = OFF_MISC + 64 + 1024;

constexpr uint32_t TM_S = 0, TM_O = 256, TM_Q = 384, TM_COLS = 512;

// S = Q . K^T: M = 128 queries, N = 128 keys, both K-major.
constexpr uint32_t IDESC_QK = idesc_bf16(BQ, BK, false, false);
// O += P . V: M = 128 queries, N = 128 dims, V MN-major (dims contiguous).
constexpr uint32_t IDESC_PV = idesc_bf16(BQ, DH, false, true);

constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units, as in the decode kernel

struct Params {
    const __nv_bfloat16* q_nope;  // [B*L, H, 128]
    const __nv_bfloat16* q_pe;    // [B*L, H, 64]
    __nv_bfloat16* u;             // [B*L, H, 128]
    float* lse;                   // [B*L, H]
    int B, L, H, nqb;             // nqb = ceil(L / 128) query blocks per sequence
    float scale_log2;             // scale * log2(e)
    int causal;
    int rope_col;                 // first RoPE column of a cache row (d_c)
};

__global__ void __launch_bounds__(THREADS, 1)
prefill_bf16_kernel(const __grid_constant__ CUtensorMap tm_kn,   // k_nope [B*L][H][128]
                    const __grid_constant__ CUtensorMap tm_kr,   // cache rows, RoPE columns
                    const __grid_constant__ CUtensorMap tm_v,    // v [B*L][H][128]
                    const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // The query blocks of one head are neighbours in launch order (x), so
    // the CTAs resident at a time share a few heads' keys and values in L2;
    // within a head the heaviest (latest) blocks go first.
    const int qb = p.nqb - 1 - (int)blockIdx.x;
    const int head = (int)blockIdx.y;
    const int seq = (int)blockIdx.z;
    const int q0 = qb * BQ;  // first query position of the block
    const int nkb = p.causal ? qb + 1 : (p.L + BK - 1) / BK;  // key blocks to visit
    const int64_t tok0 = (int64_t)seq * p.L;                  // the sequence's first token row

    poison_smem(smem, OFF_BAR);  // debug build: the key and value rings
    check_split(qb >= 0 && q0 < p.L && nkb >= 1 && (int64_t)(nkb - 1) * BK < p.L, 0x73);
    const uint32_t bar0 = smem_u32(smem + OFF_BAR);
    auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    auto K_FULL = [&](int s) { return BAR(s); };            // K(j) landed (TMA), stage j % NK
    auto K_EMPTY = [&](int s) { return BAR(NK + s); };      // S(j) done reading K(j) (commit)
    auto V_FULL = [&](int s) { return BAR(2 * NK + s); };   // V(j) landed (TMA), stage j % NV
    auto V_EMPTY = [&](int s) { return BAR(2 * NK + NV + s); };  // O(j) done reading V(j) (commit)
    constexpr int NB0 = 2 * NK + 2 * NV;
    auto S_FULL = [&](int b) { return BAR(NB0 + b); };      // S(j) in buffer j % 2 (commit)
    auto P_FULL = [&](int b) { return BAR(NB0 + 2 + b); };  // P(j) in TMEM (4 warps)
    const uint32_t O_DONE = BAR(NB0 + 4);                   // O += P(j) V(j) done (commit, phase j)
    const uint32_t Q_FULL = BAR(NB0 + 5);                   // query rows in TMEM (4 warps)
    const uint32_t DRAIN = BAR(NB0 + 6);                    // teardown: every product finished
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    int* flag = reinterpret_cast<int*>(smem + OFF_MISC + 8);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NK; ++s) {
            mbar_init(K_FULL(s), 1);
            mbar_init(K_EMPTY(s), 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(V_FULL(s), 1);
            mbar_init(V_EMPTY(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(S_FULL(b), 1);
            mbar_init(P_FULL(b), 4);
        }
        mbar_init(O_DONE, 1);
        mbar_init(Q_FULL, 4);
        mbar_init(DRAIN, 1);
        flag[0] = device_status_raised() ? 1 : 0;  // one decision for the whole CTA
        fence_mbar_init_cluster();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_kn);
        tma_prefetch_desc(&tm_kr);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const bool skip = flag[0] != 0;

    if (warp == 0) {
        // ========================================================= producer
        // K(j) then V(j) for each block in turn: a key stage is free once
        // the score product three blocks back is done, a value stage once
        // the P . V product two back is.
        int nk = 0, nv = 0;  // copies issued
        bool ok = !skip;
        if (lane == 0 && ok) {
            for (int j = 0; j < nkb; ++j) {
                const int y = (int)(tok0 + (int64_t)j * BK);  // first key row of the block
                const int sk = j % NK, sv = j % NV;
                if (!mbar_wait(K_EMPTY(sk), (uint32_t)((j / NK) & 1) ^ 1u, 0x601)) { ok = false; break; }
                const uint32_t kst = smem_u32(smem + sk * K_BYTES);
                mbar_arrive_expect_tx(K_FULL(sk), K_BYTES);
                // keys and values are read again by the head's other query
                // blocks: loaded with the normal L2 policy
                tma_load_3d_plain(kst, &tm_kn, K_FULL(sk), 0, head, y);
                tma_load_3d_plain(kst + BOX_BYTES, &tm_kn, K_FULL(sk), 64, head, y);
                tma_load_2d_plain(kst + 2 * BOX_BYTES, &tm_kr, K_FULL(sk), p.rope_col, y);
                ++nk;
                if (!mbar_wait(V_EMPTY(sv), (uint32_t)((j / NV) & 1) ^ 1u, 0x602)) { ok = false; break; }
                const uint32_t vst = smem_u32(smem + OFF_V + sv * V_BYTES);
                mbar_arrive_expect_tx(V_FULL(sv), V_BYTES);
                tma_load_3d_plain(vst, &tm_v, V_FULL(sv), 0, head, y);
                tma_load_3d_plain(vst + BOX_BYTES, &tm_v, V_FULL(sv), 64, head, y);
                ++nv;
            }
            // every copy issued here lands before the CTA can exit
            for (int i = (nk > NK ? nk - NK : 0); i < nk; ++i)
                mbar_wait_teardown(K_FULL(i % NK), (uint32_t)((i / NK) & 1), MLA_WAIT_LIMIT_NS);
            for (int i = (nv > NV ? nv - NV : 0); i < nv; ++i)
                mbar_wait_teardown(V_FULL(i % NV), (uint32_t)((i / NV) & 1), MLA_WAIT_LIMIT_NS);
        }
        __syncwarp();
    } else if (warp == 1) {
        // =============================================================== MMA
        bool ok = !skip;
        bool issued = false;
        const uint64_t dk0 = smem_desc(smem_u32(smem), 16, 1024, SWZ_128B);
        const uint64_t dv0 = smem_desc(smem_u32(smem + OFF_V), BOX_BYTES, 1024, SWZ_128B);
        auto issue_s = [&](int j) -> bool {  // S(j) = Q . K(j)^T into buffer j % 2
            const int s = j % NK;
            if (!__all_sync(0xffffffffu, mbar_wait(K_FULL(s), (uint32_t)((j / NK) & 1), 0x611))) return false;
            // buffer j % 2 last held P(j - 2), which O(j - 2) has read
            if (j >= 2 && !__all_sync(0xffffffffu, mbar_wait(O_DONE, (uint32_t)((j - 2) & 1), 0x612)))
                return false;
            tc_fence_after();
            if (elect_one_sync()) {
                const uint64_t dk = dk0 + ((uint64_t)(s * K_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < 12; ++k)  // 192 features: 3 boxes x 4 steps of 16
                    mma_ts(tmem + TM_S + BK * (j & 1), tmem + TM_Q + 8 * k,
                           dk + (uint64_t)(((k / 4) * BOX_BYTES + (k % 4) * 32) >> 4), IDESC_QK, k > 0 ? 1u : 0u);
                tc_commit(S_FULL(j & 1));
                tc_commit(K_EMPTY(s));
            }
            __syncwarp();
            issued = true;
            return true;
        };
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(Q_FULL, 0, 0x610));
        if (ok) ok = issue_s(0);
        for (int j = 0; ok && j < nkb; ++j) {
            if (j + 1 < nkb && !(ok = issue_s(j + 1))) break;
            // O += P(j) . V(j) once P(j) is in TMEM (and O rescaled, if it was)
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(P_FULL(j & 1), (uint32_t)((j >> 1) & 1), 0x613)))) break;
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(V_FULL(j % NV), (uint32_t)((j / NV) & 1), 0x614)))) break;
            tc_fence_after();
            if (elect_one_sync()) {
                const uint64_t dv = dv0 + ((uint64_t)((j % NV) * V_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)  // 16 keys per step: 8 P columns, 2 KB of V
                    mma_ts(tmem + TM_O, tmem + TM_S + BK * (j & 1) + 8 * k, dv + (uint64_t)((k * 2048) >> 4),
                           IDESC_PV, (j > 0 || k > 0) ? 1u : 0u);
                tc_commit(O_DONE);
                tc_commit(V_EMPTY(j % NV));
            }
            __syncwarp();
        }
        if (issued) {  // every product (and its commits) done before TMEM goes away
            if (elect_one_sync()) tc_commit(DRAIN);
            __syncwarp();
            mbar_wait_teardown(DRAIN, 0, MLA_WAIT_LIMIT_NS);
        }
        __syncwarp();
    } else {
        // =========================================================== softmax
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;          // this thread's query row in the block
        const int qpos = q0 + r;               // its position in the sequence
        const bool live = qpos < p.L;
        const int64_t qrow = (tok0 + (live ? qpos : 0)) * p.H + head;
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        bool ok = !skip;
        if (ok) {
            // the query row [q_nope ; q_pe] (192 bf16) into TMEM
            const uint4* qn = reinterpret_cast<const uint4*>(p.q_nope + qrow * DH);
            const uint4* qp = reinterpret_cast<const uint4*>(p.q_pe + qrow * DR);
            uint32_t v[32];
#pragma unroll
            for (int c = 0; c < 3; ++c) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint4 x = live ? __ldg((c < 2 ? qn + 8 * c : qp) + k) : make_uint4(0u, 0u, 0u, 0u);
                    v[4 * k] = x.x;
                    v[4 * k + 1] = x.y;
                    v[4 * k + 2] = x.z;
                    v[4 * k + 3] = x.w;
                }
                tmem_st32(trow + TM_Q + 32 * c, v);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(Q_FULL);
        }
        float m_ref = -INFINITY, l = 0.f, lr = 0.f;  // running max (log2 units), exact and rounded sums
        for (int j = 0; ok && j < nkb; ++j) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(S_FULL(j & 1), (uint32_t)((j >> 1) & 1), 0x620)))) break;
            tc_fence_after();
            const uint32_t sb = trow + TM_S + BK * (j & 1);
            float s[BK];
#pragma unroll
            for (int c = 0; c < BK / 32; ++c) tmem_ld32(sb + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(s + 32 * c));
            // keys visible to this query: all of the block, but at most up to
            // the query (causal, diagonal block) and to the sequence's end
            const int k0 = j * BK;
            int lim = p.L - k0;
            if (p.causal) lim = min(lim, qpos - k0 + 1);
            if (lim < BK) {
#pragma unroll
                for (int c = 0; c < BK; ++c) s[c] = c < lim ? s[c] : -INFINITY;
            }
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int c = 0; c < BK; c += 2) mx4[(c / 2) & 3] = fmax3(mx4[(c / 2) & 3], s[c], s[c + 1]);
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * p.scale_log2;
            // lazy rescaling: O moves to a new maximum only when a score
            // exceeds the reference by more than the threshold
            const bool need = mx > m_ref + RESCALE_THRESHOLD;
            const float m_used = need ? mx : m_ref;
            if (__any_sync(0xffffffffu, need) && j > 0) {
                // O holds blocks up to j - 1 once O(j - 1) is done
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(O_DONE, (uint32_t)((j - 1) & 1), 0x621)))) break;
                tc_fence_after();
                const float alpha = need ? ex2(m_ref - m_used) : 1.f;
#pragma unroll 1
                for (int c = 0; c < DH; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(trow + TM_O + c, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(trow + TM_O + c, o);
                }
                tmem_st_wait();
            }
            if (need) {
                const float f = m_ref == -INFINITY ? 0.f : ex2(m_ref - m_used);
                l *= f;
                lr *= f;
                m_ref = m_used;
            }
            // P = 2^(s * scale * log2 e - m) as bf16 pairs over the first 64
            // columns of this S buffer (its scores are all in registers)
            uint32_t pk[BK / 2];
            const bool dead = m_used == -INFINITY;  // nothing visible yet: every weight is 0
            const uint64_t nm2 = f2_pack(-m_used, -m_used);
            const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
            uint64_t sum2[2] = {0ull, 0ull}, sumr2[2] = {0ull, 0ull};
#pragma unroll
            for (int c = 0; c < BK / 2; ++c) {
                const uint64_t e = f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), c2, nm2);
                const float p0 = dead ? 0.f : ex2(f2_lo(e));
                const float p1 = dead ? 0.f : ex2(f2_hi(e));
                pk[c] = pack_bf16x2(p0, p1);
                // exact sum (lse) and sum of the rounded weights P . V takes
                // (normalises u): as in the decode kernel
                sum2[c & 1] = f2_add(sum2[c & 1], f2_pack(p0, p1));
                sumr2[c & 1] = f2_add(sumr2[c & 1], bf16x2_to_f2(pk[c]));
            }
            const uint64_t st2 = f2_add(sum2[0], sum2[1]), sr2 = f2_add(sumr2[0], sumr2[1]);
            l += f2_lo(st2) + f2_hi(st2);
            lr += f2_lo(sr2) + f2_hi(sr2);
            tmem_st32(sb, *reinterpret_cast<const uint32_t(*)[32]>(pk));
            tmem_st32(sb + 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(P_FULL(j & 1));
        }
        // ---- u = O / l (bf16) and lse, once the last product is done (its
        // phase is waited for after the one before: a wait by parity must
        // not meet the barrier two phases behind)
        if (ok && nkb >= 2)
            ok = __all_sync(0xffffffffu, mbar_wait(O_DONE, (uint32_t)((nkb - 2) & 1), 0x623));
        if (ok && nkb > 0 && __all_sync(0xffffffffu, mbar_wait(O_DONE, (uint32_t)((nkb - 1) & 1), 0x622))) {
            tc_fence_after();
            const float inv = lr > 0.f ? 1.f / lr : 0.f;
            uint4* dst = reinterpret_cast<uint4*>(p.u + qrow * DH);
#pragma unroll 1
            for (int c = 0; c < DH; c += 32) {
                uint32_t o[32];
                tmem_ld32(trow + TM_O + c, o);
                if (live) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[c / 8 + k] = make_uint4(
                            pack_bf16x2(__uint_as_float(o[8 * k]) * inv, __uint_as_float(o[8 * k + 1]) * inv),
                            pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv),
                            pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv),
                            pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv));
                }
            }
            if (live) p.lse[qrow] = l > 0.f ? (m_ref + __log2f(l)) * LN2 : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, TM_COLS);
}

}  // namespace pre
}  // namespace mla
