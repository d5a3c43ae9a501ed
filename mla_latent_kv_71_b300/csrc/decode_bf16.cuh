// decode_bf16.cuh -- absorbed MLA decode attention on tcgen05 tensor cores.
//
// What it computes (per sequence b, query token t, head i):
//     s_j = (q_lat . c_j + q_pe . k^R_j) * scale,
//     o   = sum_j softmax_j(s) c_j,  lse = ln sum_j e^{s_j}
// over the cached rows [c_j ; k^R_j] of a paged latent cache ([llms] "Query
// Key Absorption", "Value Output Absorption"; [Zhang] "Decoupled RoPE",
// "Value absorption"; [Mishra] "Step 4: decoupled RoPE").  All heads of a
// query share the cache rows, so the 128 heads form the M = 128 rows of two
// dense UMMA contractions per 64-token page:
//     S [128 x 64]  = Q [128 x 576] . K^T     (K = the page's 576-wide rows)
//     O [128 x 512] += P [128 x 64] . C       (C = the page's 512 latents)
//
// Layout on the chip.  O alone (128 x 512 fp32) fills a whole SM's TMEM, so
// a cluster of two CTAs splits the feature axis: CTA r owns latent columns
// 256r .. 256r+255 and RoPE columns 32r .. 32r+31 (288 of the 576 features).
// Each CTA loads only its half of every page (36 KB, one TMA box per 64
// columns), computes a partial S over its 288 features, and the two partial
// S tiles are exchanged through distributed shared memory (st.async with
// transaction-count completion).  Both CTAs then hold the identical full S,
// run the identical online softmax and accumulate their own 256 columns of O.
// Every cache byte is read from HBM once and no tensor work is duplicated.
//
// TMEM per CTA (512 columns allocated):
//     [0,256)   O half, fp32          [256,320) S, fp32
//     [320,352) P, bf16 pairs         [352,496) Q half, bf16 pairs
// Q and P are UMMA A operands read from TMEM; the page tile in shared memory
// is the B operand of both products: K-major for S (features contiguous),
// MN-major for O (the same bytes, read along the feature axis).
//
// Warp roles (192 threads): warp 0 loads pages with TMA (and zeroes the rows
// past the end of a partial last page), warp 1 issues UMMA and owns TMEM,
// warps 2..5 run the softmax, the score exchange and the epilogue with one
// thread per head row.
//
// Work split: the pages of all (sequence, token, head-group) units are laid
// end to end and cut into equal contiguous ranges, one per cluster, so long
// and ragged sequences are spread over every SM.  A unit that straddles a
// range boundary is finished by each cluster as a partial (normalised o and
// its lse, fp32, in the workspace) and merged by a log-sum-exp combine
// kernel launched after this one.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "status.cuh"

namespace mla {
namespace dec {

constexpr int PAGE = 64;       // tokens per page
constexpr int DC = 512;        // latent width
constexpr int DR = 64;         // RoPE key width
constexpr int HALF_C = 256;    // latent columns per CTA
constexpr int HALF_R = 32;     // RoPE columns per CTA
constexpr int HEADS = 128;     // heads per unit (UMMA M)
constexpr int NSTAGE = 4;      // page pipeline depth
constexpr int THREADS = 192;
constexpr int SM_WARP0 = 2;    // first softmax warp

constexpr uint32_t BOX_C_BYTES = PAGE * 128;                      // 64 rows x 64 bf16
constexpr uint32_t BOX_R_BYTES = PAGE * 64;                       // 64 rows x 32 bf16
constexpr uint32_t STAGE_BYTES = 4 * BOX_C_BYTES + BOX_R_BYTES;   // 36864
constexpr uint32_t X_BYTES = HEADS * PAGE * 4;                    // partial S, fp32
constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_X = NSTAGE * STAGE_BYTES;
constexpr uint32_t OFF_BAR = OFF_X + 2 * X_BYTES;
constexpr uint32_t NUM_BARS = 2 * NSTAGE + 11;
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * 32;
constexpr uint32_t OFF_SCAN = OFF_MISC + 64;
constexpr uint32_t SMEM_BYTES = OFF_SCAN + 8 * THREADS;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;  // slack for 1 KB alignment

constexpr uint32_t TM_O = 0, TM_S = 256, TM_P = 320, TM_Q = 352, TM_COLS = 512;

// S = Q . K^T: M = 128 heads, N = 64 tokens, both operands K-major.
constexpr uint32_t IDESC_QK = idesc_bf16(128, 64, false, false);
// O += P . C: M = 128 heads, N = 256 latent columns, B MN-major.
constexpr uint32_t IDESC_PV = idesc_bf16(128, 256, false, true);

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
// Lazy rescaling: the running maximum is only moved when a new score exceeds
// it by more than this (log2 units), so exponentials stay <= 2^8.
constexpr float RESCALE_THRESHOLD = 8.0f;

struct Params {
    const __nv_bfloat16* q_lat;  // [B, T, H, 512]
    const __nv_bfloat16* q_pe;   // [B, T, H, 64]
    const int32_t* page_table;   // [B, max_pages]
    const int32_t* seq_lens;     // [B]
    __nv_bfloat16* o;            // [B, T, H, 512]
    float* lse;                  // [B, T, H]
    float* ws_o;                 // [slots, 128, 512] normalised partial outputs
    float* ws_lse;               // [slots, 128]
    int2* ws_unit;               // [U] (first cluster, last cluster) of each unit
    int B, T, H, HG;             // HG = ceil(H / 128) head groups
    int max_pages;
    int64_t num_pages;
    float scale_log2;            // scale * log2(e)
    int causal;
};

// ------------------------------------------------------------------ plan
//
// The work plan is a pure function of the sequence lengths, shared by the
// kernel (every CTA derives it independently) and by the host
// (mla_decode_plan, and the decision to skip the combine launch).
//
// Units u = ((b*T + t)*HG + hg) are laid end to end by their pages; the line
// of `total` pages is cut into G = min(clusters, total) contiguous ranges,
// range g = [total*g/G, total*(g+1)/G), none of them empty.  A unit cut by a
// range boundary is processed in pieces; piece (g, u) writes partial slot
// g + u, which is unique because both g and u only grow along the line.

struct PlanView {
    const int32_t* seq_lens;  // [B]
    int B, T, HG, max_pages, causal;
};

// Visible positions and pages of unit u.
struct Unit {
    int b, t, hg;
    int64_t len;    // visible positions
    int64_t pages;  // ceil(len / 64)
    bool bad_len;   // seq_lens[b] outside [0, max_pages * 64] (clamped)
};

__host__ __device__ __forceinline__ Unit unit_of(const PlanView& v, int64_t u) {
    Unit r;
    const int64_t bt = u / v.HG;
    r.hg = (int)(u % v.HG);
    r.b = (int)(bt / v.T);
    r.t = (int)(bt % v.T);
    int64_t len = v.seq_lens[r.b];
    const int64_t cap = (int64_t)v.max_pages * PAGE;
    r.bad_len = len < 0 || len > cap;
    if (r.bad_len) len = len < 0 ? 0 : cap;
    const int64_t n = v.causal ? len - (v.T - 1 - r.t) : len;
    r.len = n < 0 ? 0 : n;
    r.pages = (r.len + PAGE - 1) / PAGE;
    return r;
}

__host__ __device__ __forceinline__ int64_t range_start(int64_t total, int64_t g, int64_t G) {
    return total * g / G;
}

// Clusters used for `total` pages when `launched` clusters run.
__host__ __device__ __forceinline__ int64_t clusters_used(int64_t total, int64_t launched) {
    return total < launched ? total : launched;
}

// The range (cluster) holding page x of the line.
__host__ __device__ __forceinline__ int64_t cluster_of_page(int64_t x, int64_t total, int64_t G) {
    int64_t g = x * G / total;
    while (g + 1 < G && range_start(total, g + 1, G) <= x) ++g;
    while (g > 0 && range_start(total, g, G) > x) --g;
    return g;
}

// A piece of a unit processed by one cluster.
struct Segment {
    int64_t u;
    Unit un;
    int64_t lp0, lp1;          // page range within the unit
    int64_t slot;              // partial slot, or -1 when the whole unit is here
    int64_t g_first, g_last;   // clusters holding the unit's first and last page
};

// Walks the units overlapping cluster g's range, in line order.
struct Walker {
    PlanView v;
    int64_t U, rs, re, total, G, g;
    int64_t u, pos;  // next unit and its first page on the line
    __host__ __device__ bool next(Segment& s) {
        if (rs >= re) return false;  // an empty range has no piece
        while (pos < re && u < U) {
            const Unit un = unit_of(v, u);
            const int64_t start = pos;
            pos += un.pages;
            const int64_t cu = u++;
            if (un.pages == 0 || pos <= rs) continue;
            s.u = cu;
            s.un = un;
            s.lp0 = (rs > start ? rs : start) - start;
            s.lp1 = (re < pos ? re : pos) - start;
            s.g_first = cluster_of_page(start, total, G);
            s.g_last = cluster_of_page(pos - 1, total, G);
            s.slot = (s.g_first == s.g_last) ? -1 : g + cu;
            return true;
        }
        return false;
    }
};

// Walker of cluster g, found by a sequential scan (host side).
inline Walker host_walker(const PlanView& v, int64_t launched, int64_t g) {
    Walker w;
    w.v = v;
    w.U = (int64_t)v.B * v.T * v.HG;
    int64_t total = 0;
    for (int64_t u = 0; u < w.U; ++u) total += unit_of(v, u).pages;
    w.total = total;
    w.G = clusters_used(total, launched);
    w.g = g;
    w.rs = w.re = 0;
    w.u = w.U;
    w.pos = 0;
    if (total == 0 || g >= w.G) return w;
    w.rs = range_start(total, g, w.G);
    w.re = range_start(total, g + 1, w.G);
    int64_t pos = 0;
    for (int64_t u = 0; u < w.U; ++u) {
        const int64_t n = unit_of(v, u).pages;
        if (w.rs < pos + n) {
            w.u = u;
            w.pos = pos;
            break;
        }
        pos += n;
    }
    return w;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
decode_bf16_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_r,
                   const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    const uint32_t bar0 = smem_u32(smem + OFF_BAR);
    auto FULL = [&](int s) { return bar0 + 8u * s; };
    auto EMPTY = [&](int s) { return bar0 + 8u * (NSTAGE + s); };
    const uint32_t S_FULL = bar0 + 8u * (2 * NSTAGE + 0);
    const uint32_t S_FREE = bar0 + 8u * (2 * NSTAGE + 1);
    const uint32_t P_FULL = bar0 + 8u * (2 * NSTAGE + 2);
    const uint32_t PV_DONE = bar0 + 8u * (2 * NSTAGE + 3);
    const uint32_t Q_FULL = bar0 + 8u * (2 * NSTAGE + 4);
    auto XFULL = [&](int b) { return bar0 + 8u * (2 * NSTAGE + 5 + b); };
    auto XFREE = [&](int b) { return bar0 + 8u * (2 * NSTAGE + 7 + b); };
    const uint32_t TAIL = bar0 + 8u * (2 * NSTAGE + 9);
    const uint32_t DRAIN = bar0 + 8u * (2 * NSTAGE + 10);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    int64_t* misc = reinterpret_cast<int64_t*>(smem + OFF_MISC + 8);
    int64_t* scan = reinterpret_cast<int64_t*>(smem + OFF_SCAN);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(FULL(s), 1);
            mbar_init(EMPTY(s), 1);
        }
        mbar_init(S_FULL, 1);
        mbar_init(S_FREE, HEADS);
        mbar_init(P_FULL, HEADS);
        mbar_init(PV_DONE, 1);
        mbar_init(Q_FULL, HEADS);
        for (int b = 0; b < 2; ++b) {
            mbar_init(XFULL(b), 1);
            mbar_init(XFREE(b), 4);  // one arrival per softmax warp of the peer
        }
        mbar_init(TAIL, 1);
        mbar_init(DRAIN, 1);
        fence_mbar_init_cluster();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_c);
        tma_prefetch_desc(&tm_r);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TM_COLS);

    // ---------------------------------------------------------------- plan
    // Every CTA derives the same cut of the page line from seq_lens.
    PlanView pv;
    pv.seq_lens = p.seq_lens;
    pv.B = p.B;
    pv.T = p.T;
    pv.HG = p.HG;
    pv.max_pages = p.max_pages;
    pv.causal = p.causal;
    const int64_t U = (int64_t)p.B * p.T * p.HG;
    const int64_t launched = num_clusters_x(), g_id = cluster_id_x();
    {
        const int64_t chunk = (U + THREADS - 1) / THREADS;
        const int64_t u0 = min(U, (int64_t)threadIdx.x * chunk), u1 = min(U, u0 + chunk);
        int64_t sum = 0;
        bool bad = false;
        for (int64_t u = u0; u < u1; ++u) {
            const Unit un = unit_of(pv, u);
            sum += un.pages;
            bad |= un.bad_len;
        }
        if (bad && rank == 0 && g_id == 0) raise_device_status(MLA_DEV_BOUNDS, 0x10);
        scan[threadIdx.x] = sum;
        __syncthreads();
        if (threadIdx.x == 0) {
            int64_t acc = 0;
            for (int i = 0; i < THREADS; ++i) {
                const int64_t v = scan[i];
                scan[i] = acc;
                acc += v;
            }
            misc[0] = acc;  // total pages
            misc[1] = U;    // first unit of this cluster's range (default: none)
            misc[2] = 0;
            misc[3] = device_status_raised() ? 1 : 0;  // one decision for the whole CTA
        }
        __syncthreads();
        const int64_t total = misc[0];
        const int64_t G = clusters_used(total, launched);
        const int64_t rs = g_id < G ? range_start(total, g_id, G) : total;
        const int64_t pre = scan[threadIdx.x];
        if (g_id < G && rs >= pre && rs < pre + sum) {
            int64_t pos = pre;
            for (int64_t u = u0; u < u1; ++u) {
                const int64_t n = unit_of(pv, u).pages;
                if (rs < pos + n) {
                    misc[1] = u;
                    misc[2] = pos;
                    break;
                }
                pos += n;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // the peer's barriers are initialised before any remote access

    const uint32_t tmem = *tmem_slot;
    Walker walk;
    walk.v = pv;
    walk.U = U;
    walk.total = misc[0];
    walk.G = clusters_used(walk.total, launched);
    walk.g = g_id;
    walk.rs = g_id < walk.G ? range_start(walk.total, g_id, walk.G) : 0;
    walk.re = g_id < walk.G ? range_start(walk.total, g_id + 1, walk.G) : 0;
    walk.u = misc[1];
    walk.pos = misc[2];
    const bool skip = misc[3] != 0;

    if (warp == 0) {
        // ========================================================= producer
        const uint64_t pol = l2_policy_evict_first();
        int64_t it = 0;
        uint32_t tail_phase = 0;
        bool ok = !skip;
        Segment sg;
        while (ok && walk.next(sg)) {
            for (int64_t lp = sg.lp0; lp < sg.lp1 && ok; ++lp, ++it) {
                const int s = (int)(it % NSTAGE);
                ok = mbar_wait(EMPTY(s), (uint32_t)((it / NSTAGE) & 1) ^ 1u, 0x201);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                int64_t pg = p.page_table[(int64_t)sg.un.b * p.max_pages + lp];
                if (pg < 0 || pg >= p.num_pages) {
                    raise_device_status(MLA_DEV_BOUNDS, 0x20);
                    pg = 0;
                }
                const int y = (int)(pg * PAGE);
                const int valid = (int)(sg.un.len - lp * PAGE < PAGE ? sg.un.len - lp * PAGE : PAGE);
                const uint32_t st = smem_u32(smem + OFF_STAGE + s * STAGE_BYTES);
                const uint32_t bar = valid == PAGE ? FULL(s) : TAIL;
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar, STAGE_BYTES);
                    for (int k = 0; k < 4; ++k)
                        tma_load_2d(st + k * BOX_C_BYTES, &tm_c, bar, (int)rank * HALF_C + 64 * k,
                                    y, pol);
                    tma_load_2d(st + 4 * BOX_C_BYTES, &tm_r, bar, DC + (int)rank * HALF_R, y, pol);
                }
                if (valid < PAGE) {
                    // Rows past the end may hold anything (even NaN); zero
                    // them so that P = 0 there cannot meet a NaN in P . C.
                    ok = mbar_wait(TAIL, tail_phase, 0x202);
                    ok = __all_sync(0xffffffffu, ok);
                    tail_phase ^= 1u;
                    if (!ok) {
                        ++it;  // the loads have landed; nothing is in flight
                        break;
                    }
                    uint8_t* tile = smem + OFF_STAGE + s * STAGE_BYTES;
                    const int rows = PAGE - valid;
                    for (int idx = lane; idx < rows * 8 * 4; idx += 32) {  // latent boxes
                        const int box = idx / (rows * 8), rem = idx % (rows * 8);
                        uint4* dst = reinterpret_cast<uint4*>(tile + box * BOX_C_BYTES +
                                                              (valid + rem / 8) * 128 + (rem % 8) * 16);
                        *dst = make_uint4(0u, 0u, 0u, 0u);
                    }
                    for (int idx = lane; idx < rows * 4; idx += 32) {  // RoPE box
                        uint4* dst = reinterpret_cast<uint4*>(tile + 4 * BOX_C_BYTES +
                                                              (valid + idx / 4) * 64 + (idx % 4) * 16);
                        *dst = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(FULL(s));
                }
            }
        }
        if (!ok) {  // let every issued copy land before the CTA can exit
            for (int64_t i = (it > NSTAGE ? it - NSTAGE : 0); i < it; ++i)
                mbar_wait(FULL((int)(i % NSTAGE)), (uint32_t)((i / NSTAGE) & 1), 0x203);
        } else {
            // Producer tail: the tensor core's last releases of the ring
            // (tcgen05.commit arrivals) land before shared memory goes away.
            for (int64_t i = (it > NSTAGE ? it - NSTAGE : 0); i < it; ++i)
                mbar_wait(EMPTY((int)(i % NSTAGE)), (uint32_t)((i / NSTAGE) & 1), 0x204);
        }
    } else if (warp == 1) {
        // ============================================================== MMA
        if (lane == 0) {
            int64_t it = 0, n_qk = 0, n_pv = 0, n_unit = 0;
            bool ok = !skip;
            bool issued = false;
            Segment sg;
            auto issue_pv = [&](int s, bool first) {
                const uint32_t st = smem_u32(smem + OFF_STAGE + s * STAGE_BYTES);
#pragma unroll
                for (int k = 0; k < PAGE / 16; ++k) {
                    // C as MN-major B: 64-column boxes 8 KB apart, 8-row
                    // groups 1 KB apart, 16 tokens = 2 KB per step.
                    const uint64_t db = smem_desc(st + k * 2048, BOX_C_BYTES, 1024, SWZ_128B);
                    mma_ts(tmem + TM_O, tmem + TM_P + 8 * k, db, IDESC_PV,
                           (first && k == 0) ? 0u : 1u);
                }
            };
            while (ok && walk.next(sg)) {
                ok = mbar_wait(Q_FULL, (uint32_t)(n_unit & 1), 0x301);
                ++n_unit;
                if (!ok) break;
                tc_fence_after();
                int prev_s = -1;
                for (int64_t lp = sg.lp0; lp < sg.lp1; ++lp, ++it) {
                    const int s = (int)(it % NSTAGE);
                    ok = mbar_wait(FULL(s), (uint32_t)((it / NSTAGE) & 1), 0x302);
                    if (ok && n_qk > 0) ok = mbar_wait(S_FREE, (uint32_t)((n_qk - 1) & 1), 0x303);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t st = smem_u32(smem + OFF_STAGE + s * STAGE_BYTES);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {  // latent features, K-major SW128
                        const uint64_t db =
                            smem_desc(st + (k / 4) * BOX_C_BYTES + (k % 4) * 32, 16, 1024, SWZ_128B);
                        mma_ts(tmem + TM_S, tmem + TM_Q + 8 * k, db, IDESC_QK, k > 0 ? 1u : 0u);
                    }
#pragma unroll
                    for (int k = 0; k < 2; ++k) {  // RoPE features, K-major SW64
                        const uint64_t db = smem_desc(st + 4 * BOX_C_BYTES + k * 32, 16, 512, SWZ_64B);
                        mma_ts(tmem + TM_S, tmem + TM_Q + 128 + 8 * k, db, IDESC_QK, 1u);
                    }
                    issued = true;
                    tc_commit(S_FULL);
                    ++n_qk;
                    if (prev_s >= 0) {
                        ok = mbar_wait(P_FULL, (uint32_t)(n_pv & 1), 0x304);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(prev_s, lp - 1 == sg.lp0);
                        tc_commit(PV_DONE);
                        tc_commit(EMPTY(prev_s));
                        ++n_pv;
                    }
                    prev_s = s;
                }
                if (!ok) break;
                ok = mbar_wait(P_FULL, (uint32_t)(n_pv & 1), 0x305);
                if (!ok) break;
                tc_fence_after();
                issue_pv(prev_s, sg.lp1 - 1 == sg.lp0);
                tc_commit(PV_DONE);
                tc_commit(EMPTY(prev_s));
                ++n_pv;
            }
            if (!ok && issued) {  // wait for the tensor core before TMEM goes away
                tc_commit(DRAIN);
                mbar_wait(DRAIN, 0, 0x306);
            }
        }
        __syncwarp();
    } else {
        // ==================================================== softmax warps
        const int q4 = warp & 3;             // TMEM lane quarter of this warp
        const int h = q4 * 32 + lane;        // head row within the group
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        const uint32_t x_base = smem_u32(smem + OFF_X);
        const uint32_t peer_x = map_to_rank(x_base, peer);
        int64_t n_s = 0, n_pv = 0, n_x = 0;
        bool ok = !skip;
        Segment sg;
        while (ok && walk.next(sg)) {
            const int head = sg.un.hg * HEADS + h;
            const bool live = head < p.H;
            const int64_t qrow = ((int64_t)sg.un.b * p.T + sg.un.t) * p.H + head;
            // ---- this CTA's half of the query row -> TMEM (bf16 pairs)
            {
                const uint4* ql = reinterpret_cast<const uint4*>(p.q_lat + qrow * DC + rank * HALF_C);
                const uint4* qp = reinterpret_cast<const uint4*>(p.q_pe + qrow * DR + rank * HALF_R);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const uint4 x = live ? __ldg(ql + c * 8 + v) : make_uint4(0u, 0u, 0u, 0u);
                        r[4 * v] = x.x;
                        r[4 * v + 1] = x.y;
                        r[4 * v + 2] = x.z;
                        r[4 * v + 3] = x.w;
                    }
                    tmem_st32(trow + TM_Q + 32 * c, r);
                }
                uint32_t r[16];
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint4 x = live ? __ldg(qp + v) : make_uint4(0u, 0u, 0u, 0u);
                    r[4 * v] = x.x;
                    r[4 * v + 1] = x.y;
                    r[4 * v + 2] = x.z;
                    r[4 * v + 3] = x.w;
                }
                tmem_st16(trow + TM_Q + 128, r);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(Q_FULL);
            }
            float m_used = -INFINITY, l = 0.f;
            for (int64_t lp = sg.lp0; lp < sg.lp1; ++lp) {
                // ---- partial scores of this CTA's features
                ok = __all_sync(0xffffffffu, mbar_wait(S_FULL, (uint32_t)(n_s & 1), 0x401));
                ++n_s;
                if (!ok) break;
                tc_fence_after();
                float s[PAGE];
                {
                    uint32_t r[32];
                    tmem_ld32(trow + TM_S, r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(r[j]);
                    tmem_ld32(trow + TM_S + 32, r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) s[32 + j] = __uint_as_float(r[j]);
                }
                tc_fence_before();
                mbar_arrive(S_FREE);
                // ---- exchange with the peer: send ours, receive theirs
                const int xb = (int)(n_x & 1);
                const uint32_t xph = (uint32_t)((n_x >> 1) & 1);
                ++n_x;
                ok = __all_sync(0xffffffffu, mbar_wait<true>(XFREE(xb), xph ^ 1u, 0x402));
                if (!ok) break;
                {
                    const uint32_t dst = peer_x + xb * X_BYTES;
                    const uint32_t pbar = map_to_rank(XFULL(xb), peer);
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        st_async_v4(dst + (k * HEADS + h) * 16, __float_as_uint(s[4 * k]),
                                    __float_as_uint(s[4 * k + 1]), __float_as_uint(s[4 * k + 2]),
                                    __float_as_uint(s[4 * k + 3]), pbar);
                }
                if (h == 0) mbar_arrive_expect_tx(XFULL(xb), X_BYTES);
                ok = __all_sync(0xffffffffu, mbar_wait<true>(XFULL(xb), xph, 0x403));
                if (!ok) break;
                {
                    const float4* src = reinterpret_cast<const float4*>(smem + OFF_X + xb * X_BYTES);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float4 v = src[k * HEADS + h];
                        s[4 * k] += v.x;
                        s[4 * k + 1] += v.y;
                        s[4 * k + 2] += v.z;
                        s[4 * k + 3] += v.w;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(map_to_rank(XFREE(xb), peer));
                // ---- online softmax (base 2), lazily rescaled
                const int valid = (int)(sg.un.len - lp * PAGE < PAGE ? sg.un.len - lp * PAGE : PAGE);
                float mx = -INFINITY;
#pragma unroll
                for (int j = 0; j < PAGE; ++j) {
                    s[j] = j < valid ? s[j] * p.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, s[j]);
                }
                const bool first = lp == sg.lp0;
                if (first) m_used = mx;
                const bool need = !first && mx > m_used + RESCALE_THRESHOLD;
                if (!first) {  // PV of the previous page done: P is free, O is stable
                    ok = __all_sync(0xffffffffu, mbar_wait(PV_DONE, (uint32_t)(n_pv & 1), 0x404));
                    ++n_pv;
                    if (!ok) break;
                    tc_fence_after();
                }
                if (__any_sync(0xffffffffu, need)) {
                    const float m_new = need ? mx : m_used;
                    const float alpha = ex2(m_used - m_new);
#pragma unroll 1
                    for (int c = 0; c < HALF_C; c += 32) {
                        uint32_t r[32];
                        tmem_ld32(trow + TM_O + c, r);
#pragma unroll
                        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
                        tmem_st32(trow + TM_O + c, r);
                    }
                    l *= alpha;
                    m_used = m_new;
                }
                {
                    uint32_t pk[32];
                    float sum = 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float p0 = ex2(s[2 * j] - m_used);
                        const float p1 = ex2(s[2 * j + 1] - m_used);
                        sum += p0 + p1;
                        pk[j] = pack_bf16x2(p0, p1);
                    }
                    l += sum;
                    tmem_st32(trow + TM_P, pk);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(P_FULL);
            }
            if (!ok) break;
            // ---- epilogue: O / l of this CTA's 256 columns, lse
            ok = __all_sync(0xffffffffu, mbar_wait(PV_DONE, (uint32_t)(n_pv & 1), 0x405));
            ++n_pv;
            if (!ok) break;
            tc_fence_after();
            const float inv_l = 1.f / l;
            if (sg.slot < 0) {
                __nv_bfloat16* dst = p.o + qrow * DC + rank * HALF_C;
#pragma unroll 1
                for (int c = 0; c < HALF_C; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(trow + TM_O + c, r);
                    if (live) {
                        uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            d4[v] = make_uint4(
                                pack_bf16x2(__uint_as_float(r[8 * v]) * inv_l, __uint_as_float(r[8 * v + 1]) * inv_l),
                                pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv_l, __uint_as_float(r[8 * v + 3]) * inv_l),
                                pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv_l, __uint_as_float(r[8 * v + 5]) * inv_l),
                                pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv_l, __uint_as_float(r[8 * v + 7]) * inv_l));
                    }
                }
                if (live && rank == 0) p.lse[qrow] = (m_used + __log2f(l)) * LN2;
            } else {
                float* dst = p.ws_o + (sg.slot * HEADS + h) * DC + rank * HALF_C;
#pragma unroll 1
                for (int c = 0; c < HALF_C; c += 32) {
                    uint32_t r[32];
                    tmem_ld32(trow + TM_O + c, r);
                    float4* d4 = reinterpret_cast<float4*>(dst + c);
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        d4[v] = make_float4(__uint_as_float(r[4 * v]) * inv_l, __uint_as_float(r[4 * v + 1]) * inv_l,
                                            __uint_as_float(r[4 * v + 2]) * inv_l, __uint_as_float(r[4 * v + 3]) * inv_l);
                }
                if (rank == 0) p.ws_lse[sg.slot * HEADS + h] = (m_used + __log2f(l)) * LN2;
            }
            if (rank == 0 && h == 0 && sg.g_first == walk.g)
                p.ws_unit[sg.u] = make_int2((int)sg.g_first, (int)sg.g_last);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, TM_COLS);
    cluster_sync();
}

// Merge the partial slots of split units (grid: U * 128 blocks of 128
// threads, one head row each); also writes o = 0, lse = -inf for units that
// see no cached position.
__global__ void __launch_bounds__(128)
decode_combine_kernel(const Params p) {
    if (device_status_raised()) return;
    const int64_t u = blockIdx.x / HEADS;
    const int h = blockIdx.x % HEADS;
    PlanView pv;
    pv.seq_lens = p.seq_lens;
    pv.B = p.B;
    pv.T = p.T;
    pv.HG = p.HG;
    pv.max_pages = p.max_pages;
    pv.causal = p.causal;
    const Unit un = unit_of(pv, u);
    const int head = un.hg * HEADS + h;
    if (head >= p.H) return;
    const int64_t qrow = ((int64_t)un.b * p.T + un.t) * p.H + head;
    const int c = 4 * threadIdx.x;
    __nv_bfloat16* dst = p.o + qrow * DC + c;
    if (un.pages == 0) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(0u, 0u);
        if (threadIdx.x == 0) p.lse[qrow] = -INFINITY;
        return;
    }
    const int2 gg = p.ws_unit[u];
    if (gg.x == gg.y) return;  // written directly by the attention kernel
    float m = -INFINITY;
    for (int g = gg.x; g <= gg.y; ++g) m = fmaxf(m, p.ws_lse[(g + u) * HEADS + h]);
    float sum = 0.f;
    for (int g = gg.x; g <= gg.y; ++g) sum += __expf(p.ws_lse[(g + u) * HEADS + h] - m);
    const float L = m + __logf(sum);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = gg.x; g <= gg.y; ++g) {
        const int64_t slot = g + u;
        const float w = __expf(p.ws_lse[slot * HEADS + h] - L);
        const float4 v = __ldcg(reinterpret_cast<const float4*>(p.ws_o + (slot * HEADS + h) * DC + c));
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    if (threadIdx.x == 0) p.lse[qrow] = L;
}

}  // namespace dec
}  // namespace mla
