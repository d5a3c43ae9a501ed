// decode_bf16.cuh -- absorbed MLA decode attention on tcgen05 tensor cores.
//
// What it computes (per sequence b, query token t, head i):
//     s_j = (q_lat . c_j + q_pe . k^R_j) * scale,
//     o   = sum_j softmax_j(s) c_j,  lse = ln sum_j e^{s_j}
// over the cached rows [c_j ; k^R_j] of a paged latent cache ([llms] "Query
// Key Absorption", "Value Output Absorption"; [Zhang] "Decoupled RoPE",
// "Value absorption"; [Mishra] "Step 4: decoupled RoPE").  All heads of a
// query share the cache rows, so the 128 heads form the M = 128 rows of two
// dense UMMA contractions per tile of 32 cached tokens:
//     S [128 x 32]  = Q [128 x 576] . K^T     (K = the tile's 576-wide rows)
//     O [128 x 512] += P [128 x 32] . C       (C = the tile's 512 latents)
//
// Layout on the chip.  O alone (128 x 512 fp32) fills a whole SM's TMEM, so
// a cluster of two CTAs splits the feature axis: CTA r owns latent columns
// 256r .. 256r+255 and RoPE columns 32r .. 32r+31 (288 of the 576 features).
// Each CTA loads only its half of every 64-token page (36 KB, as two 32-token
// tiles of one TMA box per 64 columns), computes a partial S over its 288
// features, and the two
// partial S tiles are exchanged through distributed shared memory.  Both
// CTAs then run the identical softmax and accumulate their own 256 columns
// of O.  Every cache byte is read from HBM once and no tensor work is
// duplicated.
//
// The exchange (16 KB per tile each way) is slow next to the rest of a tile,
// so it is pipelined: two groups of four warps take alternate tiles, and a
// group runs the front half of its next tile (own partial S out of TMEM and
// off to the peer with st.async) before the back half of its current one
// (the peer's partial in, online softmax, P into TMEM), so one tile's
// exchange overlaps the other's exponentials.  The only serial hand-off
// between the groups is the running maximum of each row (and, at the end of
// a unit piece, the row sums), passed through shared memory.
//
// TMEM per CTA (all 512 columns):
//     [0,256)   O half, fp32          [256,384) latent Q half, bf16 pairs
//     [384,480) partial S, 3 x 32     [480,512) P, 2 x 16 bf16 pairs
// Tile i's partial S sits in buffer i % 3 until the back half of the tile
// has re-read it (so no tile's scores are carried in registers across the
// front half of the next); its P goes to buffer i % 2.  The latent Q and P
// are UMMA A operands read from TMEM; the RoPE part of Q (128 x 32) sits in
// shared memory and feeds the two RoPE steps of S as an SS product.  The
// tile's rows in shared memory are the B operand of both products: K-major
// for S (features contiguous), MN-major for O (the same bytes, read along
// the feature axis).
//
// The ring holds eight tiles (half pages), each stage released as soon as
// its own tile's O product is done: with whole pages as stages a page's
// first tile kept its bytes until the second tile's product, and the ring's
// depth in flight is what paces the steady state (a tile lives ~9,000
// cycles from its copy's issue to its release).
//
// Warp roles (352 threads):
//   warp 0      TMA producer: tiles into the 8-stage ring, one page-table
//               read per page (and zeroes the rows past the end of a
//               partial last tile),
//   warp 1      TMEM owner; an elected lane issues each tile's S = Q.K^T as
//               soon as its tile has landed and its S buffer is free,
//   warp 2      an elected lane issues each tile's O += P.C, in tile order,
//               as soon as its P is in TMEM,
//   warps 3..6  tiles 0, 2, 4, ...: partial S -> peer, peer's partial ->
//               online softmax -> P into TMEM; lazy rescaling of O, the
//               query of a unit piece that starts on their tile, the
//               epilogue of one that ends on it,
//   warps 7..10 the same for tiles 1, 3, 5, ...
// The control warps wait with suspended (blocking) mbarrier waits, so they
// take no issue slots from the tile groups that share their sub-partitions.
// Each group covers the four TMEM lane quarters: thread (warp % 4) * 32 +
// lane owns head row h of the tile.
//
// Work split: the pages of all (sequence, token, head-group) units are laid
// end to end, with a few virtual pages charged for each unit boundary, and
// cut into equal contiguous ranges, one per cluster, so long and ragged
// sequences are spread over every SM.  A unit that straddles a range
// boundary is finished by each cluster as a partial (normalised o and its
// lse, fp32, in the workspace) and merged by a log-sum-exp combine kernel
// launched after this one.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "status.cuh"

namespace mla {
namespace dec {

constexpr int PAGE = 64;       // tokens per page (TMA unit)
constexpr int TILE = 32;       // tokens per score tile
constexpr int DC = 512;        // latent width
constexpr int DR = 64;         // RoPE key width
constexpr int HALF_C = 256;    // latent columns per CTA
constexpr int HALF_R = 32;     // RoPE columns per CTA
constexpr int HEADS = 128;     // heads per unit (UMMA M)
constexpr int NHS = 8;         // ring depth in half pages (one 32-token tile each)
constexpr int THREADS = 352;
constexpr int WG_WARP0 = 3;    // warps 3..6: tiles with even index, 7..10: odd

constexpr uint32_t HBOX_C_BYTES = TILE * 128;                      // 32 rows x 64 bf16
constexpr uint32_t HBOX_R_BYTES = TILE * 64;                       // 32 rows x 32 bf16
constexpr uint32_t HSTAGE_BYTES = 4 * HBOX_C_BYTES + HBOX_R_BYTES;  // 18432: one tile of a CTA's half
constexpr uint32_t XT_BYTES = HEADS * TILE * 4;                   // one partial S tile, fp32
constexpr uint32_t OFF_STAGE = 0;
constexpr uint32_t OFF_X = NHS * HSTAGE_BYTES;      // the peer's partial S tiles [group][slot]
constexpr uint32_t OFF_PUB = OFF_X + 4 * XT_BYTES;  // per-row state handed between the groups
constexpr uint32_t PUB_BYTES = 2 * 4 * HEADS * 4;      // [2 parities][m_used, m_ref, l_part, lr_part][128]
// This CTA's 32 RoPE columns of the query (128 rows x 64 B, the layout a
// 64-byte-swizzled TMA box would have): the A operand of the RoPE part of S.
constexpr uint32_t OFF_QPE = OFF_PUB + PUB_BYTES;      // 1 KB aligned
constexpr uint32_t QPE_BYTES = HEADS * HALF_R * 2;
constexpr uint32_t OFF_BAR = OFF_QPE + QPE_BYTES;
constexpr uint32_t NUM_BARS = 43;
constexpr uint32_t OFF_MISC = OFF_BAR + 8 * NUM_BARS;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 128;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;  // slack for 1 KB alignment

// TMEM: O (128 x 256 fp32), the latent query (128 x 256 bf16), three partial
// S buffers (tile i in i % 3, kept until its softmax has re-read it) and two
// P buffers (tile i in i % 2): 256 + 128 + 96 + 32 = all 512 columns.
constexpr int NS = 3;
constexpr uint32_t TM_O = 0, TM_Q = 256, TM_S = 384, TM_P = TM_S + 32 * NS, TM_COLS = 512;
static_assert(TM_P + 32 == TM_COLS, "TMEM map");
static_assert(OFF_QPE % 1024 == 0, "swizzled operand alignment");

// S = Q . K^T: M = 128 heads, N = 32 tokens, both operands K-major.
constexpr uint32_t IDESC_QK = idesc_bf16(128, TILE, false, false);
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
    __nv_bfloat16* o;            // [B, T, H, 512] bf16 output, or
    float* o32;                  // [B, T, H, 512] fp32 output (exactly one is set)
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
// Units u = ((b*T + t)*HG + hg) are laid end to end by their pages on a
// virtual line where each non-empty unit after the first is preceded by C
// virtual pages: starting a unit piece (the last piece's epilogue, the next
// query) costs a cluster about as much as C pages of attention, so a range
// that holds a unit boundary should get fewer real pages.  C is
// BOUNDARY_PAGES on lines of at least 8 pages per cluster and 0 otherwise.
// The line of V virtual positions is cut into G = min(clusters, total real
// pages) contiguous ranges, range g = [V*g/G, V*(g+1)/G), none of them
// without a real page (a range spans at least 8 positions when C > 0).  A
// unit cut by a range boundary is processed in pieces; piece (g, u) writes
// partial slot g + u, which is unique because both g and u only grow along
// the line.

struct PlanView {
    const int32_t* seq_lens;  // [B]
    int B, T, HG, max_pages, causal;
};

// Plan quantities (units, positions of the line, clusters, slots, tiles) are
// 32-bit: the host rejects shapes where B*T*HG*(max_pages + BOUNDARY_PAGES)
// or max_pages*64 reach 2^31, which bounds all of them.

constexpr int BOUNDARY_PAGES = 3;

// Virtual pages before each non-empty unit after the first.
__host__ __device__ __forceinline__ int boundary_pages(int total, int launched) {
    return total >= 8 * launched ? BOUNDARY_PAGES : 0;
}

// Length of the virtual line of `total` real pages in `units` non-empty units.
__host__ __device__ __forceinline__ int virtual_total(int total, int units, int C) {
    return units > 0 ? total + C * (units - 1) : 0;
}

// Line order of the units: u = (t * HG + hg) * B + b.  Each query token
// (and head group) of the batch is a stretch of the line of about the same
// length, so the clusters at the same offset of each stretch read the same
// pages at about the same time, and the later read of a page finds it in L2
// (with T query tokens a page is needed T times; one after another within a
// cluster's range, the reads would be some tens of microseconds apart, and
// most would miss).
__host__ __device__ __forceinline__ void unit_index(int u, int B, int HG, int& b, int& t, int& hg) {
    b = u % B;
    const int r = u / B;
    hg = r % HG;
    t = r / HG;
}

// Visible positions and pages of unit u.
struct Unit {
    int b, t, hg;
    int len;       // visible positions
    int pages;     // ceil(len / 64)
    bool bad_len;  // seq_lens[b] outside [0, max_pages * 64] (clamped)
};

__host__ __device__ __forceinline__ Unit unit_of(const PlanView& v, int u) {
    Unit r;
    unit_index(u, v.B, v.HG, r.b, r.t, r.hg);
    int len = v.seq_lens[r.b];
    const int cap = v.max_pages * PAGE;
    r.bad_len = len < 0 || len > cap;
    if (r.bad_len) len = len < 0 ? 0 : cap;
    const int n = v.causal ? len - (v.T - 1 - r.t) : len;
    r.len = n < 0 ? 0 : n;
    r.pages = (r.len + PAGE - 1) / PAGE;
    return r;
}

__host__ __device__ __forceinline__ int range_start(int total, int g, int G) {
    return (int)((int64_t)total * g / G);
}

// Clusters used for `total` pages when `launched` clusters run.
__host__ __device__ __forceinline__ int clusters_used(int total, int launched) {
    return total < launched ? total : launched;
}

// The range (cluster) holding position x of the line.
__host__ __device__ __forceinline__ int cluster_of_page(int x, int total, int G) {
    int g = (int)((int64_t)x * G / total);
    while (g + 1 < G && range_start(total, g + 1, G) <= x) ++g;
    while (g > 0 && range_start(total, g, G) > x) --g;
    return g;
}

// A piece of a unit processed by one cluster.
struct Segment {
    int u;
    int len;               // visible positions of the unit
    int lp0, lp1;          // page range within the unit
    int slot;              // partial slot, or -1 when the whole unit is here
    int g_first, g_last;   // clusters holding the unit's first and last page
};

// Walks the units overlapping cluster g's range, in line order (positions
// rs, re, total and pos are on the virtual line).
struct Walker {
    int U, rs, re, total, G, g, C;
    int u, pos;  // next unit and the position of its first page
    __host__ __device__ bool next(const PlanView& v, Segment& s) {
        if (rs >= re) return false;  // an empty range has no piece
        while (pos < re && u < U) {
            const Unit un = unit_of(v, u);
            const int cu = u++;
            if (un.pages == 0) continue;
            const int start = pos, end = pos + un.pages;
            pos = end + C;
            if (end <= rs) continue;
            s.u = cu;
            s.len = un.len;
            s.lp0 = (rs > start ? rs : start) - start;
            s.lp1 = (re < end ? re : end) - start;
            s.g_first = cluster_of_page(start, total, G);
            s.g_last = cluster_of_page(end - 1, total, G);
            s.slot = (s.g_first == s.g_last) ? -1 : g + cu;
            return true;
        }
        return false;
    }
};

// Walker of cluster g, found by a sequential scan (host side).
inline Walker host_walker(const PlanView& v, int launched, int g) {
    Walker w;
    w.U = v.B * v.T * v.HG;
    int total = 0, units = 0;
    for (int u = 0; u < w.U; ++u) {
        const int n = unit_of(v, u).pages;
        total += n;
        units += n > 0;
    }
    w.C = boundary_pages(total, launched);
    w.total = virtual_total(total, units, w.C);
    w.G = clusters_used(total, launched);
    w.g = g;
    w.rs = w.re = 0;
    w.u = w.U;
    w.pos = 0;
    if (total == 0 || g >= w.G) return w;
    w.rs = range_start(w.total, g, w.G);
    w.re = range_start(w.total, g + 1, w.G);
    int pos = 0;
    for (int u = 0; u < w.U; ++u) {
        const int n = unit_of(v, u).pages;
        if (n == 0) continue;
        if (w.rs < pos + n) {
            w.u = u;
            w.pos = pos;
            break;
        }
        pos += n + w.C;
    }
    return w;
}

// Host-side bound check for the 32-bit plan arithmetic.
inline bool plan_fits_int32(int B, int T, int HG, int max_pages) {
    return (int64_t)B * T * HG * (max_pages + BOUNDARY_PAGES) < ((int64_t)1 << 31) &&
           (int64_t)max_pages * PAGE < ((int64_t)1 << 31);
}

// Visible tokens of page lp of a segment's unit.
__device__ __forceinline__ int page_valid(const Segment& sg, int lp) {
    const int v = sg.len - lp * PAGE;
    return v < PAGE ? v : PAGE;
}

// Walks the tiles of a cluster's segments in order: pages of 64 tokens, each
// one or two tiles of 32 (a last page with at most 32 visible tokens has one).
// Every role of the kernel runs its own copy, so all agree on the sequence
// and on the global page / tile counters that select ring stages, buffers
// and barrier phases.
struct TileIter {
    Walker w;
    Segment sg;
    bool have;
    int seg, lp, page, tile;      // segment, page within the unit, global page and tile counters
    int t, ntp, pvalid;           // tile within the page, tiles in it, visible tokens in it

    __device__ void load_page() {
        pvalid = page_valid(sg, lp);
        ntp = pvalid > TILE ? 2 : 1;
        t = 0;
        ++page;
    }
    __device__ void begin(const Walker& w0, const PlanView& v) {
        w = w0;
        seg = -1;
        page = -1;
        tile = 0;
        have = w.next(v, sg);
        if (have) {
            seg = 0;
            lp = sg.lp0;
            load_page();
        }
    }
    __device__ void advance(const PlanView& v) {
        ++tile;
        if (t + 1 < ntp) {
            ++t;
            return;
        }
        if (lp + 1 < sg.lp1) {
            ++lp;
            load_page();
            return;
        }
        have = w.next(v, sg);
        if (have) {
            ++seg;
            lp = sg.lp0;
            load_page();
        }
    }
    __device__ int valid() const {
        const int v = pvalid - t * TILE;
        return v < TILE ? v : TILE;
    }
    __device__ bool first_in_seg() const { return lp == sg.lp0 && t == 0; }
    __device__ bool last_in_page() const { return t + 1 == ntp; }
    __device__ bool last_in_seg() const { return last_in_page() && lp + 1 == sg.lp1; }
    // ring stage of this tile (the half page it lies in) and the parity of
    // its phase of that stage's barriers
    __device__ int hstage() const { return tile % NHS; }
    __device__ uint32_t hparity() const { return (uint32_t)((tile / NHS) & 1); }
    __device__ int sbuf() const { return tile % NS; }  // TMEM partial S buffer
    // parity of the phase of an S-buffer barrier for the tile n back
    __device__ uint32_t s_parity(int back = 0) const { return (uint32_t)(((tile - back) / NS) & 1); }
    __device__ int buf() const { return (int)(tile & 1); }  // TMEM P buffer
    // parity of this tile's phase of a P-buffer barrier
    __device__ uint32_t parity() const { return (uint32_t)((tile >> 1) & 1); }
};

template <bool B>
struct BoolC {
    static constexpr bool value = B;
};

// What a tile group keeps of a tile between its two halves of work.
struct TileInfo {
    int tile, seg, u, slot, g_first, g_last, valid;
    bool first, last;
    __device__ void set(const TileIter& it) {
        tile = it.tile;
        seg = it.seg;
        u = it.sg.u;
        slot = it.sg.slot;
        g_first = it.sg.g_first;
        g_last = it.sg.g_last;
        valid = it.valid();
        first = it.first_in_seg();
        last = it.last_in_seg();
    }
};

// 11 warps share 4 register-file quarters (at most 3 warps each), so a
// thread may use at most 168 registers.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
decode_bf16_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_r,
                   const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // debug build: the page ring (written only by this CTA's own copies; the
    // exchange buffers, which the peer writes, are left alone)
    poison_smem(smem, OFF_X);
    const uint32_t bar0 = smem_u32(smem + OFF_BAR);
    auto BAR = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    // ring stage h (a half page): landed (TMA bytes), released (commit)
    auto FULL = [&](int h) { return h < 4 ? BAR(h) : BAR(35 + (h - 4)); };
    auto EMPTY = [&](int h) { return h < 4 ? BAR(4 + h) : BAR(39 + (h - 4)); };
    // Tile i's partial S is in S buffer i % 3 (the k-th use of a buffer is
    // phase k of its barriers), its P in P buffer i % 2.
    auto S_FULL = [&](int k) { return BAR(8 + k); };    // partial S of the buffer's tile (commit)
    auto S_FREE = [&](int k) { return BAR(11 + k); };   // re-read by the softmax (4 warps)
    auto P_FULL = [&](int b) { return BAR(14 + b); };   // P in TMEM (4 warps)
    auto PV_DONE = [&](int b) { return BAR(16 + b); };  // O += P.C of that tile (commit)
    // the peer's partial tile i lands in X[i % 2][(i / 2) % 2]: x = 2 * (i % 2) + (i / 2) % 2
    auto XFULL = [&](int x) { return BAR(18 + x); };    // peer partial in X (1 arrive + bytes)
    auto XFREE = [&](int x) { return BAR(22 + x); };    // peer done with our copy (4 peer warps)
    auto M_PUB = [&](int b) { return BAR(26 + b); };    // running max after the tile (4 warps)
    auto L_PUB = [&](int b) { return BAR(28 + b); };    // group's row sums after the tile (4 warps)
    const uint32_t Q_FULL = BAR(30);                    // query of a unit in TMEM + smem (4 warps)
    const uint32_t O_FREE = BAR(31);                    // epilogue read O (4 warps)
    const uint32_t TAIL = BAR(32);                      // partial last tile landed (TMA)
    auto DRAIN = [&](int k) { return BAR(33 + k); };    // teardown: MMAs of warp 1 + k finished
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    int64_t* misc = reinterpret_cast<int64_t*>(smem + OFF_MISC + 8);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NHS; ++s) {
            mbar_init(FULL(s), 1);
            mbar_init(EMPTY(s), 1);
        }
        for (int k = 0; k < NS; ++k) {
            mbar_init(S_FULL(k), 1);
            mbar_init(S_FREE(k), 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(P_FULL(b), 4);
            mbar_init(PV_DONE(b), 1);
            mbar_init(M_PUB(b), 4);
            mbar_init(L_PUB(b), 4);
        }
        for (int x = 0; x < 4; ++x) {
            mbar_init(XFULL(x), 1);
            mbar_init(XFREE(x), 4);
        }
        mbar_init(Q_FULL, 4);
        mbar_init(O_FREE, 4);
        mbar_init(TAIL, 1);
        for (int k = 0; k < 2; ++k) mbar_init(DRAIN(k), 1);
        fence_mbar_init_cluster();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_c);
        tma_prefetch_desc(&tm_r);
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TM_COLS);
    // This CTA's barriers are initialised (thread 0, fenced above): its half
    // of the cluster barrier is passed now, and the wait for the peer's half
    // comes after the plan, before any remote access, so the round trip
    // overlaps the plan instead of following it.
    cluster_arrive_relaxed();

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
    if (warp == 0) {
        // Warp 0 sums the pages (and counts the non-empty units) of
        // contiguous chunks of units and scans them with shuffles; then each
        // lane walks its units again on the virtual line, the first unit that
        // reaches into the range is recorded, and all lanes count the range's
        // tiles: two per page, less one for each unit whose last page lies in
        // the range with at most TILE visible tokens.
        const int64_t chunk = (U + 31) / 32;
        const int64_t u0 = min(U, (int64_t)lane * chunk), u1 = min(U, u0 + chunk);
        int64_t sum = 0, cnt = 0;
        bool bad = false;
        for (int64_t u = u0; u < u1; ++u) {
            const Unit un = unit_of(pv, u);
            sum += un.pages;
            cnt += un.pages > 0;
            bad |= un.bad_len;
        }
        if (bad && rank == 0 && g_id == 0) raise_device_status(MLA_DEV_BOUNDS, 0x10);
        int64_t incl = sum, incl_cnt = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
            const int64_t vc = __shfl_up_sync(0xffffffffu, incl_cnt, o);
            if (lane >= o) {
                incl += v;
                incl_cnt += vc;
            }
        }
        const int64_t total = __shfl_sync(0xffffffffu, incl, 31);
        const int64_t units = __shfl_sync(0xffffffffu, incl_cnt, 31);
        const int C = boundary_pages((int)total, (int)launched);
        const int64_t V = virtual_total((int)total, (int)units, C);
        if (lane == 0) {
            misc[0] = V;      // virtual positions of the line
            misc[1] = U;      // first unit of this cluster's range (default: none)
            misc[2] = 0;
            misc[3] = device_status_raised() ? 1 : 0;  // one decision for the whole CTA
            misc[4] = C;
            misc[5] = total;  // real pages
        }
        __syncwarp();
        const int64_t G = clusters_used(total, launched);
        const int64_t rs = g_id < G ? range_start(V, g_id, G) : V;
        const int64_t re = g_id < G ? range_start(V, g_id + 1, G) : V;
        int64_t tiles = 0, first_u = -1, first_pos = 0;
        int64_t pos = (incl - sum) + C * (incl_cnt - cnt);  // the chunk's first non-empty unit
        if (rs < re) {
            for (int64_t u = u0; u < u1 && pos < re; ++u) {
                const Unit un = unit_of(pv, u);
                if (un.pages == 0) continue;
                const int64_t s0 = pos, s1 = pos + un.pages;
                pos = s1 + C;
                if (s1 <= rs) continue;
                if (first_u < 0) {
                    first_u = u;
                    first_pos = s0;
                }
                tiles += 2 * (min(s1, re) - max(s0, rs));
                if (s1 <= re && un.len - (un.pages - 1) * PAGE <= TILE) tiles -= 1;
            }
        }
        const uint32_t found = __ballot_sync(0xffffffffu, first_u >= 0);
        if (found != 0u && lane == __ffs(found) - 1) {  // the lowest lane's is the range's first
            misc[1] = first_u;
            misc[2] = first_pos;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tiles += __shfl_xor_sync(0xffffffffu, tiles, o);
        if (lane == 0) misc[6] = misc[3] ? 0 : tiles;
    }
    __syncthreads();  // misc[1], misc[2] (the range's first unit) are written above
    Walker walk;
    walk.U = U;
    walk.total = misc[0];
    walk.C = (int)misc[4];
    walk.G = clusters_used(misc[5], launched);
    walk.g = g_id;
    walk.rs = g_id < walk.G ? range_start(walk.total, g_id, walk.G) : 0;
    walk.re = g_id < walk.G ? range_start(walk.total, g_id + 1, walk.G) : 0;
    walk.u = misc[1];
    walk.pos = misc[2];
    const bool skip = misc[3] != 0;
    if (warp == 2 && lane == 0 && !skip) {
        // The queries of this cluster's unit pieces, into L2 ahead of the
        // tile groups' loads (each piece's load is on the critical path).
        Walker w = walk;
        Segment sg;
        while (w.next(pv, sg)) {
            int ub, ut, uh;
            unit_index(sg.u, p.B, p.HG, ub, ut, uh);
            const int bt = ub * p.T + ut;  // row of q, o
            const int head0 = uh * HEADS;
            const int rows = min(HEADS, p.H - head0);
            const int64_t qrow0 = (int64_t)bt * p.H + head0;
            bulk_prefetch_l2(p.q_lat + qrow0 * DC, (uint32_t)rows * DC * 2u);
            bulk_prefetch_l2(p.q_pe + qrow0 * DR, (uint32_t)rows * DR * 2u);
        }
    }
    if (threadIdx.x == 0) {
        // The peer's partial tiles 0..3 land in the four X buffers; later
        // tiles are armed by the groups as they consume these.
        const int64_t n = misc[6];
        for (int64_t i = 0; i < n && i < 4; ++i)
            mbar_arrive_expect_tx(XFULL((int)(2 * (i & 1) + ((i >> 1) & 1))), XT_BYTES);
        for (int g = 0; g < 2; ++g) {
            misc[7 + g] = n < 4 ? n : 4;  // group g: tiles below this were armed
            misc[9 + g] = 0;              // ... and its tiles below this consumed
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // The peer's barriers are initialised before any remote access (their
    // arming needs no order: transaction bytes may land before it).
    cluster_wait();
    const uint32_t tmem = *tmem_slot;
    const int64_t n_tiles = misc[6];

    if (warp == 0) {
        // ========================================================= producer
        // A page read once can leave L2 first; a page every query token (and
        // head group) of its sequence reads -- the next unit, a cluster or
        // two away on the line, reads it some 20 pages later -- stays.
        const uint64_t pol = p.T * p.HG > 1 ? l2_policy_evict_last() : l2_policy_evict_first();
        int64_t it = 0;
        uint32_t tail_phase = 0;
        bool ok = !skip;
        Segment sg;
        while (ok && walk.next(pv, sg)) {
            // debug build: the piece lies in its unit, in this cluster, and
            // has a slot exactly when its unit is cut
            check_split(sg.lp0 >= 0 && sg.lp0 < sg.lp1 && (int64_t)sg.lp1 * PAGE < (int64_t)sg.len + PAGE &&
                            sg.g_first <= (int)g_id && (int)g_id <= sg.g_last && sg.g_last < (int)launched &&
                            (sg.slot < 0) == (sg.g_first == sg.g_last) && sg.slot < (int)(launched + U),
                        0x70);
            for (int64_t lp = sg.lp0; lp < sg.lp1 && ok; ++lp) {
                const int b_seq = sg.u % p.B;  // unit u = (t * HG + hg) * B + b
                int64_t pg = p.page_table[(int64_t)b_seq * p.max_pages + lp];
                if (pg < 0 || pg >= p.num_pages) {
                    raise_device_status(MLA_DEV_BOUNDS, 0x20);
                    pg = 0;
                }
                const int valid = page_valid(sg, lp);
                const int ntp = valid > TILE ? 2 : 1;  // the tiles the consumers take from this page
                // Each tile of the page has its own ring stage (half a page),
                // so a stage goes back to the ring as soon as its tile's
                // O product is done, not its page's second tile's.
                for (int t = 0; t < ntp && ok; ++t, ++it) {
                    const int h = (int)(it % NHS);
                    ok = mbar_wait(EMPTY(h), (uint32_t)((it / NHS) & 1) ^ 1u, 0x201);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    const int y = (int)(pg * PAGE) + t * TILE;
                    const int vt = min(TILE, valid - t * TILE);  // visible rows of this tile
                    const uint32_t st = smem_u32(smem + OFF_STAGE + h * HSTAGE_BYTES);
                    const uint32_t bar = vt == TILE ? FULL(h) : TAIL;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(bar, HSTAGE_BYTES);
                        for (int k = 0; k < 4; ++k)
                            tma_load_2d(st + k * HBOX_C_BYTES, &tm_c, bar, (int)rank * HALF_C + 64 * k, y, pol);
                        tma_load_2d(st + 4 * HBOX_C_BYTES, &tm_r, bar, DC + (int)rank * HALF_R, y, pol);
                    }
                    if (vt < TILE) {
                        // Rows past the end may hold anything (even NaN); zero
                        // them so that P = 0 there cannot meet a NaN in P . C.
                        // (The copy was issued here, so it is waited for even
                        // when another CTA has raised the status word.)
                        ok = mbar_wait_teardown(TAIL, tail_phase, MLA_WAIT_LIMIT_NS);
                        ok = __all_sync(0xffffffffu, ok);
                        tail_phase ^= 1u;
                        if (!ok) {
                            raise_device_status(MLA_DEV_TIMEOUT, 0x202u | ((blockIdx.x & 0xFFFu) << 12));
                            ++it;
                            break;
                        }
                        uint8_t* tile = smem + OFF_STAGE + h * HSTAGE_BYTES;
                        const int rows = TILE - vt;
                        for (int idx = lane; idx < rows * 8 * 4; idx += 32) {  // latent boxes
                            const int box = idx / (rows * 8), rem = idx % (rows * 8);
                            uint4* dst = reinterpret_cast<uint4*>(tile + box * HBOX_C_BYTES +
                                                                  (vt + rem / 8) * 128 + (rem % 8) * 16);
                            *dst = make_uint4(0u, 0u, 0u, 0u);
                        }
                        for (int idx = lane; idx < rows * 4; idx += 32) {  // RoPE box
                            uint4* dst = reinterpret_cast<uint4*>(tile + 4 * HBOX_C_BYTES +
                                                                  (vt + idx / 4) * 64 + (idx % 4) * 16);
                            *dst = make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(FULL(h));
                    }
                }
            }
        }
        // Every copy this warp issued lands before the CTA can exit, on the
        // normal path (where these phases have completed long ago) and after
        // an abort alike.  A partial page's FULL phase is this warp's own
        // arrive, made above once its copy had landed.  (The tensor core's
        // releases of the ring are waited for by the MMA warps themselves.)
        for (int64_t i = (it > NHS ? it - NHS : 0); i < it; ++i)
            mbar_wait_teardown(FULL((int)(i % NHS)), (uint32_t)((i / NHS) & 1), MLA_WAIT_LIMIT_NS);
    } else if (warp == 1) {
        // ========================================================= MMA: S
        // The score products S = Q.K^T, tile by tile, each as soon as its
        // page has landed, its S buffer has been read and (at the start of a
        // unit) the query is in TMEM.  One elected lane of the converged
        // warp issues them.
        TileIter qk;
        qk.begin(walk, pv);
        bool ok = !skip;
        bool issued = false;
        const uint64_t dq0 = smem_desc(smem_u32(smem + OFF_STAGE), 16, 1024, SWZ_128B);
        const uint64_t dr0 = smem_desc(smem_u32(smem + OFF_STAGE + 4 * HBOX_C_BYTES), 16, 512, SWZ_64B);
        const uint64_t dqpe = smem_desc(smem_u32(smem + OFF_QPE), 16, 512, SWZ_64B);
        while (ok && qk.have) {
            const int k3 = qk.sbuf();
            ok = __all_sync(0xffffffffu, mbar_wait(FULL(qk.hstage()), qk.hparity(), 0x301));
            // the softmax has re-read the buffer's last tile (three back)
            if (ok && qk.tile >= NS) ok = __all_sync(0xffffffffu, mbar_wait(S_FREE(k3), qk.s_parity(NS), 0x302));
            if (ok && qk.first_in_seg())
                ok = __all_sync(0xffffffffu, mbar_wait(Q_FULL, (uint32_t)(qk.seg & 1), 0x303));
            if (!ok) break;
            tc_fence_after();
            if (elect_one_sync()) {
                const uint32_t off = (uint32_t)(qk.hstage() * HSTAGE_BYTES);
                const uint64_t dc = dq0 + ((uint64_t)off >> 4);
                const uint64_t dr = dr0 + ((uint64_t)off >> 4);
                const uint32_t d = tmem + TM_S + 32 * k3;
#pragma unroll
                for (int k = 0; k < 16; ++k)  // latent features, K-major SW128
                    mma_ts(d, tmem + TM_Q + 8 * k, dc + (uint64_t)(((k / 4) * HBOX_C_BYTES + (k % 4) * 32) >> 4),
                           IDESC_QK, k > 0 ? 1u : 0u);
#pragma unroll
                for (int k = 0; k < 2; ++k)  // RoPE features, both operands K-major SW64 in smem
                    mma_ss(d, dqpe + (uint64_t)((k * 32) >> 4), dr + (uint64_t)((k * 32) >> 4), IDESC_QK, 1u);
                tc_commit(S_FULL(k3));
            }
            __syncwarp();
            issued = true;
            qk.advance(pv);
        }
        if (issued) {  // every product (and its commits) done before TMEM goes away
            if (elect_one_sync()) tc_commit(DRAIN(0));
            __syncwarp();
            mbar_wait_teardown(DRAIN(0), 0, MLA_WAIT_LIMIT_NS);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ========================================================= MMA: O
        // O += P.C, tile by tile in order (one issuing thread, so the
        // products land in tile order and every call gives the same bits),
        // each as soon as its P is in TMEM and, for a unit's first tile
        // (which overwrites O), once the last unit's epilogue has read O.
        TileIter it;
        it.begin(walk, pv);
        bool ok = !skip;
        bool issued = false;
        const uint64_t dp0 = smem_desc(smem_u32(smem + OFF_STAGE), HBOX_C_BYTES, 1024, SWZ_128B);
        while (ok && it.have) {
            const int b = it.buf();
            ok = __all_sync(0xffffffffu, mbar_wait(P_FULL(b), it.parity(), 0x401));
            if (ok && it.first_in_seg() && it.seg > 0)
                ok = __all_sync(0xffffffffu, mbar_wait(O_FREE, (uint32_t)((it.seg - 1) & 1), 0x402));
            if (!ok) break;
            tc_fence_after();
            if (elect_one_sync()) {
                // C as MN-major B: 64-column boxes 8 KB apart, 8-row
                // groups 1 KB apart, 16 tokens = 2 KB per step.
                const uint64_t db = dp0 + ((uint64_t)(it.hstage() * HSTAGE_BYTES) >> 4);
                const uint32_t acc0 = it.first_in_seg() ? 0u : 1u;
#pragma unroll
                for (int k = 0; k < TILE / 16; ++k)
                    mma_ts(tmem + TM_O, tmem + TM_P + 16 * b + 8 * k, db + (uint64_t)(k * 2048 >> 4), IDESC_PV,
                           k == 0 ? acc0 : 1u);
                tc_commit(PV_DONE(b));
                tc_commit(EMPTY(it.hstage()));
            }
            __syncwarp();
            issued = true;
            it.advance(pv);
        }
        if (issued) {  // every product (and its commits) done before TMEM goes away
            if (elect_one_sync()) tc_commit(DRAIN(1));
            __syncwarp();
            mbar_wait_teardown(DRAIN(1), 0, MLA_WAIT_LIMIT_NS);
        }
        __syncwarp();
    } else {
        // ===================================================== tile groups
        // A group's tiles are software-pipelined: the front half of its next
        // tile (query if a unit starts there, own partial scores out of TMEM
        // and off to the peer) runs before the back half of its current one
        // (own partial again from TMEM, the peer's from X, softmax, P,
        // epilogue), so the exchange of one tile overlaps the softmax of the
        // one before.
        const int grp = (warp - WG_WARP0) / 4;  // tiles with index % 2 == grp
        const int b = grp;                      // their P buffers and barriers
        const int q4 = warp & 3;
        const int h = q4 * 32 + lane;
        const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
        const uint32_t peer_x0 = map_to_rank(smem_u32(smem + OFF_X + 2 * grp * XT_BYTES), peer);
        const uint32_t peer_xfull0 = map_to_rank(XFULL(2 * grp), peer);
        float* pub = reinterpret_cast<float*>(smem + OFF_PUB);  // [2][4][HEADS]
        const bool leader = warp == WG_WARP0 + 4 * grp && lane == 0;
        const int my_g = (int)g_id;
        auto xslot = [](int i) { return (i >> 1) & 1; };
        auto xpar = [](int i) { return (uint32_t)((i >> 2) & 1); };
        auto s_par = [](int i) { return (uint32_t)((i / NS) & 1); };  // tile i's phase of its S buffer
        bool ok = !skip;
        // this group's row sums, relative to m_ref: of the exact exponentials
        // (for lse) and of their bf16 roundings, the weights P . C applies
        // (for o = P.C / lr: a weighted mean whose weights sum to exactly 1,
        // so the rounding of a row that dominates the softmax cancels)
        float m_ref = -INFINITY, l_part = 0.f, lr_part = 0.f;
        int64_t my_seg = -1;
        int64_t armed = misc[7 + grp], consumed = 0;

        // ---- front half of tile `t`
        auto front = [&](const TileIter& t, auto may_start) -> bool {
            const int i = t.tile;
            if constexpr (decltype(may_start)::value) if (t.first_in_seg()) {
                // The query of this unit replaces the last one once every
                // score product of the tile before has completed.
                if (i >= 1 && !__all_sync(0xffffffffu, mbar_wait(S_FULL((i - 1) % NS), s_par(i - 1), 0x501)))
                    return false;
                int ub, ut, uh;
                unit_index(t.sg.u, p.B, p.HG, ub, ut, uh);
                const int bt = ub * p.T + ut;  // row of q, o
                const int head = uh * HEADS + h;
                const bool live = head < p.H;
                const int64_t qrow = (int64_t)bt * p.H + head;
                const uint4* ql = reinterpret_cast<const uint4*>(p.q_lat + qrow * DC + rank * HALF_C);
                const uint4* qp = reinterpret_cast<const uint4*>(p.q_pe + qrow * DR + rank * HALF_R);
                // The RoPE columns and the first 128 latent columns are
                // loaded together (one round trip instead of two), then the
                // other 128.
                uint4 v[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) v[c] = live ? __ldg(qp + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int half = 0; half < 2; ++half) {  // latent columns into TMEM, 128 at a time
                    uint32_t r[64];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const uint4 x = live ? __ldg(ql + 16 * half + k) : make_uint4(0u, 0u, 0u, 0u);
                        r[4 * k] = x.x;
                        r[4 * k + 1] = x.y;
                        r[4 * k + 2] = x.z;
                        r[4 * k + 3] = x.w;
                    }
                    if (half == 0) {  // RoPE columns into shared memory: row h, 16-byte chunk c
                                      // at chunk c ^ ((h / 2) % 4) of its 64 bytes (64-byte swizzle)
                        uint8_t* row = smem + OFF_QPE + h * 64;
#pragma unroll
                        for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(row + 16 * (c ^ ((h >> 1) & 3))) = v[c];
                    }
                    tmem_st32(trow + TM_Q + 64 * half, *reinterpret_cast<const uint32_t(*)[32]>(r));
                    tmem_st32(trow + TM_Q + 64 * half + 32, *reinterpret_cast<const uint32_t(*)[32]>(r + 32));
                }
                tmem_st_wait();
                fence_proxy_async_smem();  // the RoPE rows, to the tensor core
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(Q_FULL);
            }
            const int k3 = i % NS;
            if (!__all_sync(0xffffffffu, mbar_wait(S_FULL(k3), s_par(i), 0x502))) return false;
            tc_fence_after();
            uint32_t r[TILE];
            tmem_ld32(trow + TM_S + 32 * k3, r);
            // our copy of this group's tile four back is done with at the peer
            if (i >= 4 && !__all_sync(0xffffffffu, mbar_wait(XFREE(2 * grp + xslot(i)), xpar(i - 4), 0x503)))
                return false;
            const uint32_t dst = peer_x0 + (uint32_t)xslot(i) * XT_BYTES;
            const uint32_t pbar = peer_xfull0 + 8u * (uint32_t)xslot(i);
#pragma unroll
            for (int k = 0; k < TILE / 4; ++k)
                st_async_v4(dst + (uint32_t)(k * HEADS + h) * 16u, r[4 * k], r[4 * k + 1], r[4 * k + 2], r[4 * k + 3], pbar);
            return true;
        };

        // ---- own partial scores of tile `c`, again from its buffer (the
        // front half waited for them), taken at the start of the group's
        // iteration: the buffer is free for tile c + 3 once all four warps
        // have them.  The loads have completed (the wait is part of
        // tmem_ld32) and no memory write is published, so the arrive is
        // relaxed.
        uint32_t own[TILE];
        auto load_own = [&](const TileInfo& c) {
            const int k3 = c.tile % NS;
            tmem_ld32(trow + TM_S + 32 * k3, own);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(S_FREE(k3));
        };

        // ---- back half of tile `c`, whose own partial scores are in `own`
        auto back = [&](const TileInfo& c, auto may_end) -> bool {
            const int i = c.tile;
            if (my_seg != c.seg) {  // a new unit piece: this group's sums restart
                my_seg = c.seg;
                m_ref = -INFINITY;
                l_part = 0.f;
                lr_part = 0.f;
            }
            const int x = 2 * grp + xslot(i);
            if (!__all_sync(0xffffffffu, mbar_wait(XFULL(x), xpar(i), 0x504))) return false;
            consumed = i + 1;
            if (leader && i + 4 < n_tiles) {
                mbar_arrive_expect_tx(XFULL(x), XT_BYTES);  // this buffer next receives tile i + 4
                armed = i + 5;
            }
            uint8_t* xbuf = smem + OFF_X + x * XT_BYTES;
            // unscaled scores as packed pairs: own + peer partial (the scale
            // scale * log2(e) > 0 is applied to the maximum here and inside
            // the exponent's fused multiply-add below)
            const ulonglong2* xp = reinterpret_cast<const ulonglong2*>(xbuf);
            uint64_t s2[TILE / 2];
#pragma unroll
            for (int k = 0; k < TILE / 4; ++k) {
                const ulonglong2 v = xp[k * HEADS + h];
                s2[2 * k] = f2_add(f2_pack(__uint_as_float(own[4 * k]), __uint_as_float(own[4 * k + 1])), v.x);
                s2[2 * k + 1] = f2_add(f2_pack(__uint_as_float(own[4 * k + 2]), __uint_as_float(own[4 * k + 3])), v.y);
            }
            if (c.valid < TILE) {  // only a unit's last tile has positions past the end
#pragma unroll
                for (int j = 0; j < TILE / 2; ++j)
                    s2[j] = f2_pack(2 * j < c.valid ? f2_lo(s2[j]) : -INFINITY, 2 * j + 1 < c.valid ? f2_hi(s2[j]) : -INFINITY);
            }
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int j = 0; j < TILE / 2; ++j) mx4[j & 3] = fmax3(mx4[j & 3], f2_lo(s2[j]), f2_hi(s2[j]));
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * p.scale_log2;
            // Every value read from this X buffer is in registers: it goes back
            // to the peer now -- except at a piece's end, where the epilogue
            // stages its rows there first (the last tile always takes the
            // epilogue-compiled path).
            __syncwarp();
            if (!c.last && lane == 0) mbar_arrive_remote_relaxed(map_to_rank(XFREE(x), peer));
            // ---- the running maximum after the tile before (the other group)
            float m_prev = -INFINITY;
            if (i >= 1) {
                if (!__all_sync(0xffffffffu, mbar_wait(M_PUB(b ^ 1), (uint32_t)(((i - 1) >> 1) & 1), 0x505)))
                    return false;
                m_prev = pub[(b ^ 1) * 4 * HEADS + h];
            }
            float m_oth = -INFINITY, l_oth = 0.f, lr_oth = 0.f;  // the other group's sums (unit's last tile only)
            if (c.last && !c.first) {
                // before this tile's maximum is published, so that the other
                // group cannot publish its next tile's sums over these
                if (!__all_sync(0xffffffffu, mbar_wait(L_PUB(b ^ 1), (uint32_t)(((i - 1) >> 1) & 1), 0x506)))
                    return false;
                m_oth = pub[((b ^ 1) * 4 + 1) * HEADS + h];
                l_oth = pub[((b ^ 1) * 4 + 2) * HEADS + h];
                lr_oth = pub[((b ^ 1) * 4 + 3) * HEADS + h];
            }
            float m_used;
            bool need = false;
            if (c.first) {
                m_used = mx;
            } else {
                need = mx > m_prev + RESCALE_THRESHOLD;
                m_used = need ? mx : m_prev;
            }
            bool p_free = i < 2;
            if (__any_sync(0xffffffffu, need)) {
                // O moves to the new maximum once the tile before has been
                // added to it (and with it every earlier one: the products
                // land in tile order), and before any later tile is.  The
                // product two back is waited for first: then the other
                // parity's barrier has only the tile before outstanding.
                if (!p_free && !__all_sync(0xffffffffu, mbar_wait(PV_DONE(b), (uint32_t)(((i - 2) >> 1) & 1), 0x508)))
                    return false;
                p_free = true;
                if (!__all_sync(0xffffffffu, mbar_wait(PV_DONE(b ^ 1), (uint32_t)(((i - 1) >> 1) & 1), 0x507)))
                    return false;
                tc_fence_after();
                const float alpha = ex2(m_prev - m_used);
#pragma unroll 1
                for (int cc = 0; cc < HALF_C; cc += 32) {
                    uint32_t r[32];
                    tmem_ld32(trow + TM_O + cc, r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
                    tmem_st32(trow + TM_O + cc, r);
                }
                tmem_st_wait();
                tc_fence_before();
            }
            pub[b * 4 * HEADS + h] = m_used;
            __syncwarp();
            if (lane == 0) mbar_arrive(M_PUB(b));
            if (m_ref != m_used) {  // this group's earlier sums, to the new reference
                const float f = m_ref == -INFINITY ? 0.f : ex2(m_ref - m_used);
                l_part *= f;
                lr_part *= f;
                m_ref = m_used;
            }
            // ---- P[b] is free once the tile two back has been multiplied
            if (!p_free) {
                if (!__all_sync(0xffffffffu, mbar_wait(PV_DONE(b), (uint32_t)(((i - 2) >> 1) & 1), 0x508)))
                    return false;
                tc_fence_after();
            }
            {
                uint32_t pk[TILE / 2];
                const uint64_t nm2 = f2_pack(-m_used, -m_used);
                const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
                uint64_t sum2 = 0ull, sumr2 = 0ull;
#pragma unroll
                for (int j = 0; j < TILE / 2; ++j) {
                    const uint64_t e = f2_fma(s2[j], c2, nm2);  // s * scale * log2(e) - m
                    const float p0 = ex2(f2_lo(e));
                    const float p1 = ex2(f2_hi(e));
                    pk[j] = pack_bf16x2(p0, p1);
                    sum2 = f2_add(sum2, f2_pack(p0, p1));
                    sumr2 = f2_add(sumr2, bf16x2_to_f2(pk[j]));
                }
                l_part += f2_lo(sum2) + f2_hi(sum2);
                lr_part += f2_lo(sumr2) + f2_hi(sumr2);
                tmem_st16(trow + TM_P + 16 * b, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            pub[(b * 4 + 1) * HEADS + h] = m_ref;
            pub[(b * 4 + 2) * HEADS + h] = l_part;
            pub[(b * 4 + 3) * HEADS + h] = lr_part;
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(P_FULL(b));
                mbar_arrive(L_PUB(b));
            }
            if constexpr (decltype(may_end)::value) if (c.last) {
                // ---- epilogue: O / l of this CTA's 256 columns, lse.  O is
                // complete once this tile's product is (the products land in
                // tile order).
                if (!__all_sync(0xffffffffu, mbar_wait(PV_DONE(b), (uint32_t)((i >> 1) & 1), 0x509))) return false;
                tc_fence_after();
                const float f_oth = c.first ? 0.f : ex2(m_oth - m_used);
                const float l = l_part + l_oth * f_oth;     // for lse
                const float lr = lr_part + lr_oth * f_oth;  // for o
                int ub, ut, uh;
                unit_index(c.u, p.B, p.HG, ub, ut, uh);
                const int bt = ub * p.T + ut;  // row of q, o
                const int head0 = uh * HEADS + q4 * 32;  // head of this warp's row 0
                const int64_t qrow0 = (int64_t)bt * p.H + head0;
                const float inv_l = 1.f / lr;
                // Rows go out through this tile's X buffer (the 4 KB this warp
                // read): each thread puts its row's 16-byte chunks in, then the
                // warp stores whole 64- or 128-byte row pieces per instruction
                // instead of 32 scattered 16-byte ones.  Chunk j of row r sits
                // in slot (r + j) % 8 of its 8-slot group, which keeps both
                // passes free of bank conflicts.
                auto stg = [&](int r, int j) -> uint4* {
                    return reinterpret_cast<uint4*>(xbuf + j * (HEADS * 16) + q4 * 512 + 16 * ((r & 24) | ((r + j) & 7)));
                };
                if (c.slot < 0 && p.o32 == nullptr) {
                    __nv_bfloat16* dst = p.o + qrow0 * DC + rank * HALF_C + 8 * (lane & 3);
#pragma unroll 1
                    for (int cc = 0; cc < HALF_C; cc += 32) {
                        uint32_t r[32];
                        tmem_ld32(trow + TM_O + cc, r);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            *stg(lane, v) = make_uint4(
                                pack_bf16x2(__uint_as_float(r[8 * v]) * inv_l, __uint_as_float(r[8 * v + 1]) * inv_l),
                                pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv_l, __uint_as_float(r[8 * v + 3]) * inv_l),
                                pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv_l, __uint_as_float(r[8 * v + 5]) * inv_l),
                                pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv_l, __uint_as_float(r[8 * v + 7]) * inv_l));
                        __syncwarp();
                        // the pieces are read first, then stored back to back
                        // (a read before each store ran the stores ~3x slower)
                        uint4 piece[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) piece[k] = *stg(8 * k + (lane >> 2), lane & 3);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {  // 8 rows x 64 bytes per store
                            const int row = 8 * k + (lane >> 2);
                            if (head0 + row < p.H) *reinterpret_cast<uint4*>(dst + (int64_t)row * DC + cc) = piece[k];
                        }
                        __syncwarp();
                    }
                    if (head0 + lane < p.H && rank == 0) p.lse[qrow0 + lane] = (m_used + __log2f(l)) * LN2;
                } else {
                    // fp32 rows: the unit's partial result in its workspace
                    // slot, or (fp32 output) the unit's own rows of o
                    const bool direct = c.slot < 0;
                    float* dst = (direct ? p.o32 + qrow0 * DC : p.ws_o + (int64_t)(c.slot * HEADS + q4 * 32) * DC) +
                                 rank * HALF_C + 4 * (lane & 7);
                    const int live_rows = direct ? min(32, p.H - head0) : 32;
#pragma unroll 1
                    for (int cc = 0; cc < HALF_C; cc += 32) {
                        uint32_t r[32];
                        tmem_ld32(trow + TM_O + cc, r);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            *stg(lane, v) = make_uint4(__float_as_uint(__uint_as_float(r[4 * v]) * inv_l),
                                                       __float_as_uint(__uint_as_float(r[4 * v + 1]) * inv_l),
                                                       __float_as_uint(__uint_as_float(r[4 * v + 2]) * inv_l),
                                                       __float_as_uint(__uint_as_float(r[4 * v + 3]) * inv_l));
                        __syncwarp();
                        uint4 piece[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) piece[k] = *stg(4 * k + (lane >> 3), lane & 7);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {  // 4 rows x 128 bytes per store
                            const int row = 4 * k + (lane >> 3);
                            if (row < live_rows) *reinterpret_cast<uint4*>(dst + (int64_t)row * DC + cc) = piece[k];
                        }
                        __syncwarp();
                    }
                    const float lse_v = (m_used + __log2f(l)) * LN2;
                    if (rank == 0) {
                        if (!direct) p.ws_lse[c.slot * HEADS + h] = lse_v;
                        else if (lane < live_rows) p.lse[qrow0 + lane] = lse_v;
                    }
                }
                if (rank == 0 && h == 0 && c.g_first == my_g)
                    p.ws_unit[c.u] = make_int2((int)c.g_first, c.g_last);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(O_FREE);
                    mbar_arrive_remote_relaxed(map_to_rank(XFREE(x), peer));  // staging done
                }
            }
            return true;
        };

        TileIter it;
        it.begin(walk, pv);
        if (it.have && (it.tile & 1) != grp) it.advance(pv);  // this group's first tile
        TileInfo cur;
        bool have_cur = false;
        if (ok && it.have) {
            ok = front(it, BoolC<true>{});
            cur.set(it);
            have_cur = true;
            it.advance(pv);
            if (it.have) it.advance(pv);
        }
        // `it` now points at the group's next tile.  Within a unit piece its
        // front half runs before the back half of `cur`, so the exchange of
        // one tile overlaps the softmax of the one before.  Where the piece
        // changes the back half goes first: the front half of a piece's first
        // tile loads the query and everything after it waits for that query's
        // scores, so the old piece's epilogue then overlaps the query load
        // instead of following it.  (A piece's last tile is always followed
        // by another piece or by nothing, so only that order needs the
        // epilogue, and only it the query load.)
        while (ok && have_cur) {
            load_own(cur);
            if (!it.have || it.seg != cur.seg) {
                ok = back(cur, BoolC<true>{});
                if (!ok || !it.have) break;
                ok = front(it, BoolC<true>{});
            } else {  // same piece: `it` does not start one
                ok = front(it, BoolC<false>{});
                if (!ok) break;
                ok = back(cur, BoolC<false>{});
            }
            if (!ok) break;
            cur.set(it);
            it.advance(pv);
            if (it.have) it.advance(pv);
        }
        if (leader) {
            misc[7 + grp] = armed;
            misc[9 + grp] = consumed;
        }

    }

    tc_fence_before();
    __syncthreads();
    // Teardown: partial S tiles the peer may still be copying into X land
    // before this CTA's shared memory can go away (only after an abort can
    // one be armed but not consumed; each wait gives up after 10 ms).
    if (threadIdx.x == 0) {
        for (int g = 0; g < 2; ++g)
            for (int64_t t = misc[9 + g]; t < misc[7 + g]; ++t)
                if ((t & 1) == g)
                    mbar_wait_teardown(XFULL((int)(2 * g + ((t >> 1) & 1))), (uint32_t)((t >> 2) & 1), 10000000ull);
    }
    if (warp == 1) tmem_dealloc(tmem, TM_COLS);
    cluster_sync();
}

// Merge the partial results of units cut between clusters.  One warp per
// head row (4 rows per 128-thread block, at most 64 registers, so that 8 blocks fit
// an SM).  Once the unit's piece range is known, the loads the merge needs are
// issued together: lane k < pieces reads piece k's lse, and each lane reads
// its 16 of the row's 512 columns from the first two pieces (further pieces
// take a loop).  The warp forms the
// log-sum-exp weights with shuffles.  Also writes o = 0, lse = -inf for
// units that see no cached position.
constexpr int COMBINE_ROWS = 4;
constexpr int COMBINE_UNROLL = 2;

__global__ void __launch_bounds__(32 * COMBINE_ROWS, 8)
decode_combine_kernel(const Params p) {
    if (device_status_raised()) return;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int row = blockIdx.x * COMBINE_ROWS + warp;  // u * HEADS + h
    const int u = row / HEADS, h = row % HEADS;
    if (u >= p.B * p.T * p.HG) return;
    int ub, ut, uh;
    unit_index(u, p.B, p.HG, ub, ut, uh);
    const int bt = ub * p.T + ut;  // row of q, o
    const int head = uh * HEADS + h;
    if (head >= p.H) return;
    const PlanView pv{p.seq_lens, p.B, p.T, p.HG, p.max_pages, p.causal};
    const int2 gg = p.ws_unit[u];         // issued together with the length read below
    const Unit un = unit_of(pv, u);
    const int64_t qrow = (int64_t)bt * p.H + head;
    __nv_bfloat16* dst = p.o + qrow * DC + 16 * lane;
    float* dst32 = p.o32 + qrow * DC + 16 * lane;
    if (un.pages == 0) {
        if (p.o32) {
#pragma unroll
            for (int v = 0; v < 4; ++v) reinterpret_cast<float4*>(dst32)[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            reinterpret_cast<uint4*>(dst)[0] = make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4*>(dst)[1] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (lane == 0) p.lse[qrow] = -INFINITY;
        return;
    }
    if (gg.x == gg.y) return;  // written directly by the attention kernel
    check_split(0 <= gg.x && gg.x < gg.y, 0x71);
    const int n = gg.y - gg.x + 1;
    const int64_t r0 = (int64_t)(gg.x + u) * HEADS + h;  // piece k's row: r0 + k * HEADS
    const float lse_l = lane < n ? p.ws_lse[r0 + (int64_t)lane * HEADS] : -INFINITY;
    float4 x[COMBINE_UNROLL][4];
#pragma unroll
    for (int k = 0; k < COMBINE_UNROLL; ++k) {
        const float4* src = reinterpret_cast<const float4*>(p.ws_o + (r0 + (int64_t)k * HEADS) * DC + 16 * lane);
#pragma unroll
        for (int v = 0; v < 4; ++v) x[k][v] = k < n ? __ldcg(src + v) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float m = lse_l;
    for (int k = lane + 32; k < n; k += 32) m = fmaxf(m, p.ws_lse[r0 + (int64_t)k * HEADS]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = __expf(lse_l - m);
    for (int k = lane + 32; k < n; k += 32) sum += __expf(p.ws_lse[r0 + (int64_t)k * HEADS] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float L = m + __logf(sum);
    const float w_l = __expf(lse_l - L);  // piece `lane`'s weight (0 past the last piece)
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
#pragma unroll
    for (int k = 0; k < COMBINE_UNROLL; ++k) {
        const float w = __shfl_sync(0xffffffffu, w_l, k);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            acc[4 * v] = fmaf(w, x[k][v].x, acc[4 * v]);
            acc[4 * v + 1] = fmaf(w, x[k][v].y, acc[4 * v + 1]);
            acc[4 * v + 2] = fmaf(w, x[k][v].z, acc[4 * v + 2]);
            acc[4 * v + 3] = fmaf(w, x[k][v].w, acc[4 * v + 3]);
        }
    }
    for (int k = COMBINE_UNROLL; k < n; ++k) {  // long runs of pieces
        const float wk = k < 32 ? __shfl_sync(0xffffffffu, w_l, k)
                                : __expf(p.ws_lse[r0 + (int64_t)k * HEADS] - L);
        const float4* src = reinterpret_cast<const float4*>(p.ws_o + (r0 + (int64_t)k * HEADS) * DC + 16 * lane);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const float4 y = __ldcg(src + v);
            acc[4 * v] = fmaf(wk, y.x, acc[4 * v]);
            acc[4 * v + 1] = fmaf(wk, y.y, acc[4 * v + 1]);
            acc[4 * v + 2] = fmaf(wk, y.z, acc[4 * v + 2]);
            acc[4 * v + 3] = fmaf(wk, y.w, acc[4 * v + 3]);
        }
    }
    if (p.o32) {
#pragma unroll
        for (int v = 0; v < 4; ++v)
            reinterpret_cast<float4*>(dst32)[v] = make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
    } else {
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                                      pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(pack_bf16x2(acc[8], acc[9]), pack_bf16x2(acc[10], acc[11]),
                                                      pack_bf16x2(acc[12], acc[13]), pack_bf16x2(acc[14], acc[15]));
    }
    if (lane == 0) p.lse[qrow] = L;
}

}  // namespace dec
}  // namespace mla
