// mla_lib.cu -- the C ABI of libmla (declared in include/mla.h): argument
// checks, TMA tensor maps, work planning and kernel launches.  The library is
// one translation unit so that the device status word has a single home.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/mla.h"
#include "decode_bf16.cuh"
#include "fold_q.cuh"
#include "gemm_bf16.cuh"
#include "kernels_fp32.cuh"
#include "prefill_bf16.cuh"
#include "prologue.cuh"
#include "ptx.cuh"
#include "status.cuh"

namespace {

using mla::dec::Params;

constexpr int kMaxDevices = 64;

// Caller-owned events recorded around the decode attention kernel (see
// mla_set_decode_events); both null when unset.
cudaEvent_t g_ev_start = nullptr, g_ev_end = nullptr;

// Kernels launched by this library (reported by mla_launch_count).
std::atomic<uint64_t> g_launches{0};

// ------------------------------------------------------------ driver entry

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Tiled bf16 tensor map; dims/strides innermost first, strides in bytes.
bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------ device facts

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int decode_clusters = 0;  // co-resident 2-CTA clusters of the decode kernel
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

bool device_info(DeviceInfo& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return false;
        if (cudaFuncSetAttribute(mla::dec::decode_bf16_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)mla::dec::SMEM_ALLOC) != cudaSuccess)
            return false;
        if (cudaFuncSetAttribute(mla::gemm::wgemm_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)mla::gemm::SMEM_CAP) != cudaSuccess ||
            cudaFuncSetAttribute(mla::gemm::wgemm_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)mla::gemm::SMEM_CAP) != cudaSuccess ||
            cudaFuncSetAttribute(mla::gemm::wgemm_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)mla::gemm::SMEM_CAP) != cudaSuccess ||
            cudaFuncSetAttribute(mla::gemm::wgemm_kernel<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)mla::gemm::SMEM_CAP) != cudaSuccess)
            return false;
        if (cudaFuncSetAttribute(mla::pre::prefill_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)mla::pre::SMEM_ALLOC) != cudaSuccess)
            return false;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (d.sms / 2), 1, 1);
        cfg.blockDim = dim3(mla::dec::THREADS, 1, 1);
        cfg.dynamicSmemBytes = mla::dec::SMEM_ALLOC;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, mla::dec::decode_bf16_kernel, &cfg) != cudaSuccess ||
            n <= 0) {
            cudaGetLastError();
            n = d.sms / 2;
        }
        d.decode_clusters = n;
        d.ready = true;
    }
    out = d;
    return true;
}

// ------------------------------------------------------------------ checks

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Status of the launch(es) just made; counts `n` launched kernels.
// Launch with programmatic stream serialization (pdl.cuh): the kernel may
// start its set-up while the one before it on the stream finishes.
template <typename... KArgs, typename... Args>
mla_status_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                        Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? MLA_OK
                                                                                          : MLA_ERR_CUDA;
}

mla_status_t launch_status(int n = 1) {
    if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
    g_launches += n;
    return MLA_OK;
}

// ------------------------------------------------------------ decode plan

// Does the plan cut some unit between clusters, or leave one without any
// visible position?  (Only then is the combine kernel needed.)
// Clusters to launch for the bf16 decode.  When every non-empty unit has the
// same number of pages n and there are no more units than co-resident
// clusters, launching one cluster per unit cuts no unit (the equal cuts of
// the line then fall in the virtual gaps between units), so the merge
// kernel and the pieces' fp32 partials drop out; it is chosen when the
// largest range grows by at most kWholeUnitSlackPages pages against the
// cut of all G clusters.  (Measured on B300: 64 sequences of 4096 -- 64 pages
// per cluster against 55.4 with cuts -- the step took 104 µs against 112.4;
// 64 x 32768 with 16 heads -- 512 pages against 443 -- 699 µs against 651.)
constexpr int kWholeUnitSlackPages = 16;

int whole_unit_clusters(const int32_t* lens, int B, int T, int HG, int max_pages, int causal, int G) {
    mla::dec::PlanView v{lens, B, T, HG, max_pages, causal};
    const int U = B * T * HG;
    int units = 0, n = -1;
    int64_t total = 0;
    for (int u = 0; u < U; ++u) {
        const mla::dec::Unit un = mla::dec::unit_of(v, u);
        if (un.bad_len) return G;
        if (un.pages == 0) continue;
        if (n >= 0 && un.pages != n) return G;
        n = un.pages;
        ++units;
        total += un.pages;
    }
    if (units == 0 || units > G) return G;
    const int C = mla::dec::boundary_pages((int)total, G);
    const int64_t V = mla::dec::virtual_total((int)total, units, C);
    const int64_t cut = (V + G - 1) / G;  // pages in the largest range with all G clusters
    return n - cut <= kWholeUnitSlackPages ? units : G;
}

bool host_plan_needs_combine(const int32_t* lens, int B, int T, int HG, int max_pages, int causal,
                             int launched) {
    mla::dec::PlanView v{lens, B, T, HG, max_pages, causal};
    const int U = B * T * HG;
    int total = 0;
    for (int u = 0; u < U; ++u) {
        const mla::dec::Unit un = mla::dec::unit_of(v, u);
        if (un.pages == 0 || un.bad_len) return true;
        total += un.pages;
    }
    const int C = mla::dec::boundary_pages(total, launched);
    const int V = mla::dec::virtual_total(total, U, C);
    const int G = mla::dec::clusters_used(total, launched);
    int pos = 0;
    for (int u = 0; u < U; ++u) {
        const int n = mla::dec::unit_of(v, u).pages;
        if (mla::dec::cluster_of_page(pos, V, G) != mla::dec::cluster_of_page(pos + n - 1, V, G))
            return true;
        pos += n + C;
    }
    return false;
}

struct DecodeWs {
    size_t unit_off, lse_off, o_off, total;
};

DecodeWs decode_ws_layout(int64_t U, int64_t G, int d_c) {
    auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
    const int64_t slots = G + U;
    DecodeWs w;
    w.unit_off = 0;
    w.lse_off = up(sizeof(int2) * (size_t)U);
    w.o_off = up(w.lse_off + sizeof(float) * (size_t)slots * mla::dec::HEADS);
    w.total = up(w.o_off + sizeof(float) * (size_t)slots * mla::dec::HEADS * (size_t)d_c);
    return w;
}

// ------------------------------------------------------------- GEMM plan

struct GemmPlan {
    int BN = 16, n_tiles = 1, m_tiles = 1, MT = 1, splits = 1, chunks = 1, items = 0, grid = 0, stages = 1;
    int mode = mla::gemm::OUT_BF16;
    size_t smem = 0, ws_part_bytes = 0, ws_count_bytes = 0;
};

enum SplitMode : int { kNoSplit = 0, kSplitReduce = 1, kSplitParts = 2 };

// The GEMM's work plan for D [M x N] per head z (M rows that exist, a
// multiple of 8) with reduction length K.  One CTA per SM walks a
// contiguous range of items.  The M tiles per item (MT) and the K split are
// chosen by a cost in SM cycles: the largest of the weight stream at the
// HBM rate, the busiest CTA's chunks (each bound by its TMA rows, about 3.1
// cycles per 128-byte row, measured, or by its products, about BN / 2
// cycles per 16-deep step of one M tile), and its epilogue stores (about 20
// bytes per cycle per SM, measured); plus the last item's stores and, for a
// split reduced in the kernel, the reducing CTA's reads.  A K split is
// considered only for few output tiles and a workspace below 256 MB; of two
// plans within 2 % of each other the one with fewer TMA rows per CTA wins.
GemmPlan gemm_plan(int M, int N, int K, int Z, int sms, SplitMode split, int max_splits = 64,
                   bool allow_pairs = true, size_t extra_smem = 0) {
    const double kRow = 3.1, kHbm = 3150.0, kStore = 20.0, kL2 = 64.0;
    GemmPlan g;
    g.BN = N >= 256 ? 256 : ((N + 15) / 16) * 16;
    g.n_tiles = (N + g.BN - 1) / g.BN;
    g.m_tiles = (M + mla::gemm::BM - 1) / mla::gemm::BM;
    const int kc = K / mla::gemm::BK;
    const double a_bytes = 2.0 * Z * g.m_tiles * mla::gemm::BM * (double)K;
    double best = 1e300, best_tma = 1e300;
    int best_s = 1, best_mt = 1;
    for (int MT = 1; MT <= 2; ++MT) {
        if (MT == 2 && (!allow_pairs || g.m_tiles % 2 != 0 || g.BN > 128)) continue;
        const int64_t units = (int64_t)Z * (g.m_tiles / MT) * g.n_tiles;
        const bool few = split == kSplitParts || units < 2 * (int64_t)sms;
        const int s_max = split == kNoSplit || !few ? 1 : std::max(1, std::min(kc, max_splits));
        for (int s = 1; s <= s_max; ++s) {
            const int cps = (kc + s - 1) / s;
            if ((kc + cps - 1) / cps != s) continue;  // the same cut as a smaller s
            const int64_t items = units * s;
            const int64_t G = std::min<int64_t>(items, sms);
            const int64_t per = (items + G - 1) / G;
            if (s > 1 && 4.0 * s * Z * (double)N * M > 256.0 * (1 << 20)) continue;
            const bool fp32 = split == kSplitParts || s > 1;
            const double tile_store = (double)mla::gemm::BM * g.BN * (fp32 ? 4 : 2) / kStore;
            const double tma =
                (double)per * cps * std::max((MT * mla::gemm::BM + g.BN) * kRow, 2.0 * MT * g.BN);
            const double stores = (double)per * MT * tile_store;
            double cost = std::max(std::max(a_bytes / kHbm, tma), stores) + MT * tile_store;
            if (split == kSplitReduce && s > 1)
                cost += s * (double)mla::gemm::BM * g.BN * 4 / kL2 + (double)mla::gemm::BM * g.BN * 2 / kStore;
            if (cost < best * (1 - 0.02) || (cost < best * (1 + 0.02) && tma < best_tma)) {
                best = std::min(best, cost);
                best_tma = tma;
                best_s = s;
                best_mt = MT;
            }
        }
    }
    g.MT = best_mt;
    g.chunks = (kc + best_s - 1) / best_s;
    g.splits = (kc + g.chunks - 1) / g.chunks;
    g.mode = split == kSplitParts ? mla::gemm::OUT_PARTS
                                  : (g.splits > 1 ? mla::gemm::OUT_REDUCE : mla::gemm::OUT_BF16);
    const int64_t tiles = (int64_t)Z * g.m_tiles * g.n_tiles;
    const int64_t items = (int64_t)Z * (g.m_tiles / g.MT) * g.n_tiles * g.splits;
    g.items = items > 0x7FFFFFFF ? 0 : (int)items;  // 0: too large (refused by the caller)
    g.grid = (int)std::min<int64_t>(items, sms);
    const size_t stage = (size_t)g.MT * mla::gemm::A_BYTES + (size_t)g.BN * mla::gemm::BK * 2;
    const size_t fixed = mla::gemm::FIXED_SMEM + extra_smem;  // extra: the query's rotation table
    g.stages = (int)std::min<size_t>(mla::gemm::MAX_STAGES, (mla::gemm::SMEM_CAP - fixed) / stage);
    // no more stages than the busiest CTA has K chunks: the rest of the
    // shared memory is then free for a dependent kernel's blocks
    const int64_t busiest = (items + g.grid - 1) / std::max(1, g.grid) * g.chunks;
    g.stages = (int)std::max<int64_t>(2, std::min<int64_t>(g.stages, busiest));
    g.smem = fixed + (size_t)g.stages * stage;
    g.ws_part_bytes = g.mode != mla::gemm::OUT_BF16 ? sizeof(float) * (size_t)g.splits * Z * N * M : 0;
    g.ws_count_bytes = g.mode == mla::gemm::OUT_REDUCE ? sizeof(int) * (size_t)tiles : 0;
    return g;
}

// Where the query projection's GEMM writes its heads (OUT_QROPE).
struct QRopeOut {
    __nv_bfloat16* q_nope;
    __nv_bfloat16* q_pe;
    const int32_t* positions;
    int H, d_h, d_r;
    const uint64_t* freq;  // rope::MAX_PAIRS fixed-point frequencies
    int table;             // the plan reserved the N tile's sin/cos table
};

// Launch the persistent GEMM.  ta2 serves the M tiles from m_split on (pass
// ta and m_split = m_tiles when there is one A map).  With qo (a plan
// without K splits) the epilogue writes the query heads instead of `out`.
mla_status_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& ta2, int m_split, const CUtensorMap& tx,
                         int M, int N, int K, int Z, int a_mn, int x_batched, const GemmPlan& g,
                         __nv_bfloat16* out, int64_t ldo, int64_t out_z, float* ws_part, int* ws_count,
                         cudaStream_t st, const QRopeOut* qo = nullptr) {
    if (g.items < 1 || M % 8 != 0) return MLA_ERR_UNSUPPORTED;
    if (g.mode != mla::gemm::OUT_BF16 && (!ws_part || !aligned16(ws_part))) return MLA_ERR_INVALID_ARG;
    if (g.mode == mla::gemm::OUT_REDUCE && !ws_count) return MLA_ERR_INVALID_ARG;
    if (qo && (g.mode != mla::gemm::OUT_BF16 || qo->d_h % 8 != 0 || qo->d_r % 8 != 0 ||
               (int64_t)qo->H * (qo->d_h + qo->d_r) != M))
        return MLA_ERR_UNSUPPORTED;
    mla::gemm::Params p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.m_tiles = g.m_tiles;
    p.MT = g.MT;
    p.m_units = g.m_tiles / g.MT;
    p.m_split = m_split;
    p.BN = g.BN;
    p.n_tiles = g.n_tiles;
    p.a_mn = a_mn;
    p.x_batched = x_batched;
    p.splits = g.splits;
    p.chunks_per_split = g.chunks;
    p.items = g.items;
    p.stages = g.stages;
    p.mode = g.mode;
    p.a_evict_first = g.n_tiles == 1 ? 1 : 0;
    p.vec_out = (aligned16(out) && ldo % 8 == 0 && out_z % 8 == 0) ? 1 : 0;
    p.out = out;
    p.ldo = ldo;
    p.out_z = out_z;
    p.ws_part = ws_part;
    p.ws_count = ws_count;
    if (qo) {
        p.mode = mla::gemm::OUT_QROPE;
        p.q_nope = qo->q_nope;
        p.q_pe = qo->q_pe;
        p.positions = qo->positions;
        p.q_heads = qo->H;
        p.d_h = qo->d_h;
        p.d_r = qo->d_r;
        p.rope_table = qo->table;
        for (int k = 0; k < mla::rope::MAX_PAIRS; ++k) p.freq[k] = qo->freq[k];
    }
    (void)Z;
    const mla_status_t s = launch_pdl(qo ? (g.MT == 2 ? mla::gemm::wgemm_kernel<2, true> : mla::gemm::wgemm_kernel<1, true>)
                                         : (g.MT == 2 ? mla::gemm::wgemm_kernel<2, false> : mla::gemm::wgemm_kernel<1, false>),
                                      dim3((unsigned)g.grid), dim3(mla::gemm::THREADS), g.smem, st, ta, ta2,
                                      tx, p);
    if (s != MLA_OK) return s;
    return launch_status();
}

mla_status_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tx, int M, int N, int K, int Z,
                         int a_mn, int x_batched, const GemmPlan& g, __nv_bfloat16* out, int64_t ldo,
                         int64_t out_z, float* ws_part, int* ws_count, cudaStream_t st) {
    return launch_gemm(ta, ta, g.m_tiles, tx, M, N, K, Z, a_mn, x_batched, g, out, ldo, out_z, ws_part,
                       ws_count, st);
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Scratch of one plain GEMM: split-K partials, then the arrival counters
// (zero before the first use; every call leaves them at zero).
size_t plain_gemm_ws_bytes(const GemmPlan& g) { return round256(g.ws_part_bytes) + g.ws_count_bytes; }

float* ws_parts(const GemmPlan& g, void* ws) {
    return g.mode != mla::gemm::OUT_BF16 ? static_cast<float*>(ws) : nullptr;
}
int* ws_counts(const GemmPlan& g, void* ws) {
    return g.mode == mla::gemm::OUT_REDUCE
               ? reinterpret_cast<int*>(static_cast<char*>(ws) + round256(g.ws_part_bytes))
               : nullptr;
}

// Tensor maps of a K-major weight W [M, K] (A operand, 128 x 64 boxes) and
// of activation rows X [N, K] with rows x_ld elements apart (BN x 64 boxes).
bool weight_map(CUtensorMap* m, const void* W, int M, int K) {
    cuuint64_t ad[3] = {(cuuint64_t)K, (cuuint64_t)M, 1};
    cuuint64_t as[2] = {(cuuint64_t)K * 2, (cuuint64_t)K * M * 2};
    cuuint32_t ab[3] = {64, 128, 1};
    return make_map(m, W, 3, ad, as, ab, CU_TENSOR_MAP_SWIZZLE_128B);
}
bool rows_map(CUtensorMap* m, const void* X, int N, int K, int64_t x_ld, int BN) {
    cuuint64_t xd[3] = {(cuuint64_t)K, 1, (cuuint64_t)N};
    cuuint64_t xs[2] = {(cuuint64_t)x_ld * 2, (cuuint64_t)x_ld * 2};
    cuuint32_t xbx[3] = {64, 1, (cuuint32_t)BN};
    return make_map(m, X, 3, xd, xs, xbx, CU_TENSOR_MAP_SWIZZLE_128B);
}

// out[n * ldo + m] = sum_k W[m, k] X[n, k] in bf16 (or the fp32 partials of
// g's mode): the weight W [M, K] (K-major) on the UMMA M axis, the
// activation rows X [N, K] on N.  X's rows are x_ld elements apart (0: K).
mla_status_t plain_gemm(const void* W, const void* X, __nv_bfloat16* out, int64_t ldo, int M, int N,
                        int K, const GemmPlan& g, void* ws, cudaStream_t st, int64_t x_ld = 0) {
    CUtensorMap ta, tx;
    if (x_ld == 0) x_ld = K;
    if (!weight_map(&ta, W, M, K) || !rows_map(&tx, X, N, K, x_ld, g.BN)) return MLA_ERR_CUDA;
    return launch_gemm(ta, tx, M, N, K, 1, 0, 0, g, out, ldo, 0, ws_parts(g, ws), ws_counts(g, ws), st);
}

}  // namespace

// =================================================================== C ABI

extern "C" {

int mla_version(void) { return 101; }

uint64_t mla_launch_count(void) { return g_launches.load(); }

void mla_set_decode_events(void* start, void* end) {
    g_ev_start = static_cast<cudaEvent_t>(start);
    g_ev_end = static_cast<cudaEvent_t>(end);
}

const char* mla_status_string(mla_status_t s) {
    switch (s) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARG: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported shape for this dtype";
        case MLA_ERR_CUDA: return "CUDA runtime error";
        case MLA_ERR_TIMEOUT: return "device: bounded wait timed out";
        case MLA_ERR_DEVICE_BOUNDS: return "device: page id or sequence length out of range";
    }
    return "unknown status";
}

mla_status_t mla_get_device_status(mla_stream_t stream, uint32_t* detail) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MLA_ERR_CUDA;
    uint32_t w = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&w, mla::g_device_status, sizeof w) != cudaSuccess) return MLA_ERR_CUDA;
    if (w != 0 && cudaMemcpyToSymbol(mla::g_device_status, &zero, sizeof zero) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (detail) *detail = w >> 8;
    switch (w & 0xFFu) {
        case mla::MLA_DEV_OK: return MLA_OK;
        case mla::MLA_DEV_TIMEOUT: return MLA_ERR_TIMEOUT;
        default: return MLA_ERR_DEVICE_BOUNDS;
    }
}

mla_status_t mla_set_wait_limit(uint64_t ns) {
    const uint64_t v = ns == 0 ? mla::MLA_WAIT_LIMIT_NS : ns;
    if (cudaMemcpyToSymbol(mla::g_wait_limit_ns, &v, sizeof v) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return MLA_ERR_CUDA;
    return MLA_OK;
}

// ------------------------------------------------------------ mla_absorb_q

mla_status_t mla_absorb_q(const void* q_nope, const void* w_uk, void* q_lat, int rows, int H,
                          int d_h, int d_c, mla_dtype_t dtype, mla_stream_t stream) {
    if (!q_nope || !w_uk || !q_lat || rows < 1 || H < 1 || d_h < 1 || d_c < 1)
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_nope) || !aligned16(w_uk) || !aligned16(q_lat)) return MLA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == MLA_FP32) {
        if ((int64_t)rows * H > 0x7FFFFFFF) return MLA_ERR_UNSUPPORTED;
        dim3 grid((unsigned)rows * H, (d_c + 127) / 128);
        mla::absorb_q_fp32_kernel<<<grid, 128, 0, st>>>(
            static_cast<const float*>(q_nope), static_cast<const float*>(w_uk),
            static_cast<float*>(q_lat), rows, H, d_h, d_c);
        return launch_status();
    }
    if (dtype != MLA_BF16) return MLA_ERR_INVALID_ARG;
    if (d_c % 128 != 0 || d_h % 64 != 0 || H > 65535) return MLA_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (!device_info(di)) return MLA_ERR_CUDA;
    const GemmPlan g = gemm_plan(d_c, rows, d_h, H, di.sms, kNoSplit);
    // A = W^UK_i^T, stored along d_c: MN-major tiles [64 d_h rows x 64 d_c]
    CUtensorMap ta, tx;
    cuuint64_t ad[3] = {(cuuint64_t)d_c, (cuuint64_t)d_h, (cuuint64_t)H};
    cuuint64_t as[2] = {(cuuint64_t)d_c * 2, (cuuint64_t)d_h * d_c * 2};
    cuuint32_t ab[3] = {64, 64, 1};
    cuuint64_t xd[3] = {(cuuint64_t)d_h, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t xs[2] = {(cuuint64_t)d_h * 2, (cuuint64_t)H * d_h * 2};
    cuuint32_t xbx[3] = {64, 1, (cuuint32_t)g.BN};
    if (!make_map(&ta, w_uk, 3, ad, as, ab, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tx, q_nope, 3, xd, xs, xbx, CU_TENSOR_MAP_SWIZZLE_128B))
        return MLA_ERR_CUDA;
    return launch_gemm(ta, tx, d_c, rows, d_h, H, 1, 1, g, static_cast<__nv_bfloat16*>(q_lat),
                       (int64_t)H * d_c, d_c, nullptr, nullptr, st);
}

// ------------------------------------------------------------ mla_out_proj

size_t mla_out_proj_workspace_size(int rows, int H, int d_h, int d, mla_dtype_t dtype) {
    if (dtype != MLA_BF16 || rows < 1 || H < 1 || d_h < 1 || d < 128) return 0;
    DeviceInfo di;
    if (!device_info(di)) return 0;
    const GemmPlan g = gemm_plan(d, rows, H * d_h, 1, di.sms, kSplitReduce);
    return plain_gemm_ws_bytes(g);
}

mla_status_t mla_out_proj(const void* o, const void* w_uv, const void* w_o, void* v_tmp, void* out,
                          int rows, int H, int d_h, int d_c, int d, void* workspace,
                          size_t workspace_bytes, mla_dtype_t dtype, mla_stream_t stream) {
    if (!o || !w_uv || !w_o || !v_tmp || !out || rows < 1 || H < 1 || d_h < 1 || d_c < 1 || d < 1)
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(w_uv) || !aligned16(w_o) || !aligned16(v_tmp) ||
        !aligned16(out))
        return MLA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == MLA_FP32) {
        const int64_t warps1 = (int64_t)rows * H * d_h, warps2 = (int64_t)rows * d;
        mla::out_proj_v_fp32_kernel<<<(unsigned)((warps1 + 3) / 4), 128, 0, st>>>(
            static_cast<const float*>(o), static_cast<const float*>(w_uv), static_cast<float*>(v_tmp),
            rows, H, d_h, d_c);
        mla::out_proj_o_fp32_kernel<<<(unsigned)((warps2 + 3) / 4), 128, 0, st>>>(
            static_cast<const float*>(v_tmp), static_cast<const float*>(w_o), static_cast<float*>(out),
            rows, H * d_h, d);
        return launch_status(2);
    }
    if (dtype != MLA_BF16) return MLA_ERR_INVALID_ARG;
    if (d_h % 128 != 0 || d_c % 64 != 0 || d % 128 != 0 || H > 65535) return MLA_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (!device_info(di)) return MLA_ERR_CUDA;
    const int K2 = H * d_h;
    const GemmPlan g1 = gemm_plan(d_h, rows, d_c, H, di.sms, kNoSplit);
    const GemmPlan g2 = gemm_plan(d, rows, K2, 1, di.sms, kSplitReduce);
    if (g2.mode != mla::gemm::OUT_BF16 &&
        (!workspace || workspace_bytes < plain_gemm_ws_bytes(g2) || !aligned16(workspace)))
        return MLA_ERR_INVALID_ARG;
    CUtensorMap ta1, tx1, ta2, tx2;
    {   // v = W^UV_i o_i : A K-major [d_h rows x 64 d_c], X = o [rows, H, d_c]
        cuuint64_t ad[3] = {(cuuint64_t)d_c, (cuuint64_t)d_h, (cuuint64_t)H};
        cuuint64_t as[2] = {(cuuint64_t)d_c * 2, (cuuint64_t)d_h * d_c * 2};
        cuuint32_t ab[3] = {64, 128, 1};
        cuuint64_t xd[3] = {(cuuint64_t)d_c, (cuuint64_t)H, (cuuint64_t)rows};
        cuuint64_t xs[2] = {(cuuint64_t)d_c * 2, (cuuint64_t)H * d_c * 2};
        cuuint32_t xbx[3] = {64, 1, (cuuint32_t)g1.BN};
        if (!make_map(&ta1, w_uv, 3, ad, as, ab, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&tx1, o, 3, xd, xs, xbx, CU_TENSOR_MAP_SWIZZLE_128B))
            return MLA_ERR_CUDA;
    }
    {   // out = W^O v : A K-major [128 d rows x 64 k], X = v [rows, H*d_h]
        cuuint64_t ad[3] = {(cuuint64_t)K2, (cuuint64_t)d, 1};
        cuuint64_t as[2] = {(cuuint64_t)K2 * 2, (cuuint64_t)K2 * d * 2};
        cuuint32_t ab[3] = {64, 128, 1};
        cuuint64_t xd[3] = {(cuuint64_t)K2, 1, (cuuint64_t)rows};
        cuuint64_t xs[2] = {(cuuint64_t)K2 * 2, (cuuint64_t)K2 * 2};
        cuuint32_t xbx[3] = {64, 1, (cuuint32_t)g2.BN};
        if (!make_map(&ta2, w_o, 3, ad, as, ab, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&tx2, v_tmp, 3, xd, xs, xbx, CU_TENSOR_MAP_SWIZZLE_128B))
            return MLA_ERR_CUDA;
    }
    mla_status_t s = launch_gemm(ta1, tx1, d_h, rows, d_c, H, 0, 1, g1,
                                 static_cast<__nv_bfloat16*>(v_tmp), (int64_t)K2, d_h, nullptr,
                                 nullptr, st);
    if (s != MLA_OK) return s;
    return launch_gemm(ta2, tx2, d, rows, K2, 1, 0, 0, g2, static_cast<__nv_bfloat16*>(out), d, 0,
                       ws_parts(g2, workspace), ws_counts(g2, workspace), st);
}

// ------------------------------------------------- merged output weight

mla_status_t mla_fold_out_weights(const void* w_uv, const void* w_o, void* w_merged, int H, int d_h,
                                  int d_c, int d, mla_dtype_t dtype, mla_stream_t stream) {
    if (!w_uv || !w_o || !w_merged || H < 1 || d_h < 1 || d_c < 1 || d < 1)
        return MLA_ERR_INVALID_ARG;
    // W_merged[n, i, :] = W^UV_i^T W^O[n, i, :] is the query absorption's
    // product with row n of W^O, head slice i, in the place of q^C.
    return mla_absorb_q(w_o, w_uv, w_merged, d, H, d_h, d_c, dtype, stream);
}

size_t mla_fold_q_workspace_size(int H, int d_h, int d_q, mla_dtype_t dtype) {
    if ((dtype != MLA_BF16 && dtype != MLA_FP32) || H < 1 || d_h < 1 || d_q < 1) return 0;
    return round256((size_t)d_q * H * d_h * (dtype == MLA_BF16 ? 2 : 4));
}

mla_status_t mla_fold_q_weights(const void* w_uk, const void* w_q, void* w_merged, int H, int d_h,
                                int d_r, int d_c, int d_q, void* workspace, size_t workspace_bytes,
                                mla_dtype_t dtype, mla_stream_t stream) {
    if (!w_uk || !w_q || !w_merged || H < 1 || d_h < 1 || d_r < 0 || d_c < 1 || d_q < 1)
        return MLA_ERR_INVALID_ARG;
    if (dtype != MLA_BF16 && dtype != MLA_FP32) return MLA_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < mla_fold_q_workspace_size(H, d_h, d_q, dtype))
        return MLA_ERR_INVALID_ARG;
    if ((int64_t)H * d_h > 65535 * 32 || d_q > 65535 * 32) return MLA_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // W^UQ^T [d_q, H, d_h] into the workspace, then the query absorption of
    // its d_q rows: row k, head slice i becomes W^UK_i^T W^UQ_i[:, k]
    const dim3 grid((unsigned)((d_q + 31) / 32), (unsigned)((H * d_h + 31) / 32));
    const dim3 block(32, 8);
    if (dtype == MLA_BF16)
        mla::foldq::uq_transpose_kernel<__nv_bfloat16><<<grid, block, 0, st>>>(
            static_cast<const __nv_bfloat16*>(w_q), static_cast<__nv_bfloat16*>(workspace), H, d_h, d_r,
            d_q);
    else
        mla::foldq::uq_transpose_kernel<float><<<grid, block, 0, st>>>(
            static_cast<const float*>(w_q), static_cast<float*>(workspace), H, d_h, d_r, d_q);
    if (launch_status() != MLA_OK) return MLA_ERR_CUDA;
    return mla_absorb_q(workspace, w_uk, w_merged, d_q, H, d_h, d_c, dtype, stream);
}

mla_status_t mla_absorb_q_merged(const void* c_q, const void* w_merged, void* q_lat, int rows, int H,
                                 int d_c, int d_q, mla_dtype_t dtype, mla_stream_t stream) {
    if (!c_q || !w_merged || !q_lat || rows < 1 || H < 1 || d_c < 1 || d_q < 1)
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(c_q) || !aligned16(w_merged) || !aligned16(q_lat)) return MLA_ERR_INVALID_ARG;
    const int64_t M = (int64_t)H * d_c;
    if (M > (1 << 30) || rows > 65535) return MLA_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == MLA_FP32) {
        const dim3 grid((unsigned)((M + 127) / 128), (unsigned)rows);
        mla::foldq::q_merged_fp32_kernel<<<grid, 128, 0, st>>>(
            static_cast<const float*>(c_q), static_cast<const float*>(w_merged), static_cast<float*>(q_lat),
            (int)M, d_q);
        return launch_status();
    }
    if (dtype != MLA_BF16) return MLA_ERR_INVALID_ARG;
    if (M % 128 != 0 || d_q % 64 != 0) return MLA_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (!device_info(di)) return MLA_ERR_CUDA;
    // q_lat = W_merged c^Q: the folded weight [d_q, H * d_c] is stored along
    // its output axis, so it is an MN-major A operand of the GEMM
    const GemmPlan g = gemm_plan((int)M, rows, d_q, 1, di.sms, kNoSplit);
    CUtensorMap ta, tx;
    cuuint64_t ad[3] = {(cuuint64_t)M, (cuuint64_t)d_q, 1};
    cuuint64_t as[2] = {(cuuint64_t)M * 2, (cuuint64_t)M * d_q * 2};
    cuuint32_t ab[3] = {64, 64, 1};
    cuuint64_t xd[3] = {(cuuint64_t)d_q, 1, (cuuint64_t)rows};
    cuuint64_t xs[2] = {(cuuint64_t)d_q * 2, (cuuint64_t)d_q * 2};
    cuuint32_t xbx[3] = {64, 1, (cuuint32_t)g.BN};
    if (!make_map(&ta, w_merged, 3, ad, as, ab, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tx, c_q, 3, xd, xs, xbx, CU_TENSOR_MAP_SWIZZLE_128B))
        return MLA_ERR_CUDA;
    return launch_gemm(ta, tx, (int)M, rows, d_q, 1, 1, 0, g, static_cast<__nv_bfloat16*>(q_lat), M, 0,
                       nullptr, nullptr, st);
}

size_t mla_out_proj_merged_workspace_size(int rows, int H, int d_c, int d, mla_dtype_t dtype) {
    if (dtype != MLA_BF16 || rows < 1 || H < 1 || d_c < 1 || d < 128) return 0;
    const int64_t K = (int64_t)H * d_c;
    if (K > (1 << 30)) return 0;
    DeviceInfo di;
    if (!device_info(di)) return 0;
    return plain_gemm_ws_bytes(gemm_plan(d, rows, (int)K, 1, di.sms, kSplitReduce));
}

mla_status_t mla_out_proj_merged(const void* o, const void* w_merged, void* out, int rows, int H,
                                 int d_c, int d, void* workspace, size_t workspace_bytes,
                                 mla_dtype_t dtype, mla_stream_t stream) {
    if (!o || !w_merged || !out || rows < 1 || H < 1 || d_c < 1 || d < 1)
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(w_merged) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
    const int64_t K = (int64_t)H * d_c;
    if (K > (1 << 30)) return MLA_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == MLA_FP32) {
        const int64_t warps = (int64_t)rows * d;
        mla::out_proj_o_fp32_kernel<<<(unsigned)((warps + 3) / 4), 128, 0, st>>>(
            static_cast<const float*>(o), static_cast<const float*>(w_merged), static_cast<float*>(out),
            rows, (int)K, d);
        return launch_status();
    }
    if (dtype != MLA_BF16) return MLA_ERR_INVALID_ARG;
    if (d % 128 != 0 || d_c % 64 != 0) return MLA_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (!device_info(di)) return MLA_ERR_CUDA;
    const GemmPlan g = gemm_plan(d, rows, (int)K, 1, di.sms, kSplitReduce);
    if (g.mode != mla::gemm::OUT_BF16 &&
        (!workspace || !aligned16(workspace) || workspace_bytes < plain_gemm_ws_bytes(g)))
        return MLA_ERR_INVALID_ARG;
    // out = W_merged o on the tensor cores: the merged weight on the UMMA M
    // axis, the rows of o (all heads' latents, H * d_c long) on N
    return plain_gemm(w_merged, o, static_cast<__nv_bfloat16*>(out), d, d, rows, (int)K, g, workspace,
                      st);
}

// ------------------------------------------- mla_cache_append / mla_project_q

// RoPE frequencies f_k = base^(-2k/d_r) / 2pi as 0.64 fixed-point fractions
// of a turn (the kernels multiply them by the position modulo 2^64), taken
// in extended precision on the host.
bool rope_freqs(uint64_t (&f)[mla::pro::MAX_PAIRS], int d_r, double base) {
    if (d_r < 2 || d_r / 2 > mla::pro::MAX_PAIRS || !(base > 0.0)) return false;
    const long double two_pi = 6.283185307179586476925286766559005768L;
    for (int k = 0; k < mla::pro::MAX_PAIRS; ++k) f[k] = 0;
    for (int k = 0; k < d_r / 2; ++k) {
        long double fr = powl((long double)base, -2.0L * k / (long double)d_r) / two_pi;
        fr -= floorl(fr);
        const long double v = ldexpl(fr, 64);
        f[k] = v >= 18446744073709551615.0L ? ~0ull : (uint64_t)v;
    }
    return true;
}

// The cache write's GEMM covers [W^DKV ; W^KR] as M = d_c + d_r rows; its
// plan (and so the workspace) depends on d_r only through the number of M
// tiles, which is d_c / 128 + 1 for every d_r <= 128.
GemmPlan cache_append_plan(int N, int d, int d_c, int d_r, int sms) {
    // one A map per item: the pair of M tiles would straddle W^DKV and W^KR
    return gemm_plan(d_c + d_r, N, d, 1, sms, kSplitParts, 64, false);
}

size_t mla_cache_append_workspace_size(int N, int d, int d_c, mla_dtype_t dtype) {
    if (dtype != MLA_BF16 || N < 1 || d < 64 || d_c < 128) return 0;
    DeviceInfo di;
    if (!device_info(di)) return 0;
    return plain_gemm_ws_bytes(cache_append_plan(N, d, d_c, 2 * mla::pro::MAX_PAIRS, di.sms));
}

mla_status_t mla_cache_append(const void* h, const void* w_dkv, const void* w_kr,
                              const int32_t* seq_ids, const int32_t* positions,
                              const int32_t* page_table, void* kv_pool, int N, int d, int d_c,
                              int d_r, int B, int page_size, int max_pages, int64_t num_pages,
                              double rope_base, void* workspace, size_t workspace_bytes,
                              mla_dtype_t dtype, mla_stream_t stream) {
    if (!h || !w_dkv || !w_kr || !seq_ids || !positions || !page_table || !kv_pool)
        return MLA_ERR_INVALID_ARG;
    // RoPE rotates pairs: an odd d_r has no meaning
    if (N < 1 || d < 1 || d_c < 1 || d_r < 2 || (d_r % 2) != 0 || B < 1 || page_size < 1 ||
        max_pages < 1 || num_pages < 1 || !(rope_base > 0.0))
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(h) || !aligned16(w_dkv) || !aligned16(w_kr) || !aligned16(kv_pool))
        return MLA_ERR_INVALID_ARG;
    if (dtype != MLA_BF16 && dtype != MLA_FP32) return MLA_ERR_INVALID_ARG;
    if (d_c % 2 != 0 || d_r > 2 * mla::pro::MAX_PAIRS) return MLA_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    mla::pro::KvParams p;
    p.h = h;
    p.w_dkv = w_dkv;
    p.w_kr = w_kr;
    p.parts = nullptr;
    p.splits = 0;
    p.seq_ids = seq_ids;
    p.positions = positions;
    p.page_table = page_table;
    p.pool = kv_pool;
    p.N = N;
    p.d = d;
    p.d_c = d_c;
    p.d_r = d_r;
    p.B = B;
    p.page = page_size;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    if (!rope_freqs(p.freq, d_r, rope_base)) return MLA_ERR_INVALID_ARG;
    if (dtype == MLA_FP32) {
        if (d % 4 != 0) return MLA_ERR_UNSUPPORTED;
        const dim3 grid((unsigned)((N + mla::pro::TOK - 1) / mla::pro::TOK),
                        (unsigned)((d_c + d_r + mla::pro::ROWS - 1) / mla::pro::ROWS));
        mla::pro::kv_rows_fp32_kernel<<<grid, mla::pro::THREADS, 0, st>>>(p);
        return launch_status();
    }
    if (d_c % 128 != 0 || d % 64 != 0 || d_r % 8 != 0) return MLA_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (!device_info(di)) return MLA_ERR_CUDA;
    const GemmPlan g = cache_append_plan(N, d, d_c, d_r, di.sms);
    if (!workspace || !aligned16(workspace) || workspace_bytes < plain_gemm_ws_bytes(g))
        return MLA_ERR_INVALID_ARG;
    // [W^DKV ; W^KR] h on the tensor cores: M tiles 0 .. d_c/128 - 1 from
    // W^DKV, the last from W^KR (its rows past d_r read as zeros), each K
    // split's fp32 partial into the workspace; then the finishing kernel
    // adds the splits, rotates k^R and writes whole pool rows.
    CUtensorMap ta, ta2, tx;
    if (!weight_map(&ta, w_dkv, d_c, d) || !weight_map(&ta2, w_kr, d_r, d) ||
        !rows_map(&tx, h, N, d, d, g.BN))
        return MLA_ERR_CUDA;
    float* parts = ws_parts(g, workspace);
    mla_status_t s = launch_gemm(ta, ta2, d_c / mla::gemm::BM, tx, d_c + d_r, N, d, 1, 0, 0, g, nullptr, 0,
                                 0, parts, nullptr, st);
    if (s != MLA_OK) return s;
    p.parts = parts;
    p.splits = g.splits;
    const unsigned threads = (unsigned)(((d_c + d_r) / 2 + 31) / 32 * 32);
    if (threads > 1024) return MLA_ERR_UNSUPPORTED;
    s = launch_pdl(mla::pro::kv_finish_bf16_kernel, dim3((unsigned)N), dim3(threads), 0, st, p);
    if (s != MLA_OK) return s;
    return launch_status();
}

// The query projection's GEMM writes q_nope / q_pe itself, rotating q^R in
// its epilogue, when its output tiles alone give at least half of the SMs
// work; with fewer (few heads, a long K) it splits K into fp32 partials that
// the finishing kernel adds up.  `fused` says which; the workspace is that
// of the plan returned (none for the direct one).  A direct plan whose N
// tile's sin / cos table (BN x d_r/2 pairs) fits ROPE_TABLE_MAX keeps it in
// shared memory (`table`), planned with those bytes taken from the ring.
GemmPlan project_q_plan(int M, int N, int d, int d_r, int sms, bool& fused, bool& table) {
    GemmPlan direct = gemm_plan(M, N, d, 1, sms, kNoSplit);
    fused = direct.items >= (sms + 1) / 2;
    table = false;
    if (!fused) return gemm_plan(M, N, d, 1, sms, kSplitParts);
    const size_t tab = (size_t)direct.BN * (d_r / 2) * sizeof(float2);
    if (tab <= (size_t)mla::gemm::ROPE_TABLE_MAX) {
        const GemmPlan with = gemm_plan(M, N, d, 1, sms, kNoSplit, 64, true, tab);
        if (with.BN == direct.BN) {
            table = true;
            return with;
        }
    }
    return direct;
}

size_t mla_project_q_workspace_size(int N, int H, int d_h, int d_r, int d, mla_dtype_t dtype) {
    if (dtype != MLA_BF16 || N < 1 || H < 1 || d_h < 1 || d_r < 1 || d < 64) return 0;
    const int64_t M = (int64_t)H * (d_h + d_r);
    if (M % 128 != 0 || M > (1 << 30)) return 0;
    DeviceInfo di;
    if (!device_info(di)) return 0;
    bool fused = false, table = false;
    return plain_gemm_ws_bytes(project_q_plan((int)M, N, d, d_r, di.sms, fused, table));
}

mla_status_t mla_project_q(const void* h, const void* w_q, const int32_t* positions, void* q_nope,
                           void* q_pe, int N, int H, int d_h, int d_r, int d, double rope_base,
                           void* workspace, size_t workspace_bytes, mla_dtype_t dtype,
                           mla_stream_t stream) {
    if (!h || !w_q || !positions || !q_nope || !q_pe) return MLA_ERR_INVALID_ARG;
    // RoPE rotates pairs: an odd d_r has no meaning
    if (N < 1 || H < 1 || d_h < 1 || d_r < 2 || (d_r % 2) != 0 || d < 1 || !(rope_base > 0.0))
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(h) || !aligned16(w_q) || !aligned16(q_nope) || !aligned16(q_pe))
        return MLA_ERR_INVALID_ARG;
    if (dtype != MLA_BF16 && dtype != MLA_FP32) return MLA_ERR_INVALID_ARG;
    if (d_h % 2 != 0 || d_r > 2 * mla::pro::MAX_PAIRS) return MLA_ERR_UNSUPPORTED;
    const int64_t M = (int64_t)H * (d_h + d_r);
    if (M > (1 << 30)) return MLA_ERR_UNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    mla::pro::QParams p;
    p.h = h;
    p.w_q = w_q;
    p.parts = nullptr;
    p.splits = 0;
    p.positions = positions;
    p.q_nope = q_nope;
    p.q_pe = q_pe;
    p.N = N;
    p.d = d;
    p.H = H;
    p.d_h = d_h;
    p.d_r = d_r;
    if (!rope_freqs(p.freq, d_r, rope_base)) return MLA_ERR_INVALID_ARG;
    if (dtype == MLA_FP32) {
        const int64_t gy = (M + mla::pro::ROWS - 1) / mla::pro::ROWS;
        if (d % 4 != 0 || gy > 65535) return MLA_ERR_UNSUPPORTED;
        const dim3 grid((unsigned)((N + mla::pro::TOK - 1) / mla::pro::TOK), (unsigned)gy);
        mla::pro::q_rows_fp32_kernel<<<grid, mla::pro::THREADS, 0, st>>>(p);
        return launch_status();
    }
    if (M % 128 != 0 || d % 64 != 0 || d_h % 8 != 0 || d_r % 8 != 0) return MLA_ERR_UNSUPPORTED;
    const int threads = mla::pro::Q_HEADS * (d_h + d_r) / 2;
    if (threads > 1024 || (H + mla::pro::Q_HEADS - 1) / mla::pro::Q_HEADS > 65535)
        return MLA_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (!device_info(di)) return MLA_ERR_CUDA;
    bool fused = false, table = false;
    const GemmPlan g = project_q_plan((int)M, N, d, d_r, di.sms, fused, table);
    const size_t need = plain_gemm_ws_bytes(g);
    if (need > 0 && (!workspace || !aligned16(workspace) || workspace_bytes < need))
        return MLA_ERR_INVALID_ARG;
    if (fused) {
        // W^Q h on the tensor cores, the epilogue splitting each row per
        // head and rotating q^R before the one rounding: one launch
        CUtensorMap ta, tx;
        if (!weight_map(&ta, w_q, (int)M, d) || !rows_map(&tx, h, N, d, d, g.BN)) return MLA_ERR_CUDA;
        const QRopeOut qo{static_cast<__nv_bfloat16*>(q_nope), static_cast<__nv_bfloat16*>(q_pe), positions,
                          H, d_h, d_r, p.freq, table ? 1 : 0};
        return launch_gemm(ta, ta, g.m_tiles, tx, (int)M, N, d, 1, 0, 0, g, nullptr, 0, 0, nullptr, nullptr, st,
                           &qo);
    }
    // W^Q h on the tensor cores, each K split's fp32 partial into the
    // workspace; then the finishing kernel adds the splits, splits each row
    // per head, rotates q^R and rounds once
    mla_status_t s = plain_gemm(w_q, h, nullptr, 0, (int)M, N, d, g, workspace, st);
    if (s != MLA_OK) return s;
    p.parts = ws_parts(g, workspace);
    p.splits = g.splits;
    const dim3 grid((unsigned)N, (unsigned)((H + mla::pro::Q_HEADS - 1) / mla::pro::Q_HEADS));
    s = launch_pdl(mla::pro::q_finish_bf16_kernel, grid, dim3((unsigned)threads), 0, st, p);
    if (s != MLA_OK) return s;
    return launch_status();
}

// ------------------------------------------------------------- prefill

size_t mla_prefill_workspace_size(int rows, int H, int d_h, int d, mla_dtype_t dtype) {
    if (dtype != MLA_BF16 || rows < 1 || H < 1 || d_h < 1 || d < 128) return 0;
    const int64_t K = (int64_t)H * d_h;
    if (K > (1 << 30)) return 0;
    DeviceInfo di;
    if (!device_info(di)) return 0;
    return plain_gemm_ws_bytes(gemm_plan(d, rows, (int)K, 1, di.sms, kSplitReduce));
}

mla_status_t mla_prefill_expand(const void* kv, const void* w_uk, const void* w_uv, void* k_nope,
                                void* v, int rows, int H, int d_h, int d_c, int d_r,
                                mla_dtype_t dtype, mla_stream_t stream) {
    if (!kv || !w_uk || !w_uv || !k_nope || !v || rows < 1 || H < 1 || d_h < 1 || d_c < 1 || d_r < 0)
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(kv) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(k_nope) || !aligned16(v))
        return MLA_ERR_INVALID_ARG;
    if (dtype != MLA_BF16) return dtype == MLA_FP32 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
    const int64_t M = (int64_t)H * d_h;
    if (M % 128 != 0 || d_c % 64 != 0 || ((d_c + d_r) * 2) % 16 != 0 || M > (1 << 30))
        return MLA_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (!device_info(di)) return MLA_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // K_nope[r, i, :] = W^UK_i c_r and V[r, i, :] = W^UV_i c_r: the stacked
    // [H * d_h x d_c] weight on the UMMA M axis, the latents c (the first d_c
    // values of each cache row) on N, no split of the short reduction
    const GemmPlan g = gemm_plan((int)M, rows, d_c, 1, di.sms, kNoSplit);
    mla_status_t s = plain_gemm(w_uk, kv, static_cast<__nv_bfloat16*>(k_nope), M, (int)M, rows, d_c, g,
                                nullptr, st, d_c + d_r);
    if (s != MLA_OK) return s;
    return plain_gemm(w_uv, kv, static_cast<__nv_bfloat16*>(v), M, (int)M, rows, d_c, g, nullptr, st,
                      d_c + d_r);
}

mla_status_t mla_prefill_attn(const void* q_nope, const void* q_pe, const void* k_nope,
                              const void* kv, const void* v, int B, int L, int H, int d_h, int d_c,
                              int d_r, float scale, int causal, void* u, float* lse,
                              mla_dtype_t dtype, mla_stream_t stream) {
    if (!q_nope || !q_pe || !k_nope || !kv || !v || !u || !lse) return MLA_ERR_INVALID_ARG;
    if (B < 1 || L < 1 || H < 1 || d_h < 1 || d_c < 1 || d_r < 1 || !std::isfinite(scale))
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(k_nope) || !aligned16(kv) ||
        !aligned16(v) || !aligned16(u))
        return MLA_ERR_INVALID_ARG;
    if (dtype != MLA_BF16) return dtype == MLA_FP32 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
    if (d_h != mla::pre::DH || d_r != mla::pre::DR || d_c % 64 != 0) return MLA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)B * L;
    if (rows > INT32_MAX - mla::pre::BK || H > 65535 || B > 65535) return MLA_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (!device_info(di)) return MLA_ERR_CUDA;
    CUtensorMap tm_kn, tm_kr, tm_v;
    {   // k_nope, v: [rows][H][128]; a box is 128 rows x 64 dims of one head
        const cuuint64_t dims[3] = {(cuuint64_t)d_h, (cuuint64_t)H, (cuuint64_t)rows};
        const cuuint64_t strides[2] = {(cuuint64_t)d_h * 2, (cuuint64_t)H * d_h * 2};
        const cuuint32_t box[3] = {64, 1, (cuuint32_t)mla::pre::BK};
        if (!make_map(&tm_kn, k_nope, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&tm_v, v, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return MLA_ERR_CUDA;
    }
    {   // the cache rows [c ; k^R]: the RoPE key is the 64 columns from d_c on
        const cuuint64_t dims[2] = {(cuuint64_t)(d_c + d_r), (cuuint64_t)rows};
        const cuuint64_t strides[1] = {(cuuint64_t)(d_c + d_r) * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)mla::pre::BK};
        if (!make_map(&tm_kr, kv, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MLA_ERR_CUDA;
    }
    mla::pre::Params p;
    p.q_nope = static_cast<const __nv_bfloat16*>(q_nope);
    p.q_pe = static_cast<const __nv_bfloat16*>(q_pe);
    p.u = static_cast<__nv_bfloat16*>(u);
    p.lse = lse;
    p.B = B;
    p.L = L;
    p.H = H;
    p.nqb = (L + mla::pre::BQ - 1) / mla::pre::BQ;
    p.scale_log2 = scale * mla::dec::LOG2E;
    p.causal = causal ? 1 : 0;
    p.rope_col = d_c;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const dim3 grid((unsigned)p.nqb, (unsigned)H, (unsigned)B);
    mla::pre::prefill_bf16_kernel<<<grid, mla::pre::THREADS, mla::pre::SMEM_ALLOC, st>>>(tm_kn, tm_kr,
                                                                                         tm_v, p);
    return launch_status();
}

mla_status_t mla_prefill_out(const void* u, const void* w_o, void* out, int rows, int H, int d_h,
                             int d, void* workspace, size_t workspace_bytes, mla_dtype_t dtype,
                             mla_stream_t stream) {
    if (!u || !w_o || !out || rows < 1 || H < 1 || d_h < 1 || d < 1) return MLA_ERR_INVALID_ARG;
    if (!aligned16(u) || !aligned16(w_o) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
    if (dtype != MLA_BF16) return dtype == MLA_FP32 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
    const int64_t K = (int64_t)H * d_h;
    if (d % 128 != 0 || K % 64 != 0 || K > (1 << 30)) return MLA_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (!device_info(di)) return MLA_ERR_CUDA;
    const GemmPlan g = gemm_plan(d, rows, (int)K, 1, di.sms, kSplitReduce);
    if (g.mode != mla::gemm::OUT_BF16 &&
        (!workspace || !aligned16(workspace) || workspace_bytes < plain_gemm_ws_bytes(g)))
        return MLA_ERR_INVALID_ARG;
    // out = W^O u: W^O [d x H * d_h] on the UMMA M axis, the rows of u on N
    return plain_gemm(w_o, u, static_cast<__nv_bfloat16*>(out), d, d, rows, (int)K, g, workspace,
                      reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------- mla_combine

mla_status_t mla_combine_splits(const float* o_part, const float* lse_part, int S, int64_t rows,
                                int d_c, void* o, float* lse, mla_dtype_t dtype,
                                mla_stream_t stream) {
    if (!o_part || !lse_part || !o || !lse || S < 1 || S > 1024 || rows < 1 || d_c < 4 ||
        d_c % 4 != 0)
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(o_part) || !aligned16(o)) return MLA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const unsigned blocks = (unsigned)((rows + 3) / 4);
    if (dtype == MLA_FP32)
        mla::combine_kernel<float><<<blocks, 128, 0, st>>>(o_part, lse_part, S, rows, d_c,
                                                           static_cast<float*>(o), lse);
    else if (dtype == MLA_BF16)
        mla::combine_kernel<__nv_bfloat16><<<blocks, 128, 0, st>>>(
            o_part, lse_part, S, rows, d_c, static_cast<__nv_bfloat16*>(o), lse);
    else
        return MLA_ERR_INVALID_ARG;
    return launch_status();
}

// ------------------------------------------------------------ mla_decode

size_t mla_decode_workspace_size(int B, int T, int H, int d_c, mla_dtype_t dtype) {
    if (dtype != MLA_BF16 || B < 1 || T < 1 || H < 1 || d_c < 1) return 0;
    DeviceInfo di;
    if (!device_info(di)) return 0;
    const int64_t HG = (H + mla::dec::HEADS - 1) / mla::dec::HEADS;
    return decode_ws_layout((int64_t)B * T * HG, di.decode_clusters, d_c).total;
}

int64_t mla_decode_plan(const int32_t* seq_lens_host, int B, int T, int H, int max_pages,
                        int causal, int clusters, int64_t* out, int64_t cap) {
    if (!seq_lens_host || B < 1 || T < 1 || H < 1 || max_pages < 1 || clusters < 0 || cap < 0 ||
        (cap > 0 && !out))
        return -1;
    if (clusters == 0) {
        DeviceInfo di;
        if (!device_info(di)) return -1;
        clusters = di.decode_clusters;
    }
    const int HG = (H + mla::dec::HEADS - 1) / mla::dec::HEADS;
    if (!mla::dec::plan_fits_int32(B, T, HG, max_pages)) return -1;
    mla::dec::PlanView v{seq_lens_host, B, T, HG, max_pages, causal ? 1 : 0};
    // as mla_decode_attn launches it: one cluster per unit where that cuts none
    clusters = whole_unit_clusters(seq_lens_host, B, T, HG, max_pages, causal ? 1 : 0, clusters);
    int64_t n = 0;
    for (int g = 0; g < clusters; ++g) {
        mla::dec::Walker w = mla::dec::host_walker(v, clusters, g);
        mla::dec::Segment sg;
        while (w.next(v, sg)) {
            if (n < cap) {
                int64_t* r = out + 7 * n;
                r[0] = g;
                r[1] = sg.u;
                r[2] = sg.lp0;
                r[3] = sg.lp1;
                r[4] = sg.slot;
                r[5] = sg.g_first;
                r[6] = sg.g_last;
            }
            ++n;
        }
    }
    return n;
}

}  // extern "C"

namespace {

// mla_decode_attn (o in the input type) and mla_decode_attn_partial (o in
// fp32 whatever the input type) share everything but the output type.
mla_status_t decode_impl(const void* q_lat, const void* q_pe, const void* kv_pool,
                         const int32_t* page_table, const int32_t* seq_lens,
                         const int32_t* seq_lens_host, int B, int T, int H, int d_c, int d_r,
                         int page_size, int max_pages, int64_t num_pages, float scale, int causal,
                         void* o, bool o_f32, float* lse, void* workspace, size_t workspace_bytes,
                         mla_dtype_t dtype, mla_stream_t stream) {
    if (!q_lat || !q_pe || !kv_pool || !page_table || !seq_lens || !o || !lse)
        return MLA_ERR_INVALID_ARG;
    if (B < 1 || T < 1 || H < 1 || d_c < 1 || d_r < 0 || page_size < 1 || max_pages < 1 ||
        num_pages < 1 || !std::isfinite(scale))
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_lat) || !aligned16(q_pe) || !aligned16(kv_pool) || !aligned16(o))
        return MLA_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == MLA_FP32) {
        if (d_c > mla::FP32_MAX_DC || d_r > mla::FP32_MAX_DR || d_c % 4 != 0)
            return MLA_ERR_UNSUPPORTED;
        dim3 grid((unsigned)B * T, (unsigned)H);
        mla::decode_fp32_kernel<<<grid, mla::FP32_WARPS * 32, 0, st>>>(
            static_cast<const float*>(q_lat), static_cast<const float*>(q_pe),
            static_cast<const float*>(kv_pool), page_table, seq_lens, T, H, d_c, d_r, page_size,
            max_pages, num_pages, scale, causal ? 1 : 0, static_cast<float*>(o), lse);
        return launch_status();
    }
    if (dtype != MLA_BF16) return MLA_ERR_INVALID_ARG;
    if (d_c != mla::dec::DC || d_r != mla::dec::DR || page_size != mla::dec::PAGE)
        return MLA_ERR_UNSUPPORTED;
    if (num_pages * mla::dec::PAGE > INT32_MAX) return MLA_ERR_UNSUPPORTED;
    const int HG = (H + mla::dec::HEADS - 1) / mla::dec::HEADS;
    if (!mla::dec::plan_fits_int32(B, T, HG, max_pages)) return MLA_ERR_UNSUPPORTED;
    DeviceInfo di;
    if (!device_info(di)) return MLA_ERR_CUDA;
    const int64_t U = (int64_t)B * T * HG;
    const int64_t G = di.decode_clusters;
    const DecodeWs wl = decode_ws_layout(U, G, d_c);
    if (!workspace || workspace_bytes < wl.total || !aligned16(workspace))
        return MLA_ERR_INVALID_ARG;

    CUtensorMap tm_c, tm_r;
    const cuuint64_t dims[2] = {(cuuint64_t)(d_c + d_r), (cuuint64_t)num_pages * page_size};
    const cuuint64_t strides[1] = {(cuuint64_t)(d_c + d_r) * 2};
    // one 32-token tile of a page per copy: the ring holds half pages
    const cuuint32_t box_c[2] = {64, (cuuint32_t)mla::dec::TILE};
    const cuuint32_t box_r[2] = {(cuuint32_t)mla::dec::HALF_R, (cuuint32_t)mla::dec::TILE};
    if (!make_map(&tm_c, kv_pool, 2, dims, strides, box_c, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tm_r, kv_pool, 2, dims, strides, box_r, CU_TENSOR_MAP_SWIZZLE_64B))
        return MLA_ERR_CUDA;

    Params p;
    p.q_lat = static_cast<const __nv_bfloat16*>(q_lat);
    p.q_pe = static_cast<const __nv_bfloat16*>(q_pe);
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.o = o_f32 ? nullptr : static_cast<__nv_bfloat16*>(o);
    p.o32 = o_f32 ? static_cast<float*>(o) : nullptr;
    p.lse = lse;
    char* ws = static_cast<char*>(workspace);
    p.ws_unit = reinterpret_cast<int2*>(ws + wl.unit_off);
    p.ws_lse = reinterpret_cast<float*>(ws + wl.lse_off);
    p.ws_o = reinterpret_cast<float*>(ws + wl.o_off);
    p.B = B;
    p.T = T;
    p.H = H;
    p.HG = HG;
    p.max_pages = max_pages;
    p.num_pages = num_pages;
    p.scale_log2 = scale * mla::dec::LOG2E;
    p.causal = causal ? 1 : 0;

    cudaEvent_t ev0 = g_ev_start, ev1 = g_ev_end;
    // Inside a stream capture an event record only orders the graph unless it
    // is recorded as external; then replaying the graph records it.
    unsigned ev_flags = cudaEventRecordDefault;
    if (ev0 && ev1) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return MLA_ERR_CUDA;
        if (cs == cudaStreamCaptureStatusActive) ev_flags = cudaEventRecordExternal;
    }
    if (ev0 && ev1 && cudaEventRecordWithFlags(ev0, st, ev_flags) != cudaSuccess) return MLA_ERR_CUDA;
    const int64_t Gl = seq_lens_host ? whole_unit_clusters(seq_lens_host, B, T, HG, max_pages, p.causal, (int)G) : G;
    mla::dec::decode_bf16_kernel<<<(unsigned)(2 * Gl), mla::dec::THREADS, mla::dec::SMEM_ALLOC, st>>>(
        tm_c, tm_r, p);
    if (launch_status() != MLA_OK) return MLA_ERR_CUDA;
    if (ev0 && ev1 && cudaEventRecordWithFlags(ev1, st, ev_flags) != cudaSuccess) return MLA_ERR_CUDA;
    if (seq_lens_host &&
        !host_plan_needs_combine(seq_lens_host, B, T, HG, max_pages, p.causal, (int)Gl))
        return MLA_OK;
    mla::dec::decode_combine_kernel<<<(unsigned)((U * mla::dec::HEADS + mla::dec::COMBINE_ROWS - 1) /
                                                 mla::dec::COMBINE_ROWS),
                                      32 * mla::dec::COMBINE_ROWS, 0, st>>>(p);
    return launch_status();
}

}  // namespace

extern "C" {

mla_status_t mla_decode_attn(const void* q_lat, const void* q_pe, const void* kv_pool,
                             const int32_t* page_table, const int32_t* seq_lens,
                             const int32_t* seq_lens_host, int B, int T, int H, int d_c,
                             int d_r, int page_size, int max_pages, int64_t num_pages,
                             float scale, int causal, void* o, float* lse, void* workspace,
                             size_t workspace_bytes, mla_dtype_t dtype, mla_stream_t stream) {
    return decode_impl(q_lat, q_pe, kv_pool, page_table, seq_lens, seq_lens_host, B, T, H, d_c, d_r,
                       page_size, max_pages, num_pages, scale, causal, o, false, lse, workspace,
                       workspace_bytes, dtype, stream);
}

mla_status_t mla_decode_attn_partial(const void* q_lat, const void* q_pe, const void* kv_pool,
                                     const int32_t* page_table, const int32_t* seq_lens,
                                     const int32_t* seq_lens_host, int B, int T, int H, int d_c,
                                     int d_r, int page_size, int max_pages, int64_t num_pages,
                                     float scale, int causal, float* o, float* lse,
                                     void* workspace, size_t workspace_bytes, mla_dtype_t dtype,
                                     mla_stream_t stream) {
    return decode_impl(q_lat, q_pe, kv_pool, page_table, seq_lens, seq_lens_host, B, T, H, d_c, d_r,
                       page_size, max_pages, num_pages, scale, causal, o, dtype == MLA_BF16, lse,
                       workspace, workspace_bytes, dtype, stream);
}

// ----------------------------------------------- mla_decode_attn_noalloc

}  // extern "C"

namespace {

// Scratch for mla_decode_attn_noalloc: a fixed array in device memory that
// the CUDA runtime sets aside on every GPU that loads this library, for as
// long as the process lives.  Calls share it and it keeps the last call's
// contents (the decode scratch needs no initial value).  64 MiB holds the
// decode scratch of up to 255 - (co-resident clusters) work units (sequence
// x query token x 128-head group) -- 181 on a 148-SM B300, e.g. B = 128
// sequences of one token and 128 heads.
constexpr size_t kNoallocScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_decode_scratch[kNoallocScratchBytes];

// Device address of g_decode_scratch, looked up with the device current and
// cached per device together with the unique id of the CUDA context it was
// looked up in.  A context created later on the same device (after
// cudaDeviceReset, say) has another id, so its first call looks the address
// up again instead of reusing a stale one.  In host code the array's name is
// only a stand-in for the symbol, never a device address.
struct ScratchAddr {
    bool valid = false;
    unsigned long long ctx_id = 0;
    void* addr = nullptr;
};
ScratchAddr g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (false when there is
// none, or the driver does not offer the query).
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

void* decode_scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchAddr& e = g_scratch_addr[dev];
    unsigned long long id = 0;
    bool have_id = current_context_id(&id);
    if (have_id && e.valid && e.ctx_id == id) return e.addr;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (!have_id) have_id = current_context_id(&id);  // the lookup made the context current
    e.valid = have_id;  // without a context id the address is looked up on every call
    e.ctx_id = id;
    e.addr = ptr;
    return ptr;
}

}  // namespace

extern "C" {

size_t mla_decode_noalloc_max_bytes(void) { return kNoallocScratchBytes; }

mla_status_t mla_decode_attn_noalloc(const void* q_lat, const void* q_pe, const void* kv_pool,
                                     const int32_t* page_table, const int32_t* seq_lens,
                                     const int32_t* seq_lens_host, int B, int T, int H, int d_c,
                                     int d_r, int page_size, int max_pages, int64_t num_pages,
                                     float scale, int causal, void* o, float* lse,
                                     mla_dtype_t dtype, mla_stream_t stream) {
    if (!q_lat || !q_pe || !kv_pool || !page_table || !seq_lens || !o || !lse)
        return MLA_ERR_INVALID_ARG;
    if (dtype != MLA_BF16 && dtype != MLA_FP32) return MLA_ERR_INVALID_ARG;
    if (B < 1 || T < 1 || H < 1 || d_c < 1) return MLA_ERR_INVALID_ARG;
    const size_t need = mla_decode_workspace_size(B, T, H, d_c, dtype);
    if (need > kNoallocScratchBytes) return MLA_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (need > 0) {
        scratch = decode_scratch_address();
        if (!scratch) return MLA_ERR_CUDA;
    }
    return mla_decode_attn(q_lat, q_pe, kv_pool, page_table, seq_lens, seq_lens_host, B, T, H, d_c,
                           d_r, page_size, max_pages, num_pages, scale, causal, o, lse, scratch,
                           need > 0 ? kNoallocScratchBytes : 0, dtype, stream);
}

}  // extern "C"
