/*
 * mla.h -- C ABI of libmla: weight-absorbed Multi-head Latent Attention (MLA)
 * decode for NVIDIA B300 (sm_103a).
 *
 * The decode step of one attention layer, for query token t of sequence b and
 * head i, against the cached rows [c_j ; k^R_j] of positions j:
 *
 *   c_j = W^DKV h_j, k^R_j = RoPE(W^KR h_j), into the pool     mla_cache_append
 *   q^C_i, q^R_i = W^Q h (per head), q^R_i rotated             mla_project_q
 *   q_lat_i = W^UK_i^T q^C_i                                   mla_absorb_q
 *   s_ij    = (q_lat_i . c_j + q^R_i . k^R_j) * scale          mla_decode_attn
 *   o_i     = sum_j softmax_j(s_ij) c_j,  lse_i = ln sum_j e^{s_ij}
 *   (pieces of one softmax merged by log-sum-exp)              mla_combine_splits
 *   out     = W^O concat_i (W^UV_i o_i)                        mla_out_proj
 *           (or with W^O W^UV merged ahead of time: mla_fold_out_weights,
 *            mla_out_proj_merged)
 *
 * Sources (web pages on MLA):
 *   [Mishra] "Multi-head Latent Attention", Neel Mishra: sections "Step 2:
 *            absorb the up-projections" and "Step 4: decoupled RoPE".
 *   [Zhang]  zhangchitc.github.io MLA post: "Matrix absorption: compression
 *            that also saves compute", "Decoupled RoPE", "Value absorption:
 *            weight and sum first, project after".
 *   [llms]   "Multi-Head Latent Attention: How Low-Rank KV Compression
 *            Scales LLM Serving": "Low-Rank Key-Value Joint Compression",
 *            "Query Key Absorption", "Value Output Absorption".
 *
 * Conventions for every entry point:
 *   - Pointers are device pointers unless the name ends in _host.  All
 *     buffers, workspaces included, are owned by the caller; the library
 *     allocates no device memory.  Tensors are dense, row-major, in the
 *     stated shape, and 16-byte aligned.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream).
 *   - Argument errors are returned before anything is launched.  Errors found
 *     on the device (a bounded wait that gave up, an out-of-range page id or
 *     length) raise a device status word that mla_get_device_status() reads;
 *     while it is raised, later calls' kernels return without results.
 *   - dtype MLA_BF16: bf16 tensors (except lse and partials, always fp32),
 *     tensor-core (tcgen05) kernels, fp32 accumulation.  dtype MLA_FP32: fp32
 *     tensors, CUDA-core kernels in fp32.  Shapes the bf16 kernels do not
 *     cover return MLA_ERR_UNSUPPORTED; there is no fallback.
 *   - The projection GEMMs and the prologue's second kernels are launched
 *     with programmatic stream serialization: they may start their set-up
 *     while the kernel before them on the stream finishes, and wait for it
 *     before touching memory it writes or reads (the cache write's second
 *     kernel looks up its pool rows in the call's inputs first: that kernel
 *     is the call's own GEMM, which writes only its partials).  They also
 *     let the next kernel launch
 *     early; a kernel of the caller's launched that way must wait
 *     (griddepcontrol.wait) before reading what they write.
 *   - The prefill calls (mla_prefill_*) and the merged-query calls also
 *     follow from the same pages ([Mishra] "Multi-head Latent Attention":
 *     the unabsorbed form in training; the fold done once offline).
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream). */
typedef struct CUstream_st* mla_stream_t;

typedef enum mla_status {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment, short workspace */
    MLA_ERR_UNSUPPORTED = 2,   /* valid shape the kernels of this dtype do not cover    */
    MLA_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch or query)          */
    MLA_ERR_TIMEOUT = 4,       /* device: a bounded wait gave up                         */
    MLA_ERR_DEVICE_BOUNDS = 5  /* device: page id or sequence length out of range       */
} mla_status_t;

typedef enum mla_dtype { MLA_BF16 = 0, MLA_FP32 = 1 } mla_dtype_t;

/*
 * mla_absorb_q -- query-side weight absorption, per head:
 *     q_lat[r, i, :] = W^UK_i^T q_nope[r, i, :]
 * ([llms] "Query Key Absorption"; [Mishra] "Step 2: absorb the
 * up-projections"; [Zhang] "Matrix absorption": the up-projection is applied
 * once to the query instead of to every cached latent.)
 *
 *   q_nope [rows, H, d_h]   content part of the query (q^C), rows = B*T
 *   w_uk   [H, d_h, d_c]    W^UK in R^{H*d_h x d_c}; head i owns rows
 *                            i*d_h .. (i+1)*d_h-1
 *   q_lat  [rows, H, d_c]   output
 * bf16: d_c % 128 == 0, d_h % 64 == 0, rows >= 1.
 */
mla_status_t mla_absorb_q(const void* q_nope, const void* w_uk, void* q_lat, int rows, int H,
                          int d_h, int d_c, mla_dtype_t dtype, mla_stream_t stream);

/*
 * Bytes of device workspace mla_decode_attn needs for this shape on the
 * current device (0 for MLA_FP32).  The content need not be initialised.
 */
size_t mla_decode_workspace_size(int B, int T, int H, int d_c, mla_dtype_t dtype);

/*
 * mla_decode_attn -- absorbed decode attention against a paged latent cache.
 * For every sequence b, query token t < T and head i < H:
 *     s_j  = (q_lat[b,t,i,:] . c_j + q_pe[b,t,i,:] . k^R_j) * scale
 *     o    = sum_j softmax_j(s) c_j,     lse = ln sum_j exp(s_j)
 * over the visible positions j: 0 .. seq_lens[b]-1, or with causal != 0,
 * 0 .. seq_lens[b]-T+t (query t sits at position seq_lens[b]-T+t).
 * ([llms] "Query Key Absorption": scores of the absorbed query against the
 * cached latent plus the decoupled RoPE term; [Zhang] "Decoupled RoPE" and
 * "Value absorption": the sum is scaled (the pages use 1/sqrt(d_h + d_r))
 * and soft-maxed, and the weights mix the latents c_j, which are never
 * expanded to keys or values; [Mishra] "Step 4: decoupled RoPE": the cache
 * row is [c_j ; k^R_j], d_c + d_r numbers shared by all heads.)
 * A query that sees no position gets o = 0 and lse = -inf.
 *
 *   q_lat      [B, T, H, d_c]            absorbed content query
 *   q_pe       [B, T, H, d_r]            RoPE query (already rotated)
 *   kv_pool    [num_pages, page_size, d_c + d_r]   cache rows [c ; k^R]
 *                                        (k^R already rotated); rows past a
 *                                        sequence's length are ignored and
 *                                        may hold anything
 *   page_table [B, max_pages] int32      position j of sequence b is row
 *                                        j % page_size of pool page
 *                                        page_table[b][j / page_size];
 *                                        entries past the last page unused
 *   seq_lens   [B] int32 (device)        cached positions per sequence
 *   seq_lens_host [B] int32 or NULL      the same lengths in host memory; when
 *                                        given, the combine launch is skipped
 *                                        if no sequence is split
 *   o          [B, T, H, d_c]            output (dtype)
 *   lse        [B, T, H] fp32            output, natural log
 *   workspace  >= mla_decode_workspace_size(B, T, H, d_c, dtype) bytes
 * bf16 kernels: d_c == 512, d_r == 64, page_size == 64, any H >= 1 (heads
 * are processed in groups of 128), any T >= 1.  The fp32 kernels take
 * d_c <= 512 (multiple of 4), d_r <= 64, any page_size.
 * Work is balanced over all SMs: long or ragged sequences are split across
 * SMs and merged by log-sum-exp inside this call (a second kernel).
 */
mla_status_t mla_decode_attn(const void* q_lat, const void* q_pe, const void* kv_pool,
                             const int32_t* page_table, const int32_t* seq_lens,
                             const int32_t* seq_lens_host, int B, int T, int H, int d_c,
                             int d_r, int page_size, int max_pages, int64_t num_pages,
                             float scale, int causal, void* o, float* lse, void* workspace,
                             size_t workspace_bytes, mla_dtype_t dtype, mla_stream_t stream);

/*
 * mla_decode_attn_partial -- mla_decode_attn with o written in fp32 whatever
 * the input type (dtype MLA_BF16 reads bf16 q_lat, q_pe and kv_pool; fp32
 * mode is mla_decode_attn itself), for attention over one part of a
 * sequence's cache whose result is merged with the other parts' later.
 * o is then that part's normalised result and lse its log-sum-exp; the
 * parts of one softmax merge exactly by
 *     lse = ln sum_s e^{lse_s},   o = sum_s e^{lse_s - lse} o_s
 * (mla_combine_splits), since the softmax over all positions weights each
 * part's normalised result by that part's share of the total.  This is the
 * exchange of one long sequence sharded by token range over several GPUs
 * ([llms] "Hardware Trade-offs and Tensor Parallelism": the latent must be
 * split or communicated across GPUs): each GPU runs this call on the pages
 * it holds, the (o, lse) pairs are all-gathered, and mla_combine_splits
 * merges them.  A part a query sees nothing of gives o = 0, lse = -inf,
 * which the merge weighs by 0.
 *
 *   o    [B, T, H, d_c] fp32 output; other arguments as mla_decode_attn
 *   workspace >= mla_decode_workspace_size(B, T, H, d_c, dtype) bytes
 */
mla_status_t mla_decode_attn_partial(const void* q_lat, const void* q_pe, const void* kv_pool,
                                     const int32_t* page_table, const int32_t* seq_lens,
                                     const int32_t* seq_lens_host, int B, int T, int H, int d_c,
                                     int d_r, int page_size, int max_pages, int64_t num_pages,
                                     float scale, int causal, float* o, float* lse,
                                     void* workspace, size_t workspace_bytes, mla_dtype_t dtype,
                                     mla_stream_t stream);

/*
 * mla_decode_plan -- how mla_decode_attn (bf16) divides a batch over the GPU,
 * computed on the host from the same arithmetic the kernel uses.
 * The pages of all units u = (t*ceil(H/128) + head_group)*B + b are laid end
 * to end on a line where each non-empty unit after the first is preceded by
 * 3 virtual pages when the line holds at least 8 pages per cluster (starting
 * a unit piece costs a cluster about that much), and the line is cut into
 * min(clusters, total pages) equal contiguous ranges, one per 2-CTA cluster;
 * a unit cut by a range boundary is computed in pieces whose partial results
 * are merged by log-sum-exp.  When every non-empty unit has the same number
 * of pages n, there are no more units than clusters, and n exceeds the
 * largest range of the cut by at most 16 pages, one cluster per unit is
 * launched instead (no unit is cut, no merge step runs); mla_decode_attn
 * does this only when given seq_lens_host.
 *   seq_lens_host [B] int32 (host), clusters: co-resident clusters (0 = the
 *   current device's value).
 *   out: up to `cap` rows of 7 int64: (cluster, unit, first page, end page
 *   (exclusive, within the unit), partial slot or -1 when the unit is whole,
 *   cluster of the unit's first page, cluster of its last page).
 * Returns the number of pieces (which may exceed cap), or -1 on bad
 * arguments.  Units that see no position produce no piece.
 */
int64_t mla_decode_plan(const int32_t* seq_lens_host, int B, int T, int H, int max_pages,
                        int causal, int clusters, int64_t* out, int64_t cap);

/*
 * mla_combine_splits -- merge S partial results of the same softmax rows,
 * each computed over a disjoint subset of the cached positions:
 *     lse = ln sum_s exp(lse_part[s]),   o = sum_s exp(lse_part[s] - lse) o_part[s]
 * A piece with lse_part = -inf carries weight 0; rows whose pieces are all
 * empty get o = 0, lse = -inf.  (The pages define one softmax over all
 * cached positions; this is the same softmax assembled from pieces.)
 *
 *   o_part   [S, rows, d_c] fp32   normalised partial outputs
 *   lse_part [S, rows] fp32        their log-sum-exps
 *   o        [rows, d_c] (dtype),  lse [rows] fp32
 * d_c % 4 == 0, 1 <= S <= 1024.
 */
mla_status_t mla_combine_splits(const float* o_part, const float* lse_part, int S, int64_t rows,
                                int d_c, void* o, float* lse, mla_dtype_t dtype,
                                mla_stream_t stream);

/*
 * Bytes of device workspace mla_out_proj needs (0 for MLA_FP32).  The
 * workspace must be zero-filled before its first use; every call leaves its
 * counters at zero again.
 */
size_t mla_out_proj_workspace_size(int rows, int H, int d_h, int d, mla_dtype_t dtype);

/*
 * mla_out_proj -- output side of the absorbed layer:
 *     v[r, i*d_h : (i+1)*d_h] = W^UV_i o[r, i, :]          (d_c -> d_h per head)
 *     out[r, :]                = W^O v[r, :]               (H*d_h -> d)
 * ([llms] "Value Output Absorption"; [Zhang] "Value absorption": W^UV is
 * pulled out of the weighted sum and applied once; the two weights are kept
 * apart rather than merged into one larger matrix.)
 *
 *   o     [rows, H, d_c]     latent outputs of mla_decode_attn
 *   w_uv  [H, d_h, d_c]      W^UV, head i owns rows i*d_h .. (i+1)*d_h-1
 *   w_o   [d, H*d_h]         W^O
 *   v_tmp [rows, H*d_h]      intermediate (dtype), caller-owned
 *   out   [rows, d]          output (dtype)
 * bf16: d_h % 128 == 0, d_c % 64 == 0, d % 128 == 0.
 */
mla_status_t mla_out_proj(const void* o, const void* w_uv, const void* w_o, void* v_tmp,
                          void* out, int rows, int H, int d_h, int d_c, int d, void* workspace,
                          size_t workspace_bytes, mla_dtype_t dtype, mla_stream_t stream);

/*
 * mla_fold_out_weights -- the output side's weights merged ahead of time:
 *     W_merged[n, i*d_c : (i+1)*d_c] = W^UV_i^T W^O[n, i*d_h : (i+1)*d_h]
 * so that out = W_merged concat_i o_i = W^O concat_i (W^UV_i o_i).
 * ([Zhang] "Value absorption: weight and sum first, project after": W^UV
 * leaves the weighted sum, and W^O W^UV may be merged ahead of time, at
 * nearly four times the weight bytes for DeepSeek-V3; [Mishra] "Step 2:
 * absorb the up-projections".)  Done once, offline; the result serves
 * mla_out_proj_merged.
 *
 *   w_uv     [H, d_h, d_c]     W^UV
 *   w_o      [d, H*d_h]        W^O
 *   w_merged [d, H*d_c]        output (dtype)
 * Same kernels and limits as mla_absorb_q with rows = d (bf16: d_c % 128
 * == 0, d_h % 64 == 0).
 */
mla_status_t mla_fold_out_weights(const void* w_uv, const void* w_o, void* w_merged, int H, int d_h,
                                  int d_c, int d, mla_dtype_t dtype, mla_stream_t stream);

/*
 * Bytes of device workspace mla_out_proj_merged needs (0 for MLA_FP32);
 * zero-filled before its first use, as for mla_out_proj.
 */
size_t mla_out_proj_merged_workspace_size(int rows, int H, int d_c, int d, mla_dtype_t dtype);

/*
 * mla_out_proj_merged -- the output projection with the merged weight:
 *     out[r, :] = W_merged o[r, :, :] (all heads' latents, H*d_c long)
 * The same result as mla_out_proj up to rounding, streaming d*H*d_c weights
 * instead of H*d_h*(d_c + d): the trade the pages weigh.
 *
 *   o        [rows, H, d_c]    latent outputs of mla_decode_attn
 *   w_merged [d, H*d_c]        from mla_fold_out_weights
 *   out      [rows, d]         output (dtype)
 * bf16: d % 128 == 0, d_c % 64 == 0.
 */
mla_status_t mla_out_proj_merged(const void* o, const void* w_merged, void* out, int rows, int H,
                                 int d_c, int d, void* workspace, size_t workspace_bytes,
                                 mla_dtype_t dtype, mla_stream_t stream);

/*
 * Bytes of device workspace mla_cache_append needs (0 for MLA_FP32): the
 * fp32 partial products of the tensor-core GEMM's K splits ([W^DKV ; W^KR] h,
 * added up by the call's second kernel).  Sized for any d_r <= 128.
 */
size_t mla_cache_append_workspace_size(int N, int d, int d_c, mla_dtype_t dtype);

/*
 * mla_cache_append -- the cache write of N new tokens, the step that feeds
 * the decode: for token n with hidden state h_n at position pos_n of
 * sequence s_n,
 *     c   = W^DKV h_n                      (d -> d_c, the joint latent)
 *     k^R = RoPE(W^KR h_n, pos_n)          (d -> d_r, shared by all heads)
 * and the row [c ; k^R] is stored at row pos_n % page_size of pool page
 * page_table[s_n][pos_n / page_size].
 * ([Mishra] "Step 1: a low-rank latent": only c is cached; "Step 4:
 * decoupled RoPE": the positional key is a separate small projection of h,
 * rotated, one vector for all heads; [llms] "Low-Rank Key-Value Joint
 * Compression" and "The Positional Problem and Decoupled RoPE".)
 * RoPE rotates pair (x_2k, x_2k+1) by the angle pos * rope_base^(-2k/d_r)
 * (y_2k = x_2k cos - x_2k+1 sin, y_2k+1 = x_2k sin + x_2k+1 cos; the pages
 * fix only that the angle depends on the position).  The angle is kept as
 * a fraction of a turn: the host passes each frequency as a 64-bit
 * fixed-point fraction, the kernel multiplies it by the position modulo one
 * turn in integers and takes fp32 sincospi of the top 24 bits (angle error
 * below 2^-25 turns for any int32 position; no fp64 on the device).
 * d_r <= 128.
 *
 *   h          [N, d]                   hidden states of the new tokens
 *   w_dkv      [d_c, d]                 W^DKV
 *   w_kr       [d_r, d]                 W^KR
 *   seq_ids    [N] int32 (device)       sequence of each token, < B
 *   positions  [N] int32 (device)       position of each token in its
 *                                       sequence, < max_pages * page_size
 *   page_table [B, max_pages] int32     as for mla_decode_attn; the entries
 *                                       the tokens land in must be valid
 *   kv_pool    [num_pages, page_size, d_c + d_r]   written in place (only
 *                                       the N rows named by the tokens)
 *   workspace  >= mla_cache_append_workspace_size(N, d, d_c, dtype) bytes
 * Two tokens must not name the same pool row.  A token whose sequence,
 * position or page id is out of range is not written and raises the device
 * status (MLA_ERR_DEVICE_BOUNDS); as after any device error, which of the
 * call's other rows were written is then unspecified (no row outside the
 * tokens' rows is touched).
 * d_r even (MLA_ERR_INVALID_ARG otherwise); d_c even; bf16: d_c % 128 == 0,
 * d % 64 == 0, d_r % 8 == 0; fp32: d % 4 == 0.
 */
mla_status_t mla_cache_append(const void* h, const void* w_dkv, const void* w_kr,
                              const int32_t* seq_ids, const int32_t* positions,
                              const int32_t* page_table, void* kv_pool, int N, int d, int d_c,
                              int d_r, int B, int page_size, int max_pages, int64_t num_pages,
                              double rope_base, void* workspace, size_t workspace_bytes,
                              mla_dtype_t dtype, mla_stream_t stream);

/*
 * Bytes of device workspace mla_project_q needs.  0 for MLA_FP32, and 0 in
 * bf16 when the GEMM's 128-row output tiles alone give at least half of the
 * SMs work (H*(d_h+d_r) = 24576 at DeepSeek widths): its epilogue then splits
 * the rows per head and rotates q^R itself, in one launch.  Otherwise (few
 * heads, a long d) the fp32 partial products of the GEMM's K splits, added
 * up by the call's second kernel.
 */
size_t mla_project_q_workspace_size(int N, int H, int d_h, int d_r, int d, mla_dtype_t dtype);

/*
 * mla_project_q -- the query of N tokens, split per head and rotated:
 *     q = W^Q h_n;  head i takes rows i*(d_h+d_r) .. (i+1)*(d_h+d_r)-1,
 *     the first d_h as q^C_i (-> q_nope), the last d_r as q^R_i, which is
 *     rotated at position pos_n (-> q_pe), with the RoPE of mla_cache_append
 *     (the rotation in fp32; each value rounded once to the output type).
 * ([llms] "The Positional Problem and Decoupled RoPE": each head's query is
 * the concatenation [q^C ; q^R] and only q^R is rotated; [Mishra] "Step 4:
 * decoupled RoPE".)  h may be the model's hidden state (one W^Q) or the
 * compressed query c^Q with W^Q = the stacked up-projections.
 *
 *   h         [N, d]                    input rows
 *   w_q       [H * (d_h + d_r), d]      W^Q, per head [content ; RoPE] rows
 *   positions [N] int32 (device)        position of each token
 *   q_nope    [N, H, d_h]               output, the content query q^C
 *   q_pe      [N, H, d_r]               output, the rotated RoPE query
 *   workspace >= mla_project_q_workspace_size(N, H, d_h, d_r, d, dtype)
 * d_r even (MLA_ERR_INVALID_ARG otherwise); d_h even, d_r <= 128; bf16:
 * H*(d_h+d_r) % 128 == 0, d % 64 == 0, d_h % 8 == 0, d_r % 8 == 0;
 * fp32: d % 4 == 0.
 */
mla_status_t mla_project_q(const void* h, const void* w_q, const int32_t* positions, void* q_nope,
                           void* q_pe, int N, int H, int d_h, int d_r, int d, double rope_base,
                           void* workspace, size_t workspace_bytes, mla_dtype_t dtype,
                           mla_stream_t stream);

/*
 * Query-side weight merge ([Mishra] "Multi-head Latent Attention": the
 * up-projections fold once, offline, W^UK_i^T W^UQ_i; [Zhang] "Matrix
 * absorption: compression that also saves compute").  With the compressed
 * query c^Q (d_q wide) and W^UQ_i the content rows of head i's block of W^Q,
 *     q_lat_i = W^UK_i^T (W^UQ_i c^Q) = (W^UK_i^T W^UQ_i) c^Q
 * so the two products of the unmerged path (mla_project_q's content part,
 * then mla_absorb_q) become one, against a weight of H * d_c * d_q values in
 * place of H * d_h * (d_q + d_c).  The RoPE part of the query still comes
 * from W^QR (mla_project_q).
 *
 * mla_fold_q_weights -- w_merged [d_q, H, d_c]: w_merged[k, i, c] =
 *   sum_e W^UK_i[e, c] W^UQ_i[e, k].
 *   w_uk  [H, d_h, d_c];  w_q [H * (d_h + d_r), d_q] (head i: d_h content
 *   rows, then d_r RoPE rows, as for mla_project_q)
 *   workspace >= mla_fold_q_workspace_size(H, d_h, d_q, dtype) bytes
 * bf16 as mla_absorb_q (d_c % 128 == 0, d_h % 64 == 0); fp32 any size.
 */
size_t mla_fold_q_workspace_size(int H, int d_h, int d_q, mla_dtype_t dtype);
mla_status_t mla_fold_q_weights(const void* w_uk, const void* w_q, void* w_merged, int H, int d_h,
                                int d_r, int d_c, int d_q, void* workspace, size_t workspace_bytes,
                                mla_dtype_t dtype, mla_stream_t stream);

/*
 * mla_absorb_q_merged -- q_lat [rows, H, d_c] = W_merged c^Q for c^Q
 * [rows, d_q] and w_merged [d_q, H, d_c] from mla_fold_q_weights.
 * bf16: H * d_c % 128 == 0, d_q % 64 == 0 (tensor cores); fp32 any size.
 */
mla_status_t mla_absorb_q_merged(const void* c_q, const void* w_merged, void* q_lat, int rows, int H,
                                 int d_c, int d_q, mla_dtype_t dtype, mla_stream_t stream);

/*
 * Prefill in the training (unabsorbed) form ([Mishra] "Multi-head Latent
 * Attention": the unabsorbed form is the one used in training; [llms]
 * "Low-Rank Key-Value Joint Compression" for the up-projections and "The
 * Positional Problem and Decoupled RoPE" for the shared RoPE key).  Every
 * cached token of a sequence is a query; per query position t and head i
 *     k_{j,i} = [W^UK_i c_j ; k^R_j],   v_{j,i} = W^UV_i c_j
 *     u_{t,i} = sum_j softmax_j(q_{t,i} . k_{j,i} * scale) v_{j,i}
 * over j <= t (causal) or all j, and out_t = W^O concat_i u_{t,i}.  With
 * many queries this costs 2(d_h + d_r) + 2 d_h FLOPs per (query, key, head)
 * against 2(d_c + d_r) + 2 d_c for the absorbed form, so prefill takes it.
 * bf16 only (MLA_FP32 returns MLA_ERR_UNSUPPORTED).
 *
 * mla_prefill_expand -- the per-head keys and values of every cache row:
 *   kv     [rows, d_c + d_r]  cache rows [c ; k^R] (contiguous, in token order)
 *   w_uk, w_uv [H, d_h, d_c]
 *   k_nope [rows, H, d_h]     output, W^UK_i c
 *   v      [rows, H, d_h]     output, W^UV_i c
 * H * d_h % 128 == 0, d_c % 64 == 0.
 */
mla_status_t mla_prefill_expand(const void* kv, const void* w_uk, const void* w_uv, void* k_nope,
                                void* v, int rows, int H, int d_h, int d_c, int d_r,
                                mla_dtype_t dtype, mla_stream_t stream);

/*
 * mla_prefill_attn -- causal (or full) attention of B sequences of L tokens:
 *   q_nope [B*L, H, d_h], q_pe [B*L, H, d_r]   queries (q^R already rotated)
 *   k_nope, v [B*L, H, d_h]                    from mla_prefill_expand
 *   kv     [B*L, d_c + d_r]                    cache rows; k^R is read from
 *                                              columns d_c .. d_c + d_r - 1
 *   u      [B*L, H, d_h]  output;  lse [B*L, H] fp32 output (natural log)
 * d_h == 128, d_r == 64, d_c % 64 == 0, any L >= 1, H >= 1.
 */
mla_status_t mla_prefill_attn(const void* q_nope, const void* q_pe, const void* k_nope,
                              const void* kv, const void* v, int B, int L, int H, int d_h, int d_c,
                              int d_r, float scale, int causal, void* u, float* lse,
                              mla_dtype_t dtype, mla_stream_t stream);

/* Bytes of workspace mla_prefill_out needs (0 when none). */
size_t mla_prefill_workspace_size(int rows, int H, int d_h, int d, mla_dtype_t dtype);

/*
 * mla_prefill_out -- out [rows, d] = W^O u for u [rows, H * d_h] and
 * W^O [d, H * d_h]; d % 128 == 0.  workspace >= mla_prefill_workspace_size.
 */
mla_status_t mla_prefill_out(const void* u, const void* w_o, void* out, int rows, int H, int d_h,
                             int d, void* workspace, size_t workspace_bytes, mla_dtype_t dtype,
                             mla_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the current device's status
 * word.  Returns MLA_OK, MLA_ERR_TIMEOUT or MLA_ERR_DEVICE_BOUNDS (or
 * MLA_ERR_CUDA if the synchronisation itself failed).  If detail is not NULL
 * it receives the word's detail field (where the error was found).
 */
mla_status_t mla_get_device_status(mla_stream_t stream, uint32_t* detail);

/*
 * Set how long a kernel of this library waits for a pipeline step (a page
 * copy, a tensor-core product, a peer CTA) before it gives up, raises
 * MLA_ERR_TIMEOUT in the device status word and winds down: `ns`
 * nanoseconds on the current device, or the default of 2 s when ns == 0.
 * The waits a CTA makes at teardown for copies and products it issued
 * itself keep their own limit, so a short limit never leaves work in
 * flight.  A very short limit makes calls fail with MLA_ERR_TIMEOUT; it is
 * meant for testing the failure path.  Synchronous; returns MLA_ERR_CUDA if
 * the write fails.  Not thread-safe against calls in flight.
 */
mla_status_t mla_set_wait_limit(uint64_t ns);

/*
 * Timing hook: while set (both non-NULL), every bf16 mla_decode_attn call
 * records `start` on its stream just before its attention kernel and `end`
 * just after it, so that a caller can time that kernel apart from the
 * combine kernel of the same call.  Arguments are CUDA events (cudaEvent_t)
 * owned by the caller; NULL, NULL clears the hook.  Process-wide, not
 * thread-safe against concurrent decode calls.  Under stream capture the
 * events are recorded as external event nodes, so each replay of the graph
 * records them.
 */
void mla_set_decode_events(void* start, void* end);

/*
 * mla_decode_attn_noalloc -- mla_decode_attn for callers that cannot
 * allocate device memory: a host that owns all of the GPU's memory and
 * hands this library only its inputs and outputs (an inference-server
 * plugin with a fixed memory budget, for instance), or a code path that
 * must not allocate because allocation could block or synchronise the
 * device.  It takes the same arguments as mla_decode_attn without the
 * workspace, computes the same result with the same kernels, and allocates
 * nothing: its scratch is a fixed array of mla_decode_noalloc_max_bytes()
 * bytes inside the library, which every GPU that loads the library holds
 * until the process exits.  (The web pages on MLA have no counterpart to
 * this call; it is an interface convenience.)
 *
 * The array is 64 MiB.  The scratch needs (G + U) * 256 KiB plus a little,
 * for U = B * T * ceil(H / 128) work units and G co-resident clusters (74
 * on a 148-SM B300), so up to about 181 units fit on a B300: every decode
 * batch of one token and 128 heads up to B = 181 (the 64-, 128- and
 * 4-sequence batches, the 32 x 2-token batch and the 64 x 16-head batch all
 * fit); 4 sequences of 64 query tokens do not.
 *
 * The first call on a device (and the first call after that device's CUDA
 * context has been replaced, as by cudaDeviceReset) looks up that array's
 * device address with the device current; make that first call before any
 * stream capture.  Every call shares the one array and overwrites what the
 * last call left there, so calls whose kernels overlap on the GPU (on
 * different streams, or from different host threads) race: serialise them.
 * A shape whose scratch (mla_decode_workspace_size) exceeds the maximum
 * returns MLA_ERR_UNSUPPORTED before anything is launched; use
 * mla_decode_attn with a caller-owned workspace for it.
 */
mla_status_t mla_decode_attn_noalloc(const void* q_lat, const void* q_pe, const void* kv_pool,
                                     const int32_t* page_table, const int32_t* seq_lens,
                                     const int32_t* seq_lens_host, int B, int T, int H, int d_c,
                                     int d_r, int page_size, int max_pages, int64_t num_pages,
                                     float scale, int causal, void* o, float* lse,
                                     mla_dtype_t dtype, mla_stream_t stream);

/* Size in bytes of the fixed scratch array of mla_decode_attn_noalloc. */
size_t mla_decode_noalloc_max_bytes(void);

/* Number of kernels this library has launched in this process so far. */
uint64_t mla_launch_count(void);

/* Static description of a status code. */
const char* mla_status_string(mla_status_t status);

/* Library ABI version (major * 100 + minor). */
int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
